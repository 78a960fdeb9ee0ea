// Paged decode attention: one new query per sequence attends to every cached
// token of that sequence, whose K/V rows are found through the sequence's
// block table.  Kernels in this file:
//   * decode_bf16_streamk_kernel -- the balanced split (bf16, and an FP8
//     variant): every warp takes an equal share of all contexts' tiles, stores
//     the step's new tokens, and merges the contexts it cuts (see its header).
//   * decode_bf16_mma_kernel / decode_simt_kernel -- fixed partitions (bf16 /
//     fp32), whose partials decode_reduce_kernel merges.
// Grouped (shared-prefix) decode and multi-token attention run on the
// tensor-core kernel of rows_attention.cu.
//
// Sources: "KV cache & PagedAttention -- vi sao chatbot AI ton bo nho"
// (aiwiki.vn), second paragraph (the current query against the keys of the
// visible positions, the weights combine the values); "PagedAttention (vLLM)
// -- Virtual memory cho AI", section "Tai sao no hoat dong", item "Kernel
// scatter-gather" (the kernel receives the block table and gathers K/V from
// scattered blocks into on-chip memory before the softmax), and section
// "Y nghia thuc te" (paging addresses capacity; the decode step itself stays
// bound by memory bandwidth -- "vLLM PagedAttention: Buoc dot pha ...",
// item "Disaggregated Prefill/Decoding").
//
// bf16 path (decode_bf16_mma_kernel), one CTA per (sequence, kv head,
// partition), NW warps that each own every NW-th 16-token tile:
//   * Each warp streams its tiles through its own ring of NS shared-memory
//     stages.  One lane issues 2-D tensor TMA loads (cp.async.bulk.tensor)
//     of the 16 x 64-element halves of K and V straight from the scattered
//     physical blocks, 128-byte swizzled, completing on the stage's mbarrier.
//   * S^T = K_tile . Q^T on the tensor cores (mma.sync m16n8k16, bf16 in,
//     fp32 accumulate): M = 16 tokens, N = the (up to 8) query heads that
//     share this KV head, K = head_dim.  Each K/V byte is read from HBM
//     once for the whole query-head group.
//   * Online softmax per query head in registers (warp shuffles across the
//     token rows), probabilities rounded to bf16 and transposed in registers
//     (movmatrix) into the B operand of O^T += V_tile^T . P^T.
//   * At the end the warps' (max, sum, output) triples are merged through
//     shared memory in a fixed order, so results depend only on logical
//     token positions, never on where the blocks sit in the pool.
// fp32 path (decode_simt_kernel): the same decomposition on CUDA cores with
// fp32 FMAs and expf, no tensor cores, no TF32.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pkv_internal.cuh"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kTile = 16;  // tokens per MMA tile and per pipeline stage
constexpr int kGMax = 8;   // max query heads per KV head (the MMA N dimension)

struct DecodeArgs {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *part_o;  // [S][Hq][max_parts][D]
    float *part_m;  // [S][Hq][max_parts]
    float *part_l;  // [S][Hq][max_parts]
    // balanced path (merge in the attention kernel): one ready flag per
    // (segment, partial slot) [S][Hkv][max_parts], set to this call's tag
    // (never 0) once the slot's partial is stored
    unsigned long long *flags;
    unsigned long long tag;
    int merge_trigger;    // merge kernel: let the next kernel start early (small merges only)
    int num_seqs, num_heads, num_kv_heads, group;
    int block_size, max_blocks, num_blocks, max_seq_len;
    int partition_size, max_parts;
    float scale;       // multiplies q.k
    float scale_log2;  // scale * log2(e), for the exp2 form of the softmax
    float f8_kscale_log2;  // FP8 cache: scale * k_scale * log2(e)
    float f8_kscale;       // FP8 cache: k_scale (quantising the appended token)
    float f8_vscale;       // FP8 cache: v_scale
    int f8_bshift;         // FP8 cache: log2(block_size)
    unsigned int *err;
    // fused append: each sequence's new token [S][Hkv][D] goes to position
    // seq_lens[s] - 1 before it is attended (nullptr: no append)
    const void *k_new;
    const void *v_new;
    void *k_cache_w;
    void *v_cache_w;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A(16x16, row) . B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held as one register per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// Per-CTA work item: (sequence, kv head, partition).
// ---------------------------------------------------------------------------
struct WorkItem {
    int seq, kvh, part;
    int len;     // context length after clamping
    int nparts;  // partitions this sequence needs (0 when len == 0)
    int tok_begin, tok_end;
};

// Returns false when this CTA has nothing to do.
__device__ __forceinline__ bool resolve_item(const DecodeArgs &a, WorkItem &w) {
    w.seq = blockIdx.x;
    w.kvh = blockIdx.y;
    w.part = blockIdx.z;
    int len = a.seq_lens[w.seq];
    const int cap = min(a.max_seq_len, a.max_blocks * a.block_size);
    if (len < 0 || len > cap) {
        if (threadIdx.x == 0 && w.kvh == 0 && w.part == 0) flag_error(a.err, PKV_DEVERR_SEQ_LEN);
        len = len < 0 ? 0 : cap;
    }
    w.len = len;
    w.nparts = (len + a.partition_size - 1) / a.partition_size;
    if (w.part >= (w.nparts > 0 ? w.nparts : 1)) return false;
    w.tok_begin = w.part * a.partition_size;
    w.tok_end = min(len, w.tok_begin + a.partition_size);
    return true;
}

template <typename T, int D>
__device__ void write_zero_rows(const DecodeArgs &a, const WorkItem &w) {
    T *out = static_cast<T *>(a.out);
    for (int i = threadIdx.x; i < a.group * D; i += blockDim.x) {
        const int g = i / D, d = i % D;
        store_out(out + ((int64_t)w.seq * a.num_heads + w.kvh * a.group + g) * D + d, 0.0f);
    }
}

// Merge the per-warp partial results held in shared memory (layout per warp:
// o[kGMax][D], then m[kGMax], then l[kGMax]) and write either the final rows
// (single-partition sequence) or this partition's partial.  `ex` is exp or
// exp2 to match the domain the running maxima were kept in.
template <typename T, int D, int NW, bool LOG2>
__device__ void merge_warps_and_store(const DecodeArgs &a, const WorkItem &w,
                                      const float *const (&warp_buf)[NW]) {
    for (int i = threadIdx.x; i < a.group * D; i += NW * 32) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < NW; ++k) M = fmaxf(M, warp_buf[k][kGMax * D + g]);
        float osum = 0.f, lsum = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float mk = warp_buf[k][kGMax * D + g];
            if (mk == -INFINITY) continue;
            const float c = LOG2 ? exp2f(mk - M) : expf(mk - M);
            osum += c * warp_buf[k][g * D + d];
            lsum += c * warp_buf[k][kGMax * D + kGMax + g];
        }
        const int64_t row = (int64_t)w.seq * a.num_heads + w.kvh * a.group + g;
        if (w.nparts == 1) {
            // lsum == 0 only when every block of the context was invalid (flagged)
            store_out(static_cast<T *>(a.out) + row * D + d, lsum > 0.f ? osum / lsum : 0.f);
        } else {
            const int64_t p = row * a.max_parts + w.part;
            a.part_o[p * D + d] = osum;
            if (d == 0) {
                a.part_m[p] = M;
                a.part_l[p] = lsum;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// bf16 tensor-core kernel
// ---------------------------------------------------------------------------
template <int D>
struct Bf16Layout {
    static constexpr int kHalves = D / 64;               // 64-element (128-byte) column halves
    static constexpr int kHalfBytes = kTile * 128;        // 16 rows x 128 bytes
    static constexpr int kKVBytes = kHalves * kHalfBytes;  // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kKVBytes;
    static constexpr int kMergeBytes = (kGMax * D + 2 * kGMax) * 4;
};

constexpr int kBtCache = 256;  // block ids of one partition kept in shared memory

template <int D, int NW, int NS>
constexpr int bf16_smem_bytes() {
    return NW * NS * Bf16Layout<D>::kStageBytes + NW * NS * 8 + kBtCache * 4 + 1024;
}

// Running softmax state of one warp for up to 8 query heads (MMA fragment
// layout: this lane holds heads 2tq and 2tq+1, head_dim rows r0 and r0+8 of
// every 16-row slice).
template <int D>
struct WarpAcc {
    float m0, m1, l0, l1;
    float o[D / 16][4];
    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }
};

// Q^T as the MMA B operand: lane holds query head r0 (zero past the group),
// head_dim pairs 16ks + 2tq (+8).
template <int D>
__device__ __forceinline__ void load_q_fragments(const DecodeArgs &a, int seq, int kvh, int lane,
                                                 uint32_t (&qb)[D / 16][2]) {
    const int r0 = lane >> 2, tq = lane & 3;
    const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(a.q) +
                                ((int64_t)seq * a.num_heads + kvh * a.group + r0) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        if (r0 < a.group) {
            qb[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * tq);
            qb[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * tq);
        } else {
            qb[ks][0] = qb[ks][1] = 0u;
        }
    }
}

// Attend one staged 16-token tile (K at sk, V at sv, 128-byte swizzled
// halves).  row_ok has a bit per token row that this query attends (inside
// its context, from a valid block); the other rows get zero weight.  Rows
// cleared in zero_ok (default: row_ok) hold stale, unwritten or substituted
// slots: their V is zeroed first so that a zero weight never meets a NaN.
// Warps sharing a stage pass the same zero_ok (only zeros are ever written).
template <int D, bool kZeroMasked = true>
__device__ __forceinline__ void attend_tile(unsigned char *sk, unsigned char *sv, uint32_t row_ok,
                                            const uint32_t (&qb)[D / 16][2], float sl2,
                                            WarpAcc<D> &acc, int lane, uint32_t zero_ok = 0x10000u) {
    using Lay = Bf16Layout<D>;
    const int r0 = lane >> 2;
    if (zero_ok == 0x10000u) zero_ok = row_ok;
    if (kZeroMasked && zero_ok != 0xffffu) {
        for (int e = lane; e < Lay::kHalves * kTile * 8; e += 32) {
            const int h = e / (kTile * 8), rr = (e / 8) % kTile, c = e % 8;
            if (!((zero_ok >> rr) & 1u))
                *reinterpret_cast<uint4 *>(sv + h * Lay::kHalfBytes + rr * 128 + c * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
    }
    const uint32_t ska = smem_u32(sk), sva = smem_u32(sv);
    const int lj = lane >> 3, lr = lane & 7;
    // this lane's row of each 8x8 ldmatrix: token row and 16-byte chunk, 128-byte swizzle
    const int ktok = lr + 8 * (lj & 1), vtok = lr + 8 * (lj >> 1);
    const uint32_t krow = ska + ktok * 128, vrow = sva + vtok * 128;
    const int kx = ktok & 7, vx = vtok & 7;

    // S^T (16 tokens x 8 heads) = K_tile . Q^T
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int chunk = 2 * (ks & 3) + (lj >> 1);
        uint32_t x0, x1, x2, x3;
        ldmatrix_x4(krow + (ks >> 2) * Lay::kHalfBytes + ((chunk ^ kx) << 4), x0, x1, x2, x3);
        mma_bf16_16816(sc, x0, x1, x2, x3, qb[ks][0], qb[ks][1]);
    }

    // online softmax, base 2; rows r0 and r0+8, columns 2tq and 2tq+1
    const bool ok_lo = (row_ok >> r0) & 1u, ok_hi = (row_ok >> (r0 + 8)) & 1u;
    const float s0 = ok_lo ? sc[0] * sl2 : -INFINITY;
    const float s1 = ok_lo ? sc[1] * sl2 : -INFINITY;
    const float s2 = ok_hi ? sc[2] * sl2 : -INFINITY;
    const float s3 = ok_hi ? sc[3] * sl2 : -INFINITY;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
    }
    const float mn0 = fmaxf(acc.m0, mx0), mn1 = fmaxf(acc.m1, mx1);
    // reference points stay finite even if nothing valid has been seen yet
    const float rf0 = mn0 == -INFINITY ? 0.f : mn0, rf1 = mn1 == -INFINITY ? 0.f : mn1;
    // the running maxima rarely move once a few tiles are in: rescale only then
    const bool moved = __any_sync(0xffffffffu, mn0 != acc.m0 || mn1 != acc.m1);
    const float al0 = exp2f(acc.m0 - rf0), al1 = exp2f(acc.m1 - rf1);
    acc.m0 = mn0;
    acc.m1 = mn1;
    const uint32_t p01 = pack_bf16x2(exp2f(s0 - rf0), exp2f(s1 - rf1));
    const uint32_t p23 = pack_bf16x2(exp2f(s2 - rf0), exp2f(s3 - rf1));
    // the sum uses the same rounded weights as the numerator
    if (moved) {
        acc.l0 = acc.l0 * al0;
        acc.l1 = acc.l1 * al1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            acc.o[mt][0] *= al0;
            acc.o[mt][1] *= al1;
            acc.o[mt][2] *= al0;
            acc.o[mt][3] *= al1;
        }
    }
    acc.l0 += bf16x2_lo(p01) + bf16x2_lo(p23);
    acc.l1 += bf16x2_hi(p01) + bf16x2_hi(p23);
    const uint32_t pb0 = movmatrix_trans(p01);
    const uint32_t pb1 = movmatrix_trans(p23);

    // O^T (head_dim x 8 heads) += V_tile^T . P^T
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int chunk = 2 * (mt & 3) + (lj & 1);
        uint32_t x0, x1, x2, x3;
        ldmatrix_x4_trans(vrow + (mt >> 2) * Lay::kHalfBytes + ((chunk ^ vx) << 4), x0, x1, x2, x3);
        mma_bf16_16816(acc.o[mt], x0, x1, x2, x3, pb0, pb1);
    }
}

// Finish a warp's sums and park (o[kGMax][D], m[kGMax], l[kGMax]) at `dst`
// for the cross-warp merge.  `empty` marks a warp that saw no tile.
// Layout at dst: o[ng][D], then m[kGMax], then l[kGMax]; heads g >= ng are
// not stored.
template <int D>
__device__ __forceinline__ void park_partial(WarpAcc<D> &acc, bool empty, float *dst, int lane,
                                             int ng = kGMax) {
    const int r0 = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {  // column sums over the 16 token rows
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, sh);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, sh);
    }
    if (empty) {
        acc.m0 = acc.m1 = -INFINITY;
        acc.l0 = acc.l1 = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = 16 * mt + r0 + 8 * (j >> 1);
            const int g = 2 * tq + (j & 1);
            if (g < ng) dst[g * D + d] = acc.o[mt][j];
        }
    }
    if (r0 == 0) {
        dst[ng * D + 2 * tq] = acc.m0;
        dst[ng * D + 2 * tq + 1] = acc.m1;
        dst[ng * D + kGMax + 2 * tq] = acc.l0;
        dst[ng * D + kGMax + 2 * tq + 1] = acc.l1;
    }
}

// Rows of the tile starting at token t0 that belong to the context (< tok_end)
// and come from a block id inside the pool.
template <typename BlockOf>
__device__ __forceinline__ uint32_t tile_rows_ok(int t0, int tok_end, int B, int boxh, int num_blocks,
                                                 BlockOf block_of) {
    uint32_t row_ok = 0;
    for (int sb = 0; sb < kTile / boxh; ++sb) {
        const int tok = t0 + sb * boxh;
        if (tok >= tok_end) break;
        const int blk = block_of(tok / B);
        if (blk >= 0 && blk < num_blocks) row_ok |= ((1u << boxh) - 1u) << (sb * boxh);
    }
    const int valid = min(kTile, tok_end - t0);
    return row_ok & ((1u << valid) - 1u);
}

// Gather the 16-token tile starting at token t0 of (sequence, kv head kvh)
// into a ring stage with 2-D TMA boxes; one lane calls this.
template <int D, typename BlockOf>
__device__ __forceinline__ void issue_tile(const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                           unsigned char *stage, uint64_t *bar, int t0, int tok_end,
                                           int kvh, const DecodeArgs &a, BlockOf block_of) {
    using Lay = Bf16Layout<D>;
    const int B = a.block_size;
    const int boxh = B < kTile ? B : kTile;
    int ys[kTile / 8];
    int nsub = 0;
    for (int sb = 0; sb < kTile / boxh; ++sb) {
        const int tok = t0 + sb * boxh;
        if (tok >= tok_end) break;
        const int lb = tok / B;
        int blk = block_of(lb);
        if (blk < 0 || blk >= a.num_blocks) {
            // never dereferenced out of range: read block 0 instead and mask
            // these rows out of the softmax (tile_rows_ok)
            flag_error(a.err, PKV_DEVERR_BLOCK_ID);
            blk = 0;
        }
        ys[nsub++] = (int)(((int64_t)blk * a.num_kv_heads + kvh) * B + (tok - lb * B));
    }
    const uint32_t bytes = (uint32_t)(nsub * Lay::kHalves * boxh * 128 * 2);
    const uint32_t b = smem_u32(bar);
    mbar_arrive_expect_tx(bar, bytes);
    const uint32_t dk = smem_u32(stage);
    const uint32_t dv = dk + Lay::kKVBytes;
    for (int sb = 0; sb < nsub; ++sb) {
#pragma unroll
        for (int h = 0; h < Lay::kHalves; ++h) {
            const uint32_t off = h * Lay::kHalfBytes + sb * boxh * 128;
            tma_load_2d(dk + off, tm_k, b, h * 64, ys[sb]);
            tma_load_2d(dv + off, tm_v, b, h * 64, ys[sb]);
        }
    }
}

// One CTA per (sequence, kv head, partition): the fixed-partition path.
template <int D, int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
decode_bf16_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using Lay = Bf16Layout<D>;
    static_assert(NS * Lay::kStageBytes >= Lay::kMergeBytes, "merge area must fit a warp's ring");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    grid_dependency_wait();
    grid_launch_dependents();

    WorkItem w;
    if (!resolve_item(a, w)) return;
    if (w.len == 0) {
        write_zero_rows<__nv_bfloat16, D>(a, w);
        return;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char *ring = smem + warp * NS * Lay::kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * NS * Lay::kStageBytes) + warp * NS;
    int *bt_s = reinterpret_cast<int *>(smem + NW * NS * Lay::kStageBytes + NW * NS * 8);
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }

    // The partition's block ids, read once into shared memory so that no TMA
    // issue waits on a global load.
    const int32_t *bt = a.block_tables + (int64_t)w.seq * a.max_blocks;
    const int lb0 = w.tok_begin / a.block_size;
    const int nblk = (w.tok_end - 1) / a.block_size - lb0 + 1;
    for (int i = threadIdx.x; i < nblk && i < kBtCache; i += NW * 32) bt_s[i] = bt[lb0 + i];
    __syncthreads();
    auto block_of = [&](int lb) { return lb - lb0 < kBtCache ? bt_s[lb - lb0] : bt[lb]; };

    uint32_t qb[D / 16][2];
    load_q_fragments<D>(a, w.seq, w.kvh, lane, qb);

    const int ntiles = (w.tok_end - w.tok_begin + kTile - 1) / kTile;
    const int nmine = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
    const int boxh = a.block_size < kTile ? a.block_size : kTile;
    auto issue = [&](int tile, int buf) {
        issue_tile<D>(&tm_k, &tm_v, ring + buf * Lay::kStageBytes, &bars[buf],
                      w.tok_begin + tile * kTile, w.tok_end, w.kvh, a, block_of);
    };
    if (lane == 0) {
        for (int i = 0; i < NS && i < nmine; ++i) issue(warp + i * NW, i);
    }

    WarpAcc<D> acc;
    acc.reset();
    bool dead = false;
    for (int i = 0; i < nmine; ++i) {
        const int buf = i % NS;
        if (!mbar_wait_bounded(&bars[buf], (uint32_t)((i / NS) & 1))) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            dead = true;
            break;
        }
        const int t0 = w.tok_begin + (warp + i * NW) * kTile;
        const uint32_t row_ok = tile_rows_ok(t0, w.tok_end, a.block_size, boxh, a.num_blocks, block_of);
        unsigned char *sk = ring + buf * Lay::kStageBytes;
        attend_tile<D>(sk, sk + Lay::kKVBytes, row_ok, qb, a.scale_log2, acc, lane);
        __syncwarp();
        if (lane == 0 && i + NS < nmine) {
            fence_proxy_async();
            issue(warp + (i + NS) * NW, buf);
        }
    }

    // Each warp parks its partial in its own (now idle) ring.
    park_partial<D>(acc, dead || nmine == 0, reinterpret_cast<float *>(ring), lane);
    __syncthreads();
    const float *bufs[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) bufs[k] = reinterpret_cast<const float *>(smem + k * NS * Lay::kStageBytes);
    merge_warps_and_store<__nv_bfloat16, D, NW, true>(a, w, bufs);
}

// ---------------------------------------------------------------------------
// Balanced (stream-K) kernel: all (sequence, kv head) segments are laid end to
// end as one list of tiles, and every warp of a persistent one-wave grid takes
// an equal, contiguous share of that list, streaming it through its own TMA
// ring across segment boundaries.  Every warp streams the same number of
// bytes, so no SM idles in a tail wave.  The helpers below: the shared-memory
// layout, a cursor over the tile list, share ownership, tile rows.
// ---------------------------------------------------------------------------
constexpr int kMinTilesPerCta = 16;  // >= 256 tokens per share: bounds pieces per segment
// Scheduling charge of a segment, in tiles: a segment with n tiles is laid
// out as kLeadTiles empty tiles (no loads, nothing attended) and then its n
// real ones, so that equal shares of the layout also balance the fixed cost
// of a piece (its queries, the store of its rows or partial) and of the merge,
// which falls to the warp holding the segment's first laid-out tile.
constexpr int kLeadTiles = 3;
__host__ __device__ __forceinline__ int laid_out_tiles(int n) { return n > 0 ? n + kLeadTiles : 0; }

constexpr int kYCache = 256;  // tiles of a CTA whose TMA rows are staged in shared memory (3 CTAs of 4 warps fit an SM up to ~750 sequences)
constexpr int kRotateTiles = 10;  // a first piece shorter than this is attended last

// Shared-memory layout of the balanced kernel (host and device agree on it).
// Offsets are from the 1024-aligned base.
struct StreamKLayout {
    int ring, bars, patch, ycache, masks, srcs, prefix, total;
    // stage_bytes: one ring stage (K and V of one tile); new_bytes: per stage,
    // room for one new K row and V row (fused append), or 0 (then no srcs)
    __host__ __device__ StreamKLayout(int D, int NW, int NS, int num_seqs, int stage_bytes, int new_bytes) {
        ring = NW * NS * stage_bytes;
        bars = ring;
        patch = bars + NW * NS * 8;      // 16-byte aligned (bulk copies)
        ycache = patch + NW * NS * new_bytes;  // int2 per cached tile
        masks = ycache + kYCache * 8;  // valid-row mask per cached tile
        srcs = masks + kYCache * 4;    // fused append: new-token row of a cached last tile, else -1
        prefix = srcs + (new_bytes ? kYCache * 4 : 0);
        total = prefix + (num_seqs + 1) * 4 + 1024;  // + alignment slack
    }
};

// Walks the tile list in increasing order: tile t lies in segment
// (seq, kvh), whose first tile is seg_start and which has n tiles.
struct SegCursor {
    int seq, kvh, n;
    int64_t seg_start;
    __device__ __forceinline__ void seek(const int *prefix, int num_seqs, int hkv, int64_t t) {
        int lo = 0, hi = num_seqs;  // largest seq with prefix[seq] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid;
        }
        seq = lo;
        n = (prefix[seq + 1] - prefix[seq]) / hkv;
        kvh = (int)((t - prefix[seq]) / n);
        seg_start = prefix[seq] + (int64_t)kvh * n;
    }
    __device__ __forceinline__ void advance_to(const int *prefix, int hkv, int64_t t) {
        while (t >= seg_start + n) {
            seg_start += n;
            if (++kvh == hkv) {
                kvh = 0;
                do {
                    ++seq;
                    n = (prefix[seq + 1] - prefix[seq]) / hkv;
                } while (n == 0);
                seg_start = prefix[seq];
            }
        }
    }
};

__device__ __forceinline__ int clamp_len(int len, int cap) { return len < 0 ? 0 : (len > cap ? cap : len); }

// TMA rows and valid-row mask of one tile: tile `tile` of segment (seq, kvh)
// of a context of `len` tokens.  y = -1 for a sub-block past the context.
struct TileRows {
    int y0, y1;
    uint32_t mask;
};

__device__ __forceinline__ uint32_t low_bits(int n) { return n >= 32 ? 0xffffffffu : (1u << n) - 1u; }

// TT = tokens per tile (16, or 32 for the FP8 path); at most two sub-blocks
template <int TT = kTile>
__device__ __forceinline__ TileRows tile_rows(const DecodeArgs &a, int seq, int kvh, int tile, int len,
                                              int tok_off = 0) {
    const int B = a.block_size;
    const int boxh = B < TT ? B : TT;
    const int32_t *bt = a.block_tables + (int64_t)seq * a.max_blocks;
    TileRows r{-1, -1, 0u};
    for (int sb = 0; sb < TT / boxh; ++sb) {
        const int tok = tok_off + tile * TT + sb * boxh;
        if (tok >= len) break;
        const int lb = tok / B;
        int blk = bt[lb];
        if (blk >= 0 && blk < a.num_blocks) {
            r.mask |= low_bits(boxh) << (sb * boxh);
        } else {
            // never dereferenced out of range: read block 0, rows masked out
            flag_error(a.err, PKV_DEVERR_BLOCK_ID);
            blk = 0;
        }
        const int y = (int)(((int64_t)blk * a.num_kv_heads + kvh) * B + (tok - lb * B));
        if (sb == 0) r.y0 = y; else r.y1 = y;
    }
    const int valid = min(TT, len - tok_off - tile * TT);
    r.mask &= low_bits(valid);
    return r;
}

template <int D>
__device__ __forceinline__ void issue_rows(const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                           unsigned char *stage, uint64_t *bar, int boxh, TileRows r,
                                           uint32_t extra_bytes = 0) {
    using Lay = Bf16Layout<D>;
    const int nsub = r.y0 < 0 ? 0 : (r.y1 < 0 ? 1 : 2);
    // extra_bytes: further copies the caller issues on the same barrier
    mbar_arrive_expect_tx(bar, (uint32_t)(nsub * Lay::kHalves * boxh * 128 * 2) + extra_bytes);
    const uint32_t b = smem_u32(bar);
    const uint32_t dk = smem_u32(stage);
    const uint32_t dv = dk + Lay::kKVBytes;
    for (int sb = 0; sb < nsub; ++sb) {
        const int y = sb == 0 ? r.y0 : r.y1;
#pragma unroll
        for (int h = 0; h < Lay::kHalves; ++h) {
            const uint32_t off = h * Lay::kHalfBytes + sb * boxh * 128;
            tma_load_2d(dk + off, tm_k, b, h * 64, y);
            tma_load_2d(dv + off, tm_v, b, h * 64, y);
        }
    }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) cache.  K tiles are 16 token rows x D codes (128-byte swizzle);
// V is stored transposed inside each block, so a V tile is D rows x 16 token
// codes.  Codes widen exactly to f16 (every E4M3 value is an f16 value), the
// queries are scaled by a power of two per head into f16's range, and both
// contractions run as f16 mma.sync with fp32 accumulation; the scales (the
// per-tensor k_scale and v_scale, the softmax scale, the query's power of
// two) are applied to the fp32 results.
// ---------------------------------------------------------------------------
// Four E4M3 codes (bytes 0..3 of x) -> f16x2 {byte0, byte1} and {byte2, byte3}.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// D += A(16x16, row) . B(16x8, col), f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float f16x2_lo(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float f16x2_hi(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// Stage sizes of one 16-token tile (K then V) for either cache type.
template <int D, bool F8>
struct TileBytes {
    static constexpr int kKV = F8 ? 2 * kTile * D : Bf16Layout<D>::kKVBytes;  // offset of V
    static constexpr int kStage = 2 * kKV;
};

// Q^T as the f16 MMA B operand for the FP8 path.  The lane with g = lane/4,
// t = lane%4 holds query head g, head_dim entries 16c + 4t .. 16c + 4t + 3 of
// chunk c: that is the order in which the K fragment below receives the
// codes, so the contraction pairs every key entry with its query entry.  Each
// head is multiplied by 2^e so that its largest |q| lies in [2^14, 2^15)
// (exact: bf16 has 8 significant bits, f16 11).  s0 / s1 return the score
// factors scale * k_scale * log2(e) * 2^-e of heads 2t and 2t+1, the columns
// of S^T this lane accumulates.
template <int D>
__device__ __forceinline__ void load_q_f16(const DecodeArgs &a, int seq, int kvh, int lane,
                                           uint32_t (&qb)[D / 16][2], float &s0, float &s1) {
    const int g = lane >> 2, t = lane & 3;
    const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(a.q) +
                                ((int64_t)seq * a.num_heads + kvh * a.group + g) * D;
    uint2 w[D / 16];
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        w[c] = g < a.group ? *reinterpret_cast<const uint2 *>(qrow + 16 * c + 4 * t) : make_uint2(0u, 0u);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16x2_lo(w[c].x)), fabsf(bf16x2_hi(w[c].x))),
                                 fmaxf(fabsf(bf16x2_lo(w[c].y)), fabsf(bf16x2_hi(w[c].y)))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // amax in [2^(E-127), 2^(E-126)): multiply by 2^(141-E), biased exponent 268-E
    const int E = (int)((__float_as_uint(amax) >> 23) & 0xffu);
    const int fe = min(253, max(1, 268 - E));
    const float f = __uint_as_float((uint32_t)fe << 23);
    const float desc = a.f8_kscale_log2 * __uint_as_float((uint32_t)(254 - fe) << 23);
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        qb[c][0] = pack_f16x2(bf16x2_lo(w[c].x) * f, bf16x2_hi(w[c].x) * f);
        qb[c][1] = pack_f16x2(bf16x2_lo(w[c].y) * f, bf16x2_hi(w[c].y) * f);
    }
    s0 = __shfl_sync(0xffffffffu, desc, 8 * t);
    s1 = __shfl_sync(0xffffffffu, desc, 8 * t + 4);
}

// FP8 counterpart of attend_tile for a 32-token tile: K at sk (32 token rows
// x D codes, 128-byte swizzle), V^T at sv as two halves (tokens 0-15, then
// 16-31), each D rows x 16 codes; per-column score factors s0 / s1.  The two
// 16-row halves give two independent MMA chains.
template <int D>
__device__ __forceinline__ void attend_tile_f8(unsigned char *sk, unsigned char *sv, uint32_t row_ok,
                                               const uint32_t (&qb)[D / 16][2], float s0, float s1,
                                               WarpAcc<D> &acc, int lane) {
    static_assert(D == 128, "FP8 tiles assume 128-byte K rows");
    const int g = lane >> 2, t = lane & 3;
    if (row_ok != 0xffffffffu) {
        // masked tokens hold stale or unwritten codes (possibly NaN): clear
        // their bytes in every V^T row so that a zero weight meets a zero
        uint32_t m[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) m[w] = ((((row_ok >> (4 * w)) & 0xfu) * 0x00204081u) & 0x01010101u) * 0xffu;
#pragma unroll
        for (int i = 0; i < 2 * D / 32; ++i) {
            const int h = (32 * i) / D;  // half: tokens 0-15 or 16-31
            uint4 *p = reinterpret_cast<uint4 *>(sv + (32 * i + lane) * kTile);
            uint4 v = *p;
            v.x &= m[4 * h];
            v.y &= m[4 * h + 1];
            v.z &= m[4 * h + 2];
            v.w &= m[4 * h + 3];
            *p = v;
        }
        __syncwarp();
    }
    const uint32_t ska = smem_u32(sk), sva = smem_u32(sv);
    const int lj = lane >> 3, lr = lane & 7;
    // ldmatrix rows: token lr (+8 for matrices 1 and 3; +16 for the second
    // half), 16-byte chunk 2kk (+1 for matrices 2 and 3); row & 7 == lr
    const uint32_t krow0 = ska + (lr + 8 * (lj & 1)) * D, krow1 = krow0 + kTile * D;

    // S^T (tokens x 8 heads) = K_tile . Q^T; a lane's 4 codes of a chunk are
    // head_dim entries 4t..4t+3, split as the fragment's k pairs (2t, 2t+1)
    // and (2t+8, 2t+9) -- the same split load_q_f16 gives the queries
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
        const uint32_t off = ((2 * kk + (lj >> 1)) ^ lr) << 4;
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3, a0, a1, a2, a3;
        ldmatrix_x4(krow0 + off, x0, x1, x2, x3);
        ldmatrix_x4(krow1 + off, y0, y1, y2, y3);
        e4m3x4_to_f16(x0, a0, a2);
        e4m3x4_to_f16(x1, a1, a3);
        mma_f16_16816(sa, a0, a1, a2, a3, qb[2 * kk][0], qb[2 * kk][1]);
        e4m3x4_to_f16(y0, a0, a2);
        e4m3x4_to_f16(y1, a1, a3);
        mma_f16_16816(sb, a0, a1, a2, a3, qb[2 * kk][0], qb[2 * kk][1]);
        e4m3x4_to_f16(x2, a0, a2);
        e4m3x4_to_f16(x3, a1, a3);
        mma_f16_16816(sa, a0, a1, a2, a3, qb[2 * kk + 1][0], qb[2 * kk + 1][1]);
        e4m3x4_to_f16(y2, a0, a2);
        e4m3x4_to_f16(y3, a1, a3);
        mma_f16_16816(sb, a0, a1, a2, a3, qb[2 * kk + 1][0], qb[2 * kk + 1][1]);
    }

    // online softmax, base 2; rows g, g+8, 16+g, 24+g; columns 2t and 2t+1
    const bool ok0 = (row_ok >> g) & 1u, ok1 = (row_ok >> (g + 8)) & 1u;
    const bool ok2 = (row_ok >> (g + 16)) & 1u, ok3 = (row_ok >> (g + 24)) & 1u;
    const float v0 = ok0 ? sa[0] * s0 : -INFINITY, v1 = ok0 ? sa[1] * s1 : -INFINITY;
    const float v2 = ok1 ? sa[2] * s0 : -INFINITY, v3 = ok1 ? sa[3] * s1 : -INFINITY;
    const float v4 = ok2 ? sb[0] * s0 : -INFINITY, v5 = ok2 ? sb[1] * s1 : -INFINITY;
    const float v6 = ok3 ? sb[2] * s0 : -INFINITY, v7 = ok3 ? sb[3] * s1 : -INFINITY;
    float mx0 = fmaxf(fmaxf(v0, v2), fmaxf(v4, v6)), mx1 = fmaxf(fmaxf(v1, v3), fmaxf(v5, v7));
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
    }
    const float mn0 = fmaxf(acc.m0, mx0), mn1 = fmaxf(acc.m1, mx1);
    const float rf0 = mn0 == -INFINITY ? 0.f : mn0, rf1 = mn1 == -INFINITY ? 0.f : mn1;
    const bool moved = __any_sync(0xffffffffu, mn0 != acc.m0 || mn1 != acc.m1);
    const float al0 = exp2f(acc.m0 - rf0), al1 = exp2f(acc.m1 - rf1);
    acc.m0 = mn0;
    acc.m1 = mn1;
    const uint32_t p01 = pack_f16x2(exp2f(v0 - rf0), exp2f(v1 - rf1));
    const uint32_t p23 = pack_f16x2(exp2f(v2 - rf0), exp2f(v3 - rf1));
    const uint32_t p45 = pack_f16x2(exp2f(v4 - rf0), exp2f(v5 - rf1));
    const uint32_t p67 = pack_f16x2(exp2f(v6 - rf0), exp2f(v7 - rf1));
    if (moved) {
        acc.l0 = acc.l0 * al0;
        acc.l1 = acc.l1 * al1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            acc.o[mt][0] *= al0;
            acc.o[mt][1] *= al1;
            acc.o[mt][2] *= al0;
            acc.o[mt][3] *= al1;
        }
    }
    acc.l0 += (f16x2_lo(p01) + f16x2_lo(p23)) + (f16x2_lo(p45) + f16x2_lo(p67));
    acc.l1 += (f16x2_hi(p01) + f16x2_hi(p23)) + (f16x2_hi(p45) + f16x2_hi(p67));

    // P^T as the B operand of O^T += V^T . P^T.  A lane's V^T fragment holds
    // tokens 4t..4t+3 of its head_dim row (k pairs (2t, 2t+1) = tokens 4t,
    // 4t+1 and (2t+8, 2t+9) = tokens 4t+2, 4t+3), so P^T must hold the same
    // tokens: after the transposes lane t' has tokens 2t', 2t'+1 (first
    // matrix) and 8+2t', 9+2t' (second) of its head; gather them from the
    // lanes of that head.
    const int src = (lane & ~3) | (2 * (t & 1));
    uint32_t pa0, pa1, pb0, pb1;
    {
        const uint32_t m0 = movmatrix_trans(p01), m1 = movmatrix_trans(p23);
        const uint32_t e0 = __shfl_sync(0xffffffffu, m0, src), e1 = __shfl_sync(0xffffffffu, m1, src);
        const uint32_t f0 = __shfl_sync(0xffffffffu, m0, src + 1), f1 = __shfl_sync(0xffffffffu, m1, src + 1);
        pa0 = t < 2 ? e0 : e1;
        pa1 = t < 2 ? f0 : f1;
    }
    {
        const uint32_t m0 = movmatrix_trans(p45), m1 = movmatrix_trans(p67);
        const uint32_t e0 = __shfl_sync(0xffffffffu, m0, src), e1 = __shfl_sync(0xffffffffu, m1, src);
        const uint32_t f0 = __shfl_sync(0xffffffffu, m0, src + 1), f1 = __shfl_sync(0xffffffffu, m1, src + 1);
        pb0 = t < 2 ? e0 : e1;
        pb1 = t < 2 ? f0 : f1;
    }

    // O^T (head_dim x 8 heads) += V^T . P^T over both halves; the matrices of
    // one ldmatrix.x4 are head_dim rows 32j + 0..7, 8..15, 16..23, 24..31
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3, a0, a1, a2, a3;
        ldmatrix_x4(sva + (32 * j + lane) * kTile, x0, x1, x2, x3);
        ldmatrix_x4(sva + kTile * D + (32 * j + lane) * kTile, y0, y1, y2, y3);
        e4m3x4_to_f16(x0, a0, a2);
        e4m3x4_to_f16(x1, a1, a3);
        mma_f16_16816(acc.o[2 * j], a0, a1, a2, a3, pa0, pa1);
        e4m3x4_to_f16(x2, a0, a2);
        e4m3x4_to_f16(x3, a1, a3);
        mma_f16_16816(acc.o[2 * j + 1], a0, a1, a2, a3, pa0, pa1);
        e4m3x4_to_f16(y0, a0, a2);
        e4m3x4_to_f16(y1, a1, a3);
        mma_f16_16816(acc.o[2 * j], a0, a1, a2, a3, pb0, pb1);
        e4m3x4_to_f16(y2, a0, a2);
        e4m3x4_to_f16(y3, a1, a3);
        mma_f16_16816(acc.o[2 * j + 1], a0, a1, a2, a3, pb0, pb1);
    }
}

// Gather one 32-token FP8 tile as two 16-token halves: K rows of the
// [blocks * Hkv * B][D] view (box D x 16) and V^T boxes of 16 token columns x D
// rows of the [blocks * Hkv * D][B] view.  With block_size 32 both halves lie
// in one block (rows y0 and y0 + 16); with block_size 16 the second half is
// the next block's (y1, or nothing past the context).  Rows of a half that
// lie past the context are loaded from inside its block and masked later.
template <int D>
__device__ __forceinline__ void issue_rows_f8(const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                              unsigned char *stage, uint64_t *bar, int bshift, TileRows r,
                                              uint32_t extra_bytes = 0) {
    const uint32_t b = smem_u32(bar);
    // extra_bytes: further copies the caller issues on the same barrier
    if (r.y0 < 0) {
        mbar_arrive_expect_tx(bar, extra_bytes);
        return;
    }
    const int y1 = bshift == 5 ? r.y0 + kTile : r.y1;
    mbar_arrive_expect_tx(bar, (uint32_t)((y1 >= 0 ? 2 : 1) * 2 * kTile * D) + extra_bytes);
    const uint32_t dk = smem_u32(stage), dv = dk + 2 * kTile * D;
    const int bh0 = r.y0 >> bshift;  // block * Hkv + kv head
    tma_load_2d(dk, tm_k, b, 0, r.y0);
    tma_load_2d(dv, tm_v, b, r.y0 - (bh0 << bshift), bh0 * D);
    if (y1 >= 0) {
        const int bh1 = y1 >> bshift;
        tma_load_2d(dk + kTile * D, tm_k, b, 0, y1);
        tma_load_2d(dv + kTile * D, tm_v, b, y1 - (bh1 << bshift), bh1 * D);
    }
}

// Fused append, FP8: quantise the new token's bf16 K and V rows (landed in
// `nrow`, K then V) and write the codes over row `row` of the landed 32-token
// tile `sk` and into the cache (the tile's TMA rows y0 / y1).  Lanes 0-7 make
// 16 K codes each (one 16-byte chunk of the K row); lanes 8-15 make 16 V codes
// each, one byte of each of 16 head_dim rows of the transposed V tile (and of
// the V block in the cache).  Kept out of line: it runs once per context and
// would otherwise raise the attention loop's register pressure.
template <int D>
__device__ __noinline__ void patch_new_row_f8(unsigned char *sk, const unsigned char *nrow, int y0, int y1, int row,
                                              int lane, float kscale, float vscale, int B, int bshift,
                                              void *k_cache, void *v_cache) {
    if (lane >= 16) return;
    const bool isv = lane >= 8;
    const int ch = lane & 7;
    const uint4 *src = reinterpret_cast<const uint4 *>(nrow + (isv ? 2 * D : 0) + 32 * ch);
    const uint4 x[2] = {src[0], src[1]};
    uint32_t w[4];
    quantize16(x, isv ? vscale : kscale, w);
    const int sub_rows = B < 2 * kTile ? B : 2 * kTile;  // rows of one TMA sub-box
    const int sub = row >> 4, rr = row & 15;
    const int64_t y = row < sub_rows ? (int64_t)y0 + row : (int64_t)y1 + (row - sub_rows);
    const int64_t bh = y >> bshift, off = y & (B - 1);
    if (!isv) {
        const uint4 codes = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4 *>(sk + sub * kTile * D + rr * D + ((ch ^ (rr & 7)) << 4)) = codes;
        *reinterpret_cast<uint4 *>(static_cast<unsigned char *>(k_cache) + y * D + 16 * ch) = codes;
    } else {
        unsigned char *vt = sk + TileBytes<D, true>::kKV + sub * kTile * D + (16 * ch) * kTile + rr;
        unsigned char *col = static_cast<unsigned char *>(v_cache) + (bh * D + 16 * ch) * B + off;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const unsigned char code = (unsigned char)(w[j >> 2] >> (8 * (j & 3)));
            vt[j * kTile] = code;
            col[(int64_t)j * B] = code;
        }
    }
}

// Store a warp's result for the piece [pa, pb) of segment `seg`: the final
// rows when the piece is the whole segment, otherwise partial slot j.
template <int D>
__device__ __forceinline__ void store_piece(const DecodeArgs &a, WarpAcc<D> &acc, bool empty,
                                            const SegCursor &seg, bool whole, int j, int lane,
                                            float oscale = 1.f) {
    const int r0 = lane >> 2, tq = lane & 3, G = a.group;
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {  // column sums over the 16 token rows
        acc.l0 += __shfl_xor_sync(0xffffffffu, acc.l0, sh);
        acc.l1 += __shfl_xor_sync(0xffffffffu, acc.l1, sh);
    }
    if (empty) {
        acc.m0 = acc.m1 = -INFINITY;
        acc.l0 = acc.l1 = 0.f;
    }
    const int64_t row0 = (int64_t)seg.seq * a.num_heads + seg.kvh * G;
    const float inv0 = acc.l0 > 0.f ? oscale / acc.l0 : 0.f, inv1 = acc.l1 > 0.f ? oscale / acc.l1 : 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int d = 16 * mt + r0 + 8 * (jj >> 1);
            const int g = 2 * tq + (jj & 1);
            if (g >= G) continue;
            const int64_t row = row0 + g;
            if (whole) {
                store_out(static_cast<__nv_bfloat16 *>(a.out) + row * D + d,
                          acc.o[mt][jj] * ((jj & 1) ? inv1 : inv0));
            } else {
                a.part_o[(row * a.max_parts + j) * D + d] = acc.o[mt][jj] * oscale;
            }
        }
    }
    if (!whole && r0 == 0) {
        if (2 * tq < G) {
            a.part_m[(row0 + 2 * tq) * a.max_parts + j] = acc.m0;
            a.part_l[(row0 + 2 * tq) * a.max_parts + j] = acc.l0;
        }
        if (2 * tq + 1 < G) {
            a.part_m[(row0 + 2 * tq + 1) * a.max_parts + j] = acc.m1;
            a.part_l[(row0 + 2 * tq + 1) * a.max_parts + j] = acc.l1;
        }
    }
}

// Merge of a segment's n partials by the warp holding its first tile: for
// every query head of the group, with M = max_j m_j,
//     out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j
// over the partial slots j = 0 .. n-1 in order (the same order whichever warp
// merges), evaluated chunk by chunk with the running maximum (earlier sums
// rescaled when it grows).  Lanes are split evenly over the (padded) heads,
// each owning a run of NV float4 of its head's row.  A warp merges after its
// share is done, when its ring is idle: each lane stages the rows it needs in
// its own kLaneBytes of the ring with cp.async (L2, no registers held), so a
// chunk costs one round trip.
template <int D, int NV, int kLaneBytes>
__device__ __forceinline__ void merge_rows(const float4 *po, const float *pm, const float *pl, int n,
                                           uint2 *dst, uint32_t stage) {
    constexpr int kChunk = kLaneBytes / (16 * NV) < 16 ? kLaneBytes / (16 * NV) : 16;  // partials per round trip
    static_assert(kChunk >= 1, "a lane must stage at least one partial row");
    float M = -INFINITY, L = 0.f;
    float4 acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n; c0 += kChunk) {
        float mj[kChunk], lj[kChunk];
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            if (c0 + r < n) {
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    cp_async16(stage + (r * NV + v) * 16, po + (int64_t)(c0 + r) * (D / 4) + v);
            }
            mj[r] = c0 + r < n ? __ldcg(pm + c0 + r) : -INFINITY;
            lj[r] = c0 + r < n ? __ldcg(pl + c0 + r) : 0.f;
        }
        float cm = -INFINITY;
#pragma unroll
        for (int r = 0; r < kChunk; ++r) cm = fmaxf(cm, mj[r]);
        const float Mn = fmaxf(M, cm);
        if (Mn != M && M != -INFINITY) {  // rescale what the earlier chunks summed
            const float a = exp2f(M - Mn);
            L *= a;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                acc[v].x *= a;
                acc[v].y *= a;
                acc[v].z *= a;
                acc[v].w *= a;
            }
        }
        M = Mn;
        cp_async_wait_all();
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            if (c0 + r < n && mj[r] != -INFINITY) {
                const float w = exp2f(mj[r] - M);
                L += w * lj[r];
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const float4 x = lds128(stage + (r * NV + v) * 16);
                    acc[v].x += w * x.x;
                    acc[v].y += w * x.y;
                    acc[v].z += w * x.z;
                    acc[v].w += w * x.w;
                }
            }
        }
    }
    // every piece empty (all blocks invalid, flagged): L stays 0, zero rows
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v)
        dst[v] = make_uint2(pack_bf16x2(acc[v].x * inv, acc[v].y * inv), pack_bf16x2(acc[v].z * inv, acc[v].w * inv));
}

template <int D, int kLaneBytes>
__device__ __forceinline__ void merge_segment(const float *part_o, const float *part_m, const float *part_l,
                                              __nv_bfloat16 *out, int64_t row0, int G, int max_parts, int n,
                                              int lane, uint32_t ring) {
    const int gp = G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8));
    const int lph = min(32 / gp, D / 4);  // lanes per head
    const int dpl = D / lph;              // head_dim entries per lane
    const int h = lane / lph, part = lane % lph;
    if (h >= G) return;
    const int64_t row = row0 + h;
    const float *pm = part_m + row * max_parts, *pl = part_l + row * max_parts;
    const float4 *po = reinterpret_cast<const float4 *>(part_o + row * max_parts * D + part * dpl);
    uint2 *dst = reinterpret_cast<uint2 *>(out + row * D + part * dpl);
    const uint32_t stage = ring + lane * kLaneBytes;
    switch (dpl / 4) {
        case 1: merge_rows<D, 1, kLaneBytes>(po, pm, pl, n, dst, stage); break;
        case 2: merge_rows<D, 2, kLaneBytes>(po, pm, pl, n, dst, stage); break;
        case 4: merge_rows<D, 4, kLaneBytes>(po, pm, pl, n, dst, stage); break;
        default: merge_rows<D, 8, kLaneBytes>(po, pm, pl, n, dst, stage); break;
    }
}

// Balanced kernel: every warp of the grid takes an equal contiguous share of
// the tile list (at least kMinTilesPerCta tiles) and streams it through its own
// TMA ring.  Where a segment (sequence, kv head) ends inside a share, the warp
// stores its result for that piece -- the final rows if the share holds the
// whole segment, otherwise a partial -- and carries on with the next segment.
// Partials are merged in this kernel: a share cuts at most its first and last segment, and the
// warp holding a split segment's first tile (its share's last segment) merges
// it once the other pieces -- processed at the start of their own shares --
// have flagged their partials.  That is the only wait between warps; it is
// bounded, and every warp it waits for is resident (the grid is one wave,
// launched cooperatively, so a grid that cannot be resident at once is refused
// at launch) and never waits itself.  A merge that gives up writes NaN rows and
// sets PKV_DEVERR_TIMEOUT.
//
// F8: the cache holds E4M3 codes (K rows, V transposed per block); tiles are
// attended by attend_tile_f8 and the queries are loaded by load_q_f16.
template <int D, int NW, int NS, bool F8, bool APPEND>
__global__ void __launch_bounds__(NW * 32, 3)
decode_bf16_streamk_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using Lay = TileBytes<D, F8>;
    constexpr int TT = F8 ? 2 * kTile : kTile;  // tokens per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int kNewBytes = APPEND ? 4 * D : 0;  // one new K row and V row (bf16)
    constexpr int kChunks = D * 2 / 16;            // 16-byte chunks of one bf16 K (or V) row
    constexpr bool has_new = APPEND;
    const StreamKLayout L(D, NW, NS, a.num_seqs, Lay::kStage, kNewBytes);
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + L.bars);
    int2 *ycache = reinterpret_cast<int2 *>(smem + L.ycache);
    uint32_t *mcache = reinterpret_cast<uint32_t *>(smem + L.masks);
    int *scache = reinterpret_cast<int *>(smem + L.srcs);
    int *prefix = reinterpret_cast<int *>(smem + L.prefix);
    __shared__ int warp_sums[NW];
    __shared__ int carry;

    // Programmatic dependent launch.  The prologue below (length scan, row
    // staging, first queries) reads only this call's inputs (lengths, block
    // tables, queries) and writes only shared memory, so it may overlap the
    // previous kernel (the previous call's tail); the wait comes before the
    // first access to the cache (new-token stores, then TMA) and to the
    // workspace.  Kernels that let this one start early must not write those
    // inputs after their trigger.
    grid_launch_dependents();

    const int S = a.num_seqs, Hkv = a.num_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cap = min(a.max_seq_len, a.max_blocks * a.block_size);

    // prefix[s] = tiles of all segments of the sequences before s
    __shared__ int seg_max;  // tiles of the longest segment
    if (threadIdx.x == 0) {
        prefix[0] = 0;
        carry = 0;
        seg_max = 0;
    }
    __syncthreads();
    int my_max = 0;
    // the first kScanAhead passes' lengths, all loads in flight at once (one
    // memory latency instead of one per pass of NW * 32 sequences)
    constexpr int kScanAhead = 4;
    int ahead[kScanAhead];
#pragma unroll
    for (int k = 0; k < kScanAhead; ++k) {
        const int sq = k * NW * 32 + threadIdx.x;
        ahead[k] = sq < S ? a.seq_lens[sq] : 0;
    }
    for (int base = 0, pass = 0; base < S; base += NW * 32, ++pass) {
        const int sq = base + threadIdx.x;
        int v = 0;
        if (sq < S) {
            int raw = ahead[0];
#pragma unroll
            for (int k = 1; k < kScanAhead; ++k)
                if (pass == k) raw = ahead[k];
            if (pass >= kScanAhead) raw = a.seq_lens[sq];
            if ((raw < 0 || raw > cap) && blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_SEQ_LEN);
            const int len = clamp_len(raw, cap);
            v = Hkv * laid_out_tiles((len + TT - 1) / TT);
            my_max = max(my_max, laid_out_tiles((len + TT - 1) / TT));
        }
        int x = v;  // inclusive warp scan
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, sh);
            if (lane >= sh) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        int before = carry;
        for (int k = 0; k < warp; ++k) before += warp_sums[k];
        if (sq < S) prefix[sq + 1] = before + x;
        __syncthreads();
        if (threadIdx.x == NW * 32 - 1) carry = before + x;
        __syncthreads();
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) my_max = max(my_max, __shfl_xor_sync(0xffffffffu, my_max, sh));
    if (lane == 0) atomicMax(&seg_max, my_max);
    __syncthreads();
    {
        // No merge kernel follows: this kernel writes the zero rows of empty
        // contexts (no tile, hence no piece).  CTA c takes sequences c, c + grid, ...
        bool mine = false;
        for (int sq = blockIdx.x; sq < S && !mine; sq += gridDim.x) mine = prefix[sq + 1] == prefix[sq];
        if (mine) {
            grid_dependency_wait();  // `out` may still be read by the previous kernel
            constexpr int kRowChunks = D * 2 / 16;
            for (int sq = blockIdx.x; sq < S; sq += gridDim.x) {
                if (prefix[sq + 1] != prefix[sq]) continue;
                uint4 *row = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) +
                                                       (int64_t)sq * a.num_heads * D);
                for (int i = threadIdx.x; i < a.num_heads * kRowChunks; i += NW * 32)
                    row[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    const int64_t T = prefix[S];
    // Warps that get a share.  A segment of n tiles meets at most
    // ceil(n / share) + 1 shares and has own_slots partial slots, so shares
    // hold at least ceil(seg_max / (own_slots - 1)) tiles; that is at most
    // kMinTilesPerCta, and less when every segment is short, which spreads
    // many short contexts over more warps.
    const int64_t parts = balanced_parts(T, seg_max, a.max_parts, (int64_t)gridDim.x * NW);
    const int64_t gw0 = (int64_t)blockIdx.x * NW;
    if (T == 0 || gw0 >= parts) return;
    const int64_t cta_lo = gw0 * T / parts;
    const int64_t cta_hi = (gw0 + NW < parts ? gw0 + NW : parts) * T / parts;

    // Walk order.  Tiles [lo, hi) are attended from r to hi, then from lo to
    // r.  Normally r = lo; but a warp whose share starts with a short piece
    // (the tail of a segment begun by the previous warp) takes that piece
    // last (r = its end): storing a partial early, while every warp's first
    // tile loads are queued, stalls the warp for many microseconds.  Only when
    // every tile of the CTA has its rows staged (no cursor walks past them).
    const int64_t gw = gw0 + warp;
    const int64_t lo = gw * T / parts, hi = (gw + 1) * T / parts;
    const int ncache = (int)(cta_hi - cta_lo < kYCache ? cta_hi - cta_lo : kYCache);
    SegCursor seg_lo;  // segment of tile lo
    int64_t r = lo;
    SegCursor seg;  // the segment being attended
    uint32_t qb[D / 16][2], qn[D / 16][2];
    float qs0 = 0.f, qs1 = 0.f, qns0 = 0.f, qns1 = 0.f;  // FP8: score factors of qb / qn
    auto load_q = [&](const SegCursor &c, uint32_t(&dst)[D / 16][2], float &f0, float &f1) {
        if constexpr (F8) load_q_f16<D>(a, c.seq, c.kvh, lane, dst, f0, f1);
        else load_q_fragments<D>(a, c.seq, c.kvh, lane, dst);
    };
    // Fused append: the new token of a segment (position len - 1) sits
    // in the segment's last tile; the producer brings its K and V rows into
    // the stage's new-row slot with the tile, and the piece that attends the
    // tile writes them over the tile's stale row.  new_row: the token's row
    // in that tile (-1: no append), read with the piece's queries.
    int new_row = -1, new_row_n = -1;
    auto load_new = [&](const SegCursor &c, int &row) {
        row = -1;
        if (!has_new) return;
        const int64_t last = c.seg_start + c.n - 1;
        if (last < lo || last >= hi) return;
        row = (clamp_len(a.seq_lens[c.seq], cap) - 1) % TT;  // the segment has tiles: len >= 1
    };
    bool qn_loaded = false;  // qn holds the second piece's queries
    // The queries of the first two pieces: fetched now, ahead of the burst of
    // tile loads that every warp issues after the staging below.
    if (gw < parts) {
        seg_lo.seek(prefix, S, Hkv, lo);
        const int64_t first_end = seg_lo.seg_start + seg_lo.n;
        if (first_end < hi && first_end - lo < kRotateTiles * kTile / TT && ncache == cta_hi - cta_lo)
            r = first_end;
        seg = seg_lo;
        if (r != lo) seg.advance_to(prefix, Hkv, r);
        load_q(seg, qb, qs0, qs1);
        load_new(seg, new_row);
        const int64_t end1 = seg.seg_start + seg.n;  // the first piece ends at min(hi, end1)
        if (end1 < hi || r != lo) {
            SegCursor second = seg_lo;
            if (end1 < hi) {
                second = seg;
                second.advance_to(prefix, Hkv, end1);
            }
            load_q(second, qn, qns0, qns1);
            load_new(second, new_row_n);
            qn_loaded = true;
        }
    }

    // Stage the TMA rows and valid-row masks of the CTA's first tiles, so that
    // neither issuing nor attending a tile waits on a global load.  Each thread
    // handles up to kPer tiles and issues all their loads (lengths and block
    // ids, read speculatively and masked afterwards) before using any.
    {
        constexpr int kPer = (kYCache + NW * 32 - 1) / (NW * 32);
        const int B = a.block_size;
        const int boxh = B < TT ? B : TT;
        int sq[kPer], kv[kPer], tl[kPer], ln[kPer], b0[kPer], b1[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = threadIdx.x + u * NW * 32;
            sq[u] = -1;
            if (i < ncache) {
                SegCursor c;
                c.seek(prefix, S, Hkv, cta_lo + i);
                tl[u] = (int)(cta_lo + i - c.seg_start) - kLeadTiles;  // < 0: a lead tile
                if (tl[u] >= 0) {
                    sq[u] = c.seq;
                    kv[u] = c.kvh;
                } else {
                    ycache[i] = make_int2(-1, -1);  // nothing to load or attend
                    mcache[i] = 0u;
                    if (APPEND) scache[i] = -1;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            if (sq[u] < 0) continue;
            const int32_t *bt = a.block_tables + (int64_t)sq[u] * a.max_blocks;
            // the tile's tokens lie inside the clamped length, hence inside the table
            const int lb0 = min(tl[u] * TT / B, a.max_blocks - 1);
            const int lb1 = min((tl[u] * TT + boxh) / B, a.max_blocks - 1);
            ln[u] = a.seq_lens[sq[u]];
            b0[u] = bt[lb0];
            b1[u] = bt[lb1];
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            if (sq[u] < 0) continue;
            const int len = clamp_len(ln[u], cap);
            TileRows r{-1, -1, 0u};
            for (int sb = 0; sb < TT / boxh; ++sb) {
                const int tok = tl[u] * TT + sb * boxh;
                if (tok >= len) break;
                const int lb = tok / B;
                int blk = sb == 0 ? b0[u] : b1[u];
                if (blk >= 0 && blk < a.num_blocks) {
                    r.mask |= low_bits(boxh) << (sb * boxh);
                } else {
                    flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                    blk = 0;
                }
                const int y = (int)(((int64_t)blk * Hkv + kv[u]) * B + (tok - lb * B));
                if (sb == 0) r.y0 = y; else r.y1 = y;
            }
            const int valid = min(TT, len - tl[u] * TT);
            r.mask &= low_bits(valid);
            if (APPEND)  // the segment's last tile carries its new token
                scache[threadIdx.x + u * NW * 32] = (tl[u] + 1) * TT >= len ? sq[u] * Hkv + kv[u] : -1;
            const int i = threadIdx.x + u * NW * 32;
            ycache[i] = make_int2(r.y0, r.y1);
            // bf16: valid rows in bits 16..20 (the fused append reads them)
            mcache[i] = F8 ? r.mask : (r.mask | ((uint32_t)valid << 16));
        }
    }
    unsigned char *ring = smem + warp * NS * Lay::kStage;
    uint64_t *bars = bars_all + warp * NS;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (gw >= parts) return;  // no CTA-wide barrier follows
    grid_dependency_wait();
    const int ntiles = (int)(hi - lo);
    const int boxh = a.block_size < kTile ? a.block_size : kTile;

    // rows/mask of tile t (staged, or computed for tiles past the cache)
    auto rows_of = [&](int64_t t, const SegCursor &c) -> TileRows {
        const int64_t i = t - cta_lo;
        if (i < ncache) {
            const int2 y = ycache[i];
            return TileRows{y.x, y.y, F8 ? mcache[i] : (mcache[i] & 0xffffu)};
        }
        const int tl = (int)(t - c.seg_start) - kLeadTiles;
        if (tl < 0) return TileRows{-1, -1, 0u};  // a lead tile: nothing to load or attend
        return tile_rows<TT>(a, c.seq, c.kvh, tl, clamp_len(a.seq_lens[c.seq], cap));
    };

    // k-th tile in walk order
    const int64_t run1 = hi - r;
    auto tile_at = [&](int k) -> int64_t { return k < run1 ? r + k : lo + (k - run1); };
    SegCursor prod;  // lane 0: segment of the tile being issued (needed past the cache; r == lo then)
    if (lane == 0) prod.seek(prefix, S, Hkv, lo);
    unsigned char *newrows = smem + L.patch + warp * NS * kNewBytes;
    auto issue = [&](int k, int buf) {
        const int64_t t = tile_at(k);
        const bool cached = t - cta_lo < ncache;
        if (!cached) prod.advance_to(prefix, Hkv, t);
        // fused append: the segment's last tile also brings the new token's K and V rows
        int64_t src = -1;
        if constexpr (APPEND)
            src = cached ? scache[t - cta_lo]
                         : (t == prod.seg_start + prod.n - 1 ? (int64_t)prod.seq * Hkv + prod.kvh : -1);
        if constexpr (F8)
            issue_rows_f8<D>(&tm_k, &tm_v, ring + buf * Lay::kStage, &bars[buf], a.f8_bshift, rows_of(t, prod),
                             src >= 0 ? kNewBytes : 0u);
        else
            issue_rows<D>(&tm_k, &tm_v, ring + buf * Lay::kStage, &bars[buf], boxh, rows_of(t, prod),
                          src >= 0 ? kNewBytes : 0u);
        if (APPEND && src >= 0) {
            const uint32_t dst = smem_u32(newrows + buf * kNewBytes), b = smem_u32(&bars[buf]);
            bulk_load(dst, static_cast<const __nv_bfloat16 *>(a.k_new) + src * D, 2 * D, b);
            bulk_load(dst + 2 * D, static_cast<const __nv_bfloat16 *>(a.v_new) + src * D, 2 * D, b);
        }
    };
    if (lane == 0) {
        for (int i = 0; i < NS && i < ntiles; ++i) issue(i, i);
    }

    int k = 0;
    bool dead = false;
    WarpAcc<D> acc;
    int64_t merge_seg = -1;  // the split segment this warp merges (its share's last), if any
    int merge_n = 0;
    for (;;) {
        const int64_t pa = tile_at(k);  // this piece: tiles [pa, pb), walk positions [k, kend)
        const int64_t seg_end = seg.seg_start + seg.n;
        const int64_t run_end = k < run1 ? hi : r;
        const int64_t pb = run_end < seg_end ? run_end : seg_end;
        const int kend = k + (int)(pb - pa);
        SegCursor nxt = seg;
        if (kend < ntiles) {  // fetch the next piece's queries while this one runs
            const int64_t tn = tile_at(kend);
            if (tn == pb) nxt.advance_to(prefix, Hkv, tn);
            else nxt = seg_lo;  // the walk wraps to lo
            if (!qn_loaded) {
                load_q(nxt, qn, qns0, qns1);
                load_new(nxt, new_row_n);
            }
            qn_loaded = false;
        }
        acc.reset();
        for (; k < kend; ++k) {
            const int buf = k % NS;
            if (!dead && !mbar_wait_bounded(&bars[buf], (uint32_t)((k / NS) & 1))) {
                if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
                dead = true;
            }
            if (dead) continue;
            const int64_t t = tile_at(k);
            const TileRows rw = rows_of(t, seg);
            unsigned char *sk = ring + buf * Lay::kStage;
            if (APPEND && F8 && new_row >= 0 && t == seg.seg_start + seg.n - 1 && ((rw.mask >> new_row) & 1u)) {
                patch_new_row_f8<D>(sk, newrows + buf * kNewBytes, rw.y0, rw.y1, new_row, lane, a.f8_kscale,
                                    a.f8_vscale, a.block_size, a.f8_bshift, a.k_cache_w, a.v_cache_w);
                __syncwarp();
            }
            if (APPEND && !F8 && new_row >= 0 && t == seg.seg_start + seg.n - 1 && ((rw.mask >> new_row) & 1u)) {
                // The new token: its rows, landed in the stage's new-row slot,
                // overwrite the tile's row (the stale slot the TMA brought)
                // before the tile is attended, and are stored to the cache for
                // later calls.  Nothing in this call reads that cache row: only
                // this warp attends the tile.
                if (lane < 2 * kChunks) {
                    const uint4 nv = *reinterpret_cast<const uint4 *>(newrows + buf * kNewBytes + lane * 16);
                    const int ch = lane % kChunks, h = ch >> 3, c = ch & 7;
                    *reinterpret_cast<uint4 *>(sk + (lane < kChunks ? 0 : Lay::kKV) + h * (kTile * 128) +
                                               new_row * 128 + ((c ^ (new_row & 7)) << 4)) = nv;
                    const int64_t dst = new_row < boxh ? (int64_t)rw.y0 + new_row : (int64_t)rw.y1 + (new_row - boxh);
                    static_cast<uint4 *>(lane < kChunks ? a.k_cache_w : a.v_cache_w)[dst * kChunks + ch] = nv;
                }
                __syncwarp();
            }
            if (rw.mask != 0u) {  // lead tiles have no rows
                if constexpr (F8)
                    attend_tile_f8<D>(sk, sk + Lay::kKV, rw.mask, qb, qs0, qs1, acc, lane);
                else
                    attend_tile<D>(sk, sk + Lay::kKV, rw.mask, qb, a.scale_log2, acc, lane);
            }
            __syncwarp();
            if (lane == 0 && k + NS < ntiles) {
                fence_proxy_async();
                issue(k + NS, buf);
            }
        }
        const bool whole = pa == seg.seg_start && pb == seg_end;
        const int64_t w0 = share_owner(seg.seg_start, T, parts);
        store_piece<D>(a, acc, dead, seg, whole, (int)(gw - w0), lane, F8 ? a.f8_vscale : 1.f);
        if (!whole) {
            // Split segment: the warp holding its first tile merges it (the
            // segment is the last of that warp's share, so the merge waits for
            // nothing but pieces processed at the start of other shares); every
            // other piece announces its partial.
            const int n = (int)(share_owner(seg_end - 1, T, parts) - w0 + 1);
            const int64_t sg = (int64_t)seg.seq * Hkv + seg.kvh;
            if (gw == w0) {
                merge_seg = sg;
                merge_n = n;
            } else {
                fence_acq_rel_gpu();
                __syncwarp();
                if (lane == 0)
                    *reinterpret_cast<volatile unsigned long long *>(a.flags + sg * a.max_parts + (gw - w0)) = a.tag;
            }
        }
        if (kend >= ntiles) break;
        seg = nxt;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qb[ks][0] = qn[ks][0];
            qb[ks][1] = qn[ks][1];
        }
        qs0 = qns0;
        qs1 = qns1;
        new_row = new_row_n;
    }
    if (merge_seg >= 0) {
        // Wait (bounded) until the other pieces' flags carry this call's tag,
        // merge through the now idle ring, then clear the flags so that a
        // replay with the same tag waits again.
        unsigned long long *fl = a.flags + merge_seg * a.max_parts;
        // this warp's own partial (slot 0) is read back by its own lanes: the
        // warp barrier orders those stores before the reads
        __syncwarp();
        const bool ready = wait_flags_bounded(fl + 1, merge_n - 1, a.tag, lane);
        const int sq = (int)(merge_seg / Hkv), kvh = (int)(merge_seg - (int64_t)sq * Hkv);
        const int64_t row0 = (int64_t)sq * a.num_heads + kvh * a.group;
        if (ready) {
            merge_segment<D, NS * Lay::kStage / 32>(a.part_o, a.part_m, a.part_l, static_cast<__nv_bfloat16 *>(a.out),
                                                    row0, a.group, a.max_parts, merge_n, lane, smem_u32(ring));
        } else {
            // a piece never came: NaN rows rather than a merge over stale slots
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + row0 * D;
            for (int i = lane; i < a.group * D; i += 32) o[i] = __ushort_as_bfloat16((unsigned short)0x7fc0);
        }
        for (int j = 1 + lane; j < merge_n; j += 32) fl[j] = 0ull;
    }
}

// Store each sequence's new token at position seq_lens[s] - 1 (looked up in
// its block table): the write half of paged_attention_decode_append on the
// paths that do not fuse it.  One thread per 16-byte chunk of K and of V.
__global__ void __launch_bounds__(256)
append_tokens_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, uint4 *k_cache,
                     uint4 *v_cache, const int32_t *__restrict__ block_tables,
                     const int32_t *__restrict__ seq_lens, int num_seqs, int num_kv_heads, int chunks,
                     int block_size, int max_blocks, int num_blocks, int cap, unsigned int *err) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t total = (int64_t)num_seqs * num_kv_heads * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sh = i / chunks;
        const int c = (int)(i - sh * chunks);
        const int s = (int)(sh / num_kv_heads), h = (int)(sh - (int64_t)s * num_kv_heads);
        const int len = clamp_len(seq_lens[s], cap);
        if (len == 0) continue;
        const int pos = len - 1, lb = pos / block_size;
        const int blk = block_tables[(int64_t)s * max_blocks + lb];
        if (blk < 0 || blk >= num_blocks) {
            if (c == 0) flag_error(err, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        const int64_t row = ((int64_t)blk * num_kv_heads + h) * block_size + (pos - lb * block_size);
        k_cache[row * chunks + c] = k_new[i];
        v_cache[row * chunks + c] = v_new[i];
    }
}

// ---------------------------------------------------------------------------
// CUDA-core kernel (fp32 I/O; also instantiated for bf16 storage)
// ---------------------------------------------------------------------------
template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32) decode_simt_kernel(const DecodeArgs a) {
    constexpr int E = D / 32;  // head_dim elements per lane: d = lane + 32 j
    __shared__ float merge_buf[NW][kGMax * D + 2 * kGMax];
    grid_dependency_wait();
    grid_launch_dependents();

    WorkItem w;
    if (!resolve_item(a, w)) return;
    if (w.len == 0) {
        write_zero_rows<T, D>(a, w);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group, Hkv = a.num_kv_heads, B = a.block_size;

    float qf[kGMax][E], o[kGMax][E], m[kGMax], l[kGMax];
    const T *qbase = static_cast<const T *>(a.q) + ((int64_t)w.seq * a.num_heads + w.kvh * G) * D;
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            qf[g][j] = g < G ? to_float(qbase[g * D + lane + 32 * j]) : 0.f;
            o[g][j] = 0.f;
        }
    }
    const T *kc = static_cast<const T *>(a.k_cache);
    const T *vc = static_cast<const T *>(a.v_cache);
    const int32_t *bt = a.block_tables + (int64_t)w.seq * a.max_blocks;

    for (int t = w.tok_begin + warp; t < w.tok_end; t += NW) {
        const int lb = t / B;
        const int blk = bt[lb];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        const int64_t row = (((int64_t)blk * Hkv + w.kvh) * B + (t - lb * B)) * D;
        float kf[E], vf[E];
#pragma unroll
        for (int j = 0; j < E; ++j) {
            kf[j] = to_float(kc[row + lane + 32 * j]);
            vf[j] = to_float(vc[row + lane + 32 * j]);
        }
#pragma unroll
        for (int g = 0; g < kGMax; ++g) {
            if (g >= G) break;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) dot = fmaf(qf[g][j], kf[j], dot);
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
            const float x = dot * a.scale;
            const float mn = fmaxf(m[g], x);
            const float al = expf(m[g] - mn);
            const float p = expf(x - mn);
            l[g] = l[g] * al + p;
#pragma unroll
            for (int j = 0; j < E; ++j) o[g][j] = fmaf(p, vf[j], o[g][j] * al);
            m[g] = mn;
        }
    }

    float *mine = merge_buf[warp];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
#pragma unroll
        for (int j = 0; j < E; ++j) mine[g * D + lane + 32 * j] = o[g][j];
        if (lane == 0) {
            mine[kGMax * D + g] = m[g];
            mine[kGMax * D + kGMax + g] = l[g];
        }
    }
    __syncthreads();
    const float *bufs[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) bufs[k] = merge_buf[k];
    merge_warps_and_store<T, D, NW, false>(a, w, bufs);
}

// ---------------------------------------------------------------------------
// Partition merge (fixed partitions): out = sum_j e^{m_j - M} o_j / sum_j
// e^{m_j - M} l_j over the ceil(len / P) partials of each (sequence, head).
// ---------------------------------------------------------------------------
template <typename T, int D, bool LOG2>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeArgs a) {
    constexpr int E = D / 32;  // consecutive head_dim elements per lane
    constexpr int U = 8;       // partials whose rows are loaded together
    grid_dependency_wait();
    // the next kernel may start its prologue (it waits before touching what this
    // one writes); only for merges of at most one CTA per SM, whose CTAs leave
    // the next kernel room instead of competing with it for every SM
    if (a.merge_trigger) grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;  // (sequence, query head)
    if (row >= (int64_t)a.num_seqs * a.num_heads) return;
    const int seq = (int)(row / a.num_heads);
    const int cap = min(a.max_seq_len, a.max_blocks * a.block_size);
    const float *pm = a.part_m + row * a.max_parts;
    const float *pl = a.part_l + row * a.max_parts;
    const float *po = a.part_o + row * a.max_parts * D + lane * E;
    // issue the length and the first 32 (max, sum) pairs at once; pairs past
    // the partition count are masked below
    const int raw_len = a.seq_lens[seq];
    float mj = -INFINITY, lj = 0.f;
    if (lane < a.max_parts) {
        mj = pm[lane];
        lj = pl[lane];
    }
    const int len = raw_len < 0 ? 0 : (raw_len > cap ? cap : raw_len);
    T *dst = static_cast<T *>(a.out) + row * D + lane * E;
    const int total = (len + a.partition_size - 1) / a.partition_size;
    if (total <= 1) return;
    if (lane >= total) {
        mj = -INFINITY;
        lj = 0.f;
    }
    float M = mj;
    for (int j = lane + 32; j < total; j += 32) M = fmaxf(M, pm[j]);
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
    if (M == -INFINITY) M = 0.f;  // only if every block was invalid (flagged)
    auto ex = [&](float x) { return x == -INFINITY ? 0.f : (LOG2 ? exp2f(x - M) : expf(x - M)); };
    const float wl = ex(mj);  // weight of partial `lane`
    float lsum = wl * lj;
    for (int j = lane + 32; j < total; j += 32) lsum += ex(pm[j]) * pl[j];
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, sh);

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int j0 = 0; j0 < total; j0 += U) {
        float v[U][E];
#pragma unroll
        for (int u = 0; u < U; ++u) {  // U independent row loads in flight
            const int j = j0 + u < total ? j0 + u : total - 1;
#pragma unroll
            for (int e = 0; e < E; ++e) v[u][e] = po[(int64_t)j * D + e];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u;
            const float wsh = __shfl_sync(0xffffffffu, wl, j & 31);
            const float w = j >= total ? 0.f : (j < 32 ? wsh : ex(pm[j]));
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] += w * v[u][e];
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) store_out(dst + e, lsum > 0.f ? acc[e] / lsum : 0.f);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Fixed partitions used when the caller passes partition_size = 0 but the
// balanced path does not apply (fp32, or more sequences than it scans).
constexpr int kDefaultPartition = 512;
constexpr int kMaxBalancedSeqs = 8192;

struct WorkspaceLayout {
    size_t o_off, m_off, l_off, flags_off, total;
};

// parts = partial slots per (sequence, query head); `flags` adds the ready
// flags of the balanced path's in-kernel merge, 8 bytes per slot.
static WorkspaceLayout workspace_layout(int64_t S, int64_t Hq, int64_t D, int64_t parts, bool flags) {
    WorkspaceLayout w;
    w.o_off = 0;
    w.m_off = round256((size_t)(S * Hq * parts * D * 4));
    w.l_off = w.m_off + round256((size_t)(S * Hq * parts * 4));
    w.flags_off = w.l_off + round256((size_t)(S * Hq * parts * 4));
    w.total = w.flags_off + (flags ? round256((size_t)(S * Hq * parts * 8)) : 0);
    return w;
}

// Balanced path: a segment of L tokens spans at most ceil(L / 256) + 1 shares
// because every share holds at least kMinTilesPerCta tiles (256 tokens).
static int64_t balanced_slots(int max_seq_len) {
    return ((int64_t)max_seq_len + kMinTilesPerCta * kTile - 1) / (kMinTilesPerCta * kTile) + 1;
}

static bool make_cache_maps(const DecodeArgs &a, int D, CUtensorMap *mk, CUtensorMap *mv) {
    const int boxh = a.block_size < kTile ? a.block_size : kTile;
    const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * a.block_size;
    return make_cache_map(mk, a.k_cache, rows, D, boxh) && make_cache_map(mv, a.v_cache, rows, D, boxh);
}

// Launch shapes (warps per CTA x ring stages per warp): the shapes measured
// fastest on GB300 (4 warps x 2 stages for the fixed-partition and balanced
// kernels, bf16 and FP8).
template <int D, int NW, int NS>
static pkv_status launch_bf16(const DecodeArgs &a, dim3 grid, cudaStream_t st) {
    static bool done[128] = {};
    constexpr int smem = bf16_smem_bytes<D, NW, NS>();
    auto kern = decode_bf16_mma_kernel<D, NW, NS>;
    if (!ensure_smem(kern, smem, done)) return PKV_ERR_CUDA;
    CUtensorMap mk, mv;
    if (!make_cache_maps(a, D, &mk, &mv)) return PKV_ERR_CUDA;
    return launch_pdl(kern, grid, dim3(NW * 32), smem, st, mk, mv, a);
}

template <int D>
static pkv_status dispatch_bf16(const DecodeArgs &a, dim3 grid, cudaStream_t st) {
    return launch_bf16<D, 4, 2>(a, grid, st);
}

template <int D, int NW, int NS, bool APPEND>
static pkv_status launch_balanced(const DecodeArgs &a, cudaStream_t st) {
    static bool done[128] = {};
    auto kern = decode_bf16_streamk_kernel<D, NW, NS, false, APPEND>;
    constexpr int stage = TileBytes<D, false>::kStage, nb = APPEND ? 4 * D : 0;
    if (!ensure_smem(kern, StreamKLayout(D, NW, NS, kMaxBalancedSeqs, stage, nb).total, done)) return PKV_ERR_CUDA;
    const int smem = StreamKLayout(D, NW, NS, a.num_seqs, stage, nb).total;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem) != cudaSuccess ||
        per_sm < 1)
        return PKV_ERR_CUDA;
    const int sms = sm_count();
    if (sms < 1) return PKV_ERR_CUDA;
    CUtensorMap mk, mv;
    if (!make_cache_maps(a, D, &mk, &mv)) return PKV_ERR_CUDA;
    // every CTA resident at once: the in-kernel merge waits on other CTAs
    static std::atomic<int> mode{-1};
    return launch_resident(mode, kern, dim3((unsigned)(sms * per_sm)), dim3(NW * 32), smem, st, mk, mv, a);
}

template <int D>
static pkv_status dispatch_balanced(const DecodeArgs &a, cudaStream_t st) {
    return a.k_new ? launch_balanced<D, 4, 2, true>(a, st) : launch_balanced<D, 4, 2, false>(a, st);
}

// FP8 cache views.  K: [blocks * Hkv * B][D] bytes, box D x 16 rows, 128-byte
// swizzle.  V (transposed per block): [blocks * Hkv * D][B] bytes, box 16
// token columns x D rows, unswizzled (a row of the box is one 16-byte vector).
static bool make_f8_maps(const DecodeArgs &a, int D, CUtensorMap *mk, CUtensorMap *mv) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t nbh = (int64_t)a.num_blocks * a.num_kv_heads;
    cuuint32_t estr[2] = {1u, 1u};
    cuuint64_t kdims[2] = {(cuuint64_t)D, (cuuint64_t)(nbh * a.block_size)};
    cuuint64_t kstr[1] = {(cuuint64_t)D};
    cuuint32_t kbox[2] = {(cuuint32_t)D, (cuuint32_t)kTile};
    if (enc(mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(a.k_cache), kdims, kstr, kbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    cuuint64_t vdims[2] = {(cuuint64_t)a.block_size, (cuuint64_t)(nbh * D)};
    cuuint64_t vstr[1] = {(cuuint64_t)a.block_size};
    cuuint32_t vbox[2] = {(cuuint32_t)kTile, (cuuint32_t)D};
    return enc(mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(a.v_cache), vdims, vstr, vbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int NW, int NS, bool APPEND>
static pkv_status launch_balanced_f8(const DecodeArgs &a, cudaStream_t st) {
    static bool done[128] = {};
    auto kern = decode_bf16_streamk_kernel<D, NW, NS, true, APPEND>;
    constexpr int stage = TileBytes<D, true>::kStage, nb = APPEND ? 4 * D : 0;
    if (!ensure_smem(kern, StreamKLayout(D, NW, NS, kMaxBalancedSeqs, stage, nb).total, done)) return PKV_ERR_CUDA;
    const int smem = StreamKLayout(D, NW, NS, a.num_seqs, stage, nb).total;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem) != cudaSuccess ||
        per_sm < 1)
        return PKV_ERR_CUDA;
    const int sms = sm_count();
    if (sms < 1) return PKV_ERR_CUDA;
    CUtensorMap mk, mv;
    if (!make_f8_maps(a, D, &mk, &mv)) return PKV_ERR_CUDA;
    // every CTA resident at once: the in-kernel merge waits on other CTAs
    static std::atomic<int> mode{-1};
    return launch_resident(mode, kern, dim3((unsigned)(sms * per_sm)), dim3(NW * 32), smem, st, mk, mv, a);
}

static pkv_status dispatch_balanced_f8(const DecodeArgs &a, cudaStream_t st) {
    return a.k_new ? launch_balanced_f8<128, 4, 2, true>(a, st) : launch_balanced_f8<128, 4, 2, false>(a, st);
}

template <typename T, int D>
static pkv_status dispatch_simt(const DecodeArgs &a, dim3 grid, cudaStream_t st) {
    return launch_pdl(decode_simt_kernel<T, D, 4>, grid, dim3(128), 0, st, a);
}

template <typename T, int D, bool LOG2>
static pkv_status launch_reduce(const DecodeArgs &a, cudaStream_t st) {
    const int64_t rows = (int64_t)a.num_seqs * a.num_heads;
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    DecodeArgs m = a;
    m.merge_trigger = (int64_t)blocks <= (int64_t)sm_count() ? 1 : 0;
    return launch_pdl(decode_reduce_kernel<T, D, LOG2>, dim3(blocks), dim3(128), 0, st, m);
}

}  // namespace pkv

using namespace pkv;

PKV_API size_t paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim,
                                              int max_seq_len, int partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
    if (partition_size < 0 || partition_size % kTile != 0) return 0;
    if (partition_size == 0) {
        // large enough for the balanced path and for its fixed-partition fallback
        return workspace_layout(num_seqs, num_heads, head_dim, balanced_slots(max_seq_len), true).total;
    }
    const int64_t parts = ((int64_t)max_seq_len + partition_size - 1) / partition_size;
    if (parts <= 1) return 0;
    return workspace_layout(num_seqs, num_heads, head_dim, parts, false).total;
}

namespace pkv {

// The store of each sequence's new token at position seq_lens[s] - 1 (looked
// up in its block table), for the paths that do not fuse it into attention.
pkv_status append_new_tokens(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                                int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                                int num_blocks, int max_seq_len, int dtype, cudaStream_t st) {
    if (num_kv_heads < 1 || max_blocks_per_seq < 1 || num_blocks < 1 || max_seq_len < 0)
        return PKV_ERR_INVALID;
    if (!k_cache || !v_cache || !block_tables || !seq_lens || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID;
    const int elt = dtype == PKV_F32 ? 4 : 2;
    const int chunks = head_dim * elt / 16;
    const int64_t total = (int64_t)num_seqs * num_kv_heads * chunks;
    const int64_t blocks = (total + 255) / 256;
    const int cap = (int)std::min<int64_t>(max_seq_len, (int64_t)max_blocks_per_seq * block_size);
    return launch_pdl(append_tokens_kernel, dim3((unsigned)(blocks < 65536 ? blocks : 65536)), dim3(256), 0, st,
                      (const uint4 *)k_new, (const uint4 *)v_new, (uint4 *)k_cache, (uint4 *)v_cache,
                      block_tables, seq_lens, num_seqs, num_kv_heads, chunks, block_size, max_blocks_per_seq,
                      num_blocks, cap, device_error_word());
}

}  // namespace pkv

static pkv_status decode_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
                              int partition_size, void *workspace, size_t workspace_bytes, int dtype,
                              void *stream, const void *k_new, const void *v_new) {
    if (num_seqs < 0 || num_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 ||
        num_blocks < 1 || max_seq_len < 0 || partition_size < 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
    if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > kGMax) return PKV_ERR_UNSUPPORTED;
    if (partition_size % kTile != 0) return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID;
    // TMA row coordinates are 32-bit: every (block, kv head, row) must be addressable.
    const int64_t rows = ((int64_t)num_blocks + 1) * num_kv_heads * block_size;
    if (rows > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PKV_ERR_INVALID;
    // the balanced path counts tiles of all segments in 32-bit integers
    if ((int64_t)num_seqs * num_kv_heads * ((max_seq_len + kTile - 1) / kTile + kLeadTiles) > INT32_MAX / 2)
        return PKV_ERR_UNSUPPORTED;

    const bool balanced = partition_size == 0 && dtype == PKV_BF16 && max_seq_len > 0 &&
                          num_seqs <= kMaxBalancedSeqs;
    const int P = partition_size > 0 ? partition_size : kDefaultPartition;
    const int64_t parts64 = max_seq_len > P ? ((int64_t)max_seq_len + P - 1) / P : 1;
    if (parts64 > 65535) return PKV_ERR_INVALID;
    const int parts = (int)parts64;

    DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_heads / num_kv_heads;
    a.block_size = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.partition_size = P;
    a.max_parts = parts;
    a.scale = scale;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.err = device_error_word();
    a.k_new = balanced ? k_new : nullptr;
    a.v_new = balanced ? v_new : nullptr;
    a.k_cache_w = const_cast<void *>(k_cache);
    a.v_cache_w = const_cast<void *>(v_cache);

    const bool split = balanced || parts > 1;
    if (split) {
        // partition_size == 0 sizes the workspace for the balanced layout (which
        // also holds the fixed-partition fallback); otherwise fixed partitions
        const int64_t slots = partition_size == 0 ? balanced_slots(max_seq_len) : parts;
        const WorkspaceLayout lay = workspace_layout(num_seqs, num_heads, head_dim, slots, partition_size == 0);
        if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return PKV_ERR_INVALID;
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        a.part_o = reinterpret_cast<float *>(ws + lay.o_off);
        a.part_m = reinterpret_cast<float *>(ws + lay.m_off);
        a.part_l = reinterpret_cast<float *>(ws + lay.l_off);
        if (balanced) {  // the attention kernel merges split contexts itself
            a.flags = reinterpret_cast<unsigned long long *>(ws + lay.flags_off);
            a.tag = next_call_tag();
        }
        a.max_parts = (int)slots;  // stride of the partial slots
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid((unsigned)num_seqs, (unsigned)num_kv_heads, (unsigned)parts);
    pkv_status rc;
    if (balanced) {
        rc = head_dim == 128 ? dispatch_balanced<128>(a, st) : dispatch_balanced<64>(a, st);
    } else if (dtype == PKV_BF16) {
        rc = head_dim == 128 ? dispatch_bf16<128>(a, grid, st) : dispatch_bf16<64>(a, grid, st);
        if (rc == PKV_OK && parts > 1)
            rc = head_dim == 128 ? launch_reduce<__nv_bfloat16, 128, true>(a, st)
                                 : launch_reduce<__nv_bfloat16, 64, true>(a, st);
    } else {
        rc = head_dim == 128 ? dispatch_simt<float, 128>(a, grid, st) : dispatch_simt<float, 64>(a, grid, st);
        if (rc == PKV_OK && parts > 1)
            rc = head_dim == 128 ? launch_reduce<float, 128, false>(a, st)
                                 : launch_reduce<float, 64, false>(a, st);
    }
    return rc;
}

static pkv_status decode_fp8_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                                  int num_heads, int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
                                  float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                                  void *stream, const void *k_new, const void *v_new) {
    if (num_seqs < 0 || num_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        max_seq_len < 0 || !std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale) ||
        !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > kGMax) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > kMaxBalancedSeqs) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID;
    // TMA row coordinates are 32-bit: K rows (block, head, token) and V^T rows (block, head, dim)
    if (((int64_t)num_blocks + 1) * num_kv_heads * std::max(block_size, head_dim) > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PKV_ERR_INVALID;
    if ((int64_t)num_seqs * num_kv_heads * ((max_seq_len + kTile - 1) / kTile + kLeadTiles) > INT32_MAX / 2)
        return PKV_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (max_seq_len == 0)  // every context is empty: all-zero rows
        return cudaMemsetAsync(out, 0, (size_t)num_seqs * num_heads * head_dim * 2, st) == cudaSuccess
                   ? PKV_OK : PKV_ERR_CUDA;
    const int64_t slots = balanced_slots(max_seq_len);
    const WorkspaceLayout lay = workspace_layout(num_seqs, num_heads, head_dim, slots, true);
    if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_INVALID;

    DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_heads / num_kv_heads;
    a.block_size = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.partition_size = kDefaultPartition;
    a.scale = scale;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.f8_kscale_log2 = (float)((double)scale * (double)k_scale * 1.4426950408889634);
    a.f8_kscale = k_scale;
    a.f8_vscale = v_scale;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache_w = const_cast<void *>(k_cache);
    a.v_cache_w = const_cast<void *>(v_cache);
    a.f8_bshift = block_size == 16 ? 4 : 5;
    a.err = device_error_word();
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.part_o = reinterpret_cast<float *>(ws + lay.o_off);
    a.part_m = reinterpret_cast<float *>(ws + lay.m_off);
    a.part_l = reinterpret_cast<float *>(ws + lay.l_off);
    a.flags = reinterpret_cast<unsigned long long *>(ws + lay.flags_off);
    a.tag = next_call_tag();
    a.max_parts = (int)slots;
    return dispatch_balanced_f8(a, st);
}

PKV_API pkv_status paged_attention_decode_fp8(void *out, const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_tables,
                                              const int32_t *seq_lens, int num_seqs, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                              float scale, float k_scale, float v_scale, void *workspace,
                                              size_t workspace_bytes, void *stream) {
    return decode_fp8_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads,
                           head_dim, block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale, k_scale,
                           v_scale, workspace, workspace_bytes, stream, nullptr, nullptr);
}

PKV_API pkv_status paged_attention_decode_append_fp8(void *out, const void *q, const void *k_new,
                                                     const void *v_new, void *k_cache, void *v_cache,
                                                     const int32_t *block_tables, const int32_t *seq_lens,
                                                     int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                     int block_size, int max_blocks_per_seq, int num_blocks,
                                                     int max_seq_len, float scale, float k_scale, float v_scale,
                                                     void *workspace, size_t workspace_bytes, void *stream) {
    if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID;
    // every context holds at least its new token
    if (num_seqs > 0 && max_seq_len < 1) return PKV_ERR_INVALID;
    return decode_fp8_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads,
                           head_dim, block_size, max_blocks_per_seq, num_blocks, max_seq_len, scale, k_scale,
                           v_scale, workspace, workspace_bytes, stream, k_new, v_new);
}

PKV_API pkv_status paged_attention_decode(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *seq_lens, int num_seqs, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                          float scale, int partition_size, void *workspace,
                                          size_t workspace_bytes, int dtype, void *stream) {
    return decode_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, max_seq_len,
                       scale, partition_size, workspace, workspace_bytes, dtype, stream, nullptr, nullptr);
}

PKV_API pkv_status paged_attention_decode_append(
    void *out, const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
    const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int num_heads, int num_kv_heads,
    int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale,
    int partition_size, void *workspace, size_t workspace_bytes, int dtype, void *stream) {
    if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID;
    // The balanced path stores the new tokens inside the attention kernel (also
    // for batches of many (sequence, kv head) segments: with the merge inside
    // the attention kernel, 256 x 8 segments ran 66.6 us fused against 70.1 us
    // with a separate store kernel).
    const bool fused = partition_size == 0 && dtype == PKV_BF16 && num_seqs > 0 &&
                       num_seqs <= kMaxBalancedSeqs && max_seq_len > 0;
    if (!fused) {
        // other paths: the plain write (slot of position seq_lens[s] - 1 is
        // looked up on the device) followed by the decode
        if (num_seqs == 0) return PKV_OK;
        if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
        if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
        if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
        const pkv_status rc = append_new_tokens(k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                                            num_seqs, num_kv_heads, head_dim, block_size,
                                            max_blocks_per_seq, num_blocks, max_seq_len, dtype,
                                            static_cast<cudaStream_t>(stream));
        if (rc != PKV_OK) return rc;
        return paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                      num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                      num_blocks, max_seq_len, scale, partition_size, workspace,
                                      workspace_bytes, dtype, stream);
    }
    return decode_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, max_seq_len,
                       scale, partition_size, workspace, workspace_bytes, dtype, stream, k_new, v_new);
}

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace (paged_attention_decode_noalloc).
// For callers that cannot allocate device memory, the split-K partials live
// in this array, compiled into the library and resident on every device that
// loads it until the process exits.  Host code must not use the symbol's
// name as a device address (on the host it is only a stand-in); the device
// address is looked up once per device below.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current CUDA context, looked up
// on the first call in that context (with the device current) and cached per
// device together with the context it was taken in: a call from another
// context (a non-primary context, or a primary context created again after
// cudaDeviceReset) looks the address up again.  nullptr on failure.
static void *noalloc_scratch_address() {
    static std::mutex mu;
    static void *ptrs[128] = {};
    static CUcontext ctxs[128] = {};
    static PFN_cuCtxGetCurrent_v4000 get_ctx = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuCtxGetCurrent_v4000) nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    if (!get_ctx) return nullptr;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ctx || !ptrs[dev] || ctxs[dev] != ctx) {
        // (the lookup makes the device's primary context current if none is)
        void *p = nullptr;
        if (cudaGetSymbolAddress((void **)&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
        ptrs[dev] = p;
        ctxs[dev] = ctx;
    }
    return ptrs[dev];
}

PKV_API pkv_status paged_attention_decode_noalloc(void *out, const void *q, const void *k_cache,
                                                  const void *v_cache, const int32_t *block_tables,
                                                  const int32_t *seq_lens, int num_seqs, int num_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int max_blocks_per_seq, int num_blocks,
                                                  int max_seq_len, float scale, int partition_size,
                                                  int dtype, void *stream) {
    if (partition_size < 0 || partition_size % kTile != 0) return PKV_ERR_INVALID;
    const int P = partition_size > 0 ? partition_size : 512;
    const size_t need = paged_attention_workspace_size(num_seqs, num_heads, head_dim, max_seq_len, P);
    if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_TOO_LARGE;
    void *scratch = nullptr;
    if (need > 0) {
        scratch = noalloc_scratch_address();
        if (!scratch) return PKV_ERR_CUDA;
    }
    return paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                  num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                  num_blocks, max_seq_len, scale, P, scratch,
                                  need > 0 ? PKV_NOALLOC_SCRATCH_BYTES : 0, dtype, stream);
}

// ---------------------------------------------------------------------------
// Failure detection: the two bounded waits of the attention kernels, run once
// by one warp with a caller-chosen poll limit.
// ---------------------------------------------------------------------------
namespace pkv {
__global__ void __launch_bounds__(32) bounded_wait_kernel(const unsigned long long *flags, int n, unsigned long long tag,
                                                          int arrive, uint32_t polls, unsigned int *err) {
    __shared__ uint64_t bar;
    const int lane = threadIdx.x;
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (n > 0 && !wait_flags_bounded(flags, n, tag, lane, polls) && lane == 0) flag_error(err, PKV_DEVERR_TIMEOUT);
    if (lane == 0) {
        if (arrive) mbar_arrive(&bar);
        if (!mbar_wait_bounded(&bar, 0u, polls)) flag_error(err, PKV_DEVERR_TIMEOUT);
    }
}
}  // namespace pkv

PKV_API pkv_status pkv_bounded_wait_check(const uint64_t *flags, int n_flags, uint64_t tag, int arrive, uint32_t polls,
                                          void *stream) {
    if (n_flags < 0 || (n_flags > 0 && !flags) || polls < 1) return PKV_ERR_INVALID;
    unsigned int *err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const unsigned long long *>(flags), n_flags, (unsigned long long)tag, arrive, polls, err);
    return launch_status();
}

// ---------------------------------------------------------------------------
// Diagnostics: the balanced split's arithmetic, for host-side tests.
// ---------------------------------------------------------------------------
PKV_API int64_t pkv_balanced_split_parts(int64_t total_tiles, int max_segment_tiles, int max_seq_len,
                                         int64_t warps) {
    if (total_tiles < 0 || max_segment_tiles < 0 || max_seq_len < 0 || warps < 1) return -1;
    if (total_tiles == 0) return 0;
    return balanced_parts(total_tiles, max_segment_tiles, (int)balanced_slots(max_seq_len), warps);
}

PKV_API int64_t pkv_balanced_share_owner(int64_t tile, int64_t total_tiles, int64_t parts) {
    if (total_tiles < 1 || parts < 1 || tile < 0 || tile >= total_tiles) return -1;
    return share_owner(tile, total_tiles, parts);
}

PKV_API int pkv_balanced_segment_tiles(int tiles) { return tiles < 0 ? -1 : laid_out_tiles(tiles); }

PKV_API int pkv_balanced_slots(int max_seq_len) {
    return max_seq_len < 0 ? -1 : (int)balanced_slots(max_seq_len);
}

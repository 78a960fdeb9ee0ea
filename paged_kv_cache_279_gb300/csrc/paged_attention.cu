// Paged decode attention: one new query per sequence attends to every cached
// token of that sequence, whose K/V rows are found through the sequence's
// block table.  Long contexts are split into partitions that are attended
// independently; a reduction kernel merges their partial results.
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

#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

constexpr int kTile = 16;  // tokens per MMA tile and per pipeline stage
constexpr int kGMax = 8;   // max query heads per KV head (the MMA N dimension)
constexpr uint32_t kWaitLimit = 1u << 22;  // bounded mbarrier polling

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
    int num_seqs, num_heads, num_kv_heads, group;
    int block_size, max_blocks, num_blocks, max_seq_len;
    int partition_size, max_parts;
    float scale;       // multiplies q.k
    float scale_log2;  // scale * log2(e), for the exp2 form of the softmax
    unsigned int *err;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Polls a bounded number of times; false means the wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float bf16x2_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

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

template <int D, int NW, int NS>
constexpr int bf16_smem_bytes() {
    return NW * NS * Bf16Layout<D>::kStageBytes + NW * NS * 8 + 1024;
}

template <int D, int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
decode_bf16_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using Lay = Bf16Layout<D>;
    static_assert(NS * Lay::kStageBytes >= Lay::kMergeBytes, "merge area must fit a warp's ring");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    WorkItem w;
    if (!resolve_item(a, w)) return;
    if (w.len == 0) {
        write_zero_rows<__nv_bfloat16, D>(a, w);
        return;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char *ring = smem + warp * NS * Lay::kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * NS * Lay::kStageBytes) + warp * NS;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncwarp();

    const int G = a.group;
    const int Hkv = a.num_kv_heads;
    const int B = a.block_size;
    const int r0 = lane >> 2;  // fragment row group
    const int tq = lane & 3;   // fragment thread-in-group

    // Q^T as the MMA B operand: lane holds query head r0, head_dim pairs.
    uint32_t qb[D / 16][2];
    {
        const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(a.q) +
                                    ((int64_t)w.seq * a.num_heads + w.kvh * G + r0) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            if (r0 < G) {
                qb[ks][0] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * tq);
                qb[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * tq);
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
    }

    const int32_t *bt = a.block_tables + (int64_t)w.seq * a.max_blocks;
    const int ntiles = (w.tok_end - w.tok_begin + kTile - 1) / kTile;
    const int nmine = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
    const int boxh = B < kTile ? B : kTile;

    // Lane 0 only: gather tile `tile` of this item into ring slot `buf`.
    auto issue = [&](int tile, int buf) {
        const int t0 = w.tok_begin + tile * kTile;
        int ys[kTile / 8];
        int nsub = 0;
        for (int sb = 0; sb < kTile / boxh; ++sb) {
            const int tok = t0 + sb * boxh;
            if (tok >= w.tok_end) break;
            const int lb = tok / B;
            int blk = bt[lb];
            if (blk < 0 || blk >= a.num_blocks) {
                // never dereferenced out of range: read block 0 instead and
                // mask these rows out of the softmax (see row_ok below)
                flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                blk = 0;
            }
            ys[nsub++] = (int)(((int64_t)blk * Hkv + w.kvh) * B + (tok - lb * B));
        }
        const uint32_t bytes = (uint32_t)(nsub * Lay::kHalves * boxh * 128 * 2);
        const uint32_t bar = smem_u32(&bars[buf]);
        mbar_arrive_expect_tx(&bars[buf], bytes);
        const uint32_t dk = smem_u32(ring + buf * Lay::kStageBytes);
        const uint32_t dv = dk + Lay::kKVBytes;
        for (int sb = 0; sb < nsub; ++sb) {
#pragma unroll
            for (int h = 0; h < Lay::kHalves; ++h) {
                const uint32_t off = h * Lay::kHalfBytes + sb * boxh * 128;
                tma_load_2d(dk + off, &tm_k, bar, h * 64, ys[sb]);
                tma_load_2d(dv + off, &tm_v, bar, h * 64, ys[sb]);
            }
        }
    };

    if (lane == 0) {
        for (int i = 0; i < NS && i < nmine; ++i) issue(warp + i * NW, i);
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    const float sl2 = a.scale_log2;
    bool dead = false;

    for (int i = 0; i < nmine; ++i) {
        const int buf = i % NS;
        if (!mbar_wait_bounded(&bars[buf], (uint32_t)((i / NS) & 1))) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
            dead = true;
            break;
        }
        const int tile = warp + i * NW;
        const int t0 = w.tok_begin + tile * kTile;
        // rows of this tile that hold a token of the context from a valid block
        uint32_t row_ok = 0;
        for (int sb = 0; sb < kTile / boxh; ++sb) {
            const int tok = t0 + sb * boxh;
            if (tok >= w.tok_end) break;
            const int blk = bt[tok / B];
            if (blk >= 0 && blk < a.num_blocks) row_ok |= ((1u << boxh) - 1u) << (sb * boxh);
        }
        const int valid = min(kTile, w.tok_end - t0);
        row_ok &= (1u << valid) - 1u;
        unsigned char *sk = ring + buf * Lay::kStageBytes;
        unsigned char *sv = sk + Lay::kKVBytes;
        if (row_ok != 0xffffu) {
            // masked rows hold stale, unwritten or substituted slots: zero their
            // V so that a zero weight never meets a NaN
            for (int e = lane; e < Lay::kHalves * kTile * 8; e += 32) {
                const int h = e / (kTile * 8), rr = (e / 8) % kTile, c = e % 8;
                if (!((row_ok >> rr) & 1u))
                    *reinterpret_cast<uint4 *>(sv + h * Lay::kHalfBytes + rr * 128 + c * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        const uint32_t ska = smem_u32(sk), sva = smem_u32(sv);
        const int lj = lane >> 3, lr = lane & 7;

        // S^T (16 tokens x 8 heads) = K_tile . Q^T
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int tok = lr + 8 * (lj & 1);
            const int chunk = 2 * (ks & 3) + (lj >> 1);
            const uint32_t addr = ska + (ks >> 2) * Lay::kHalfBytes + tok * 128 + ((chunk ^ (tok & 7)) << 4);
            uint32_t x0, x1, x2, x3;
            ldmatrix_x4(addr, x0, x1, x2, x3);
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
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // reference points stay finite even if nothing valid has been seen yet
        const float rf0 = mn0 == -INFINITY ? 0.f : mn0, rf1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0 - rf0), al1 = exp2f(m1 - rf1);
        m0 = mn0;
        m1 = mn1;
        const uint32_t p01 = pack_bf16x2(exp2f(s0 - rf0), exp2f(s1 - rf1));
        const uint32_t p23 = pack_bf16x2(exp2f(s2 - rf0), exp2f(s3 - rf1));
        // the sum uses the same rounded weights as the numerator
        l0 = l0 * al0 + (bf16x2_lo(p01) + bf16x2_lo(p23));
        l1 = l1 * al1 + (bf16x2_hi(p01) + bf16x2_hi(p23));
        const uint32_t pb0 = movmatrix_trans(p01);
        const uint32_t pb1 = movmatrix_trans(p23);

        // O^T (head_dim x 8 heads) = O^T * alpha + V_tile^T . P^T
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
            const int tok = lr + 8 * (lj >> 1);
            const int chunk = 2 * (mt & 3) + (lj & 1);
            const uint32_t addr = sva + (mt >> 2) * Lay::kHalfBytes + tok * 128 + ((chunk ^ (tok & 7)) << 4);
            uint32_t x0, x1, x2, x3;
            ldmatrix_x4_trans(addr, x0, x1, x2, x3);
            mma_bf16_16816(o[mt], x0, x1, x2, x3, pb0, pb1);
        }
        __syncwarp();
        if (lane == 0 && i + NS < nmine) {
            fence_proxy_async();
            issue(warp + (i + NS) * NW, buf);
        }
    }

    // column sums over the 16 token rows held across lanes r0 = 0..7
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }
    if (dead || nmine == 0) {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    // Each warp parks its partial in its own (now idle) ring.
    float *mine = reinterpret_cast<float *>(ring);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = 16 * mt + r0 + 8 * (j >> 1);
            const int g = 2 * tq + (j & 1);
            mine[g * D + d] = o[mt][j];
        }
    }
    if (r0 == 0) {
        mine[kGMax * D + 2 * tq] = m0;
        mine[kGMax * D + 2 * tq + 1] = m1;
        mine[kGMax * D + kGMax + 2 * tq] = l0;
        mine[kGMax * D + kGMax + 2 * tq + 1] = l1;
    }
    __syncthreads();
    const float *bufs[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) bufs[k] = reinterpret_cast<const float *>(smem + k * NS * Lay::kStageBytes);
    merge_warps_and_store<__nv_bfloat16, D, NW, true>(a, w, bufs);
}

// ---------------------------------------------------------------------------
// CUDA-core kernel (fp32 I/O; also instantiated for bf16 storage)
// ---------------------------------------------------------------------------
template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32) decode_simt_kernel(const DecodeArgs a) {
    constexpr int E = D / 32;  // head_dim elements per lane: d = lane + 32 j
    __shared__ float merge_buf[NW][kGMax * D + 2 * kGMax];

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
// Partition merge: out = sum_j e^{m_j - M} o_j / sum_j e^{m_j - M} l_j
// ---------------------------------------------------------------------------
template <typename T, int D, bool LOG2>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeArgs a) {
    constexpr int E = D / 32;  // consecutive head_dim elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;  // (sequence, query head)
    if (row >= (int64_t)a.num_seqs * a.num_heads) return;
    const int seq = (int)(row / a.num_heads);
    const int cap = min(a.max_seq_len, a.max_blocks * a.block_size);
    int len = a.seq_lens[seq];
    len = len < 0 ? 0 : (len > cap ? cap : len);
    const int nparts = (len + a.partition_size - 1) / a.partition_size;
    if (nparts <= 1) return;

    const float *pm = a.part_m + row * a.max_parts;
    const float *pl = a.part_l + row * a.max_parts;
    const float *po = a.part_o + row * a.max_parts * D;
    float M = -INFINITY;
    for (int j = lane; j < nparts; j += 32) M = fmaxf(M, pm[j]);
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
    if (M == -INFINITY) M = 0.f;  // only if every block was invalid (flagged)
    float lsum = 0.f;
    for (int j = lane; j < nparts; j += 32) lsum += (LOG2 ? exp2f(pm[j] - M) : expf(pm[j] - M)) * pl[j];
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, sh);

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int j = 0; j < nparts; ++j) {
        const float c = LOG2 ? exp2f(pm[j] - M) : expf(pm[j] - M);
        const float *src = po + (int64_t)j * D + lane * E;
        if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            acc[0] += c * v.x;
            acc[1] += c * v.y;
            acc[2] += c * v.z;
            acc[3] += c * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2 *>(src);
            acc[0] += c * v.x;
            acc[1] += c * v.y;
        }
    }
    T *dst = static_cast<T *>(a.out) + row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) store_out(dst + e, lsum > 0.f ? acc[e] / lsum : 0.f);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int auto_partition_size(int num_seqs, int max_seq_len) {
    (void)num_seqs;
    (void)max_seq_len;
    return 512;
}

static size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WorkspaceLayout {
    size_t o_off, m_off, l_off, total;
};

static WorkspaceLayout workspace_layout(int64_t S, int64_t Hq, int64_t D, int64_t parts) {
    WorkspaceLayout w;
    w.o_off = 0;
    w.m_off = round256((size_t)(S * Hq * parts * D * 4));
    w.l_off = w.m_off + round256((size_t)(S * Hq * parts * 4));
    w.total = w.l_off + round256((size_t)(S * Hq * parts * 4));
    return w;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of a bf16 cache: rows = num_blocks * Hkv * B, columns = head_dim.
// Box = 64 columns (128 bytes, 128-byte swizzle) x min(B, 16) rows.
static bool make_cache_map(CUtensorMap *map, const void *base, int64_t rows, int D, int boxh) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)boxh};
    cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt a kernel in to the dynamic shared memory it needs (once per device).
template <typename K>
static bool ensure_smem(K kernel, int bytes, bool (&done)[128]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return false;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

// Launch shapes of the bf16 kernel: warps per CTA x ring stages per warp.
// PKV_DECODE_VARIANT selects one for tuning sweeps; the default is the one
// measured fastest on GB300.
static int decode_variant() {
    static int v = [] {
        const char *s = std::getenv("PKV_DECODE_VARIANT");
        return s ? std::atoi(s) : 0;
    }();
    return v;
}

template <int D, int NW, int NS>
static pkv_status launch_bf16(const DecodeArgs &a, dim3 grid, cudaStream_t st) {
    static bool done[128] = {};
    constexpr int smem = bf16_smem_bytes<D, NW, NS>();
    auto kern = decode_bf16_mma_kernel<D, NW, NS>;
    if (!ensure_smem(kern, smem, done)) return PKV_ERR_CUDA;
    const int boxh = a.block_size < kTile ? a.block_size : kTile;
    const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * a.block_size;
    CUtensorMap mk, mv;
    if (!make_cache_map(&mk, a.k_cache, rows, D, boxh) || !make_cache_map(&mv, a.v_cache, rows, D, boxh))
        return PKV_ERR_CUDA;
    kern<<<grid, NW * 32, smem, st>>>(mk, mv, a);
    return launch_status();
}

template <int D>
static pkv_status dispatch_bf16(const DecodeArgs &a, dim3 grid, cudaStream_t st) {
    switch (decode_variant()) {
        case 1: return launch_bf16<D, 4, 2>(a, grid, st);
        case 2: return launch_bf16<D, 4, 4>(a, grid, st);
        case 3: return launch_bf16<D, 8, 2>(a, grid, st);
        default: return launch_bf16<D, 4, 3>(a, grid, st);
    }
}

template <typename T, int D>
static pkv_status dispatch_simt(const DecodeArgs &a, dim3 grid, cudaStream_t st) {
    decode_simt_kernel<T, D, 4><<<grid, 128, 0, st>>>(a);
    return launch_status();
}

template <typename T, int D, bool LOG2>
static pkv_status launch_reduce(const DecodeArgs &a, cudaStream_t st) {
    const int64_t rows = (int64_t)a.num_seqs * a.num_heads;
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    decode_reduce_kernel<T, D, LOG2><<<blocks, 128, 0, st>>>(a);
    return launch_status();
}

}  // namespace pkv

using namespace pkv;

PKV_API size_t paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim,
                                              int max_seq_len, int partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
    const int P = partition_size > 0 ? partition_size : auto_partition_size(num_seqs, max_seq_len);
    if (P <= 0 || P % kTile != 0) return 0;
    const int64_t parts = ((int64_t)max_seq_len + P - 1) / P;
    if (parts <= 1) return 0;
    return workspace_layout(num_seqs, num_heads, head_dim, parts).total;
}

PKV_API pkv_status paged_attention_decode(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *seq_lens, int num_seqs, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                          float scale, int partition_size, void *workspace,
                                          size_t workspace_bytes, int dtype, void *stream) {
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
    // TMA row coordinates are 32-bit: every (block, kv head, row) must be addressable,
    // plus one out-of-range block used to neutralise bad block ids.
    const int64_t rows = ((int64_t)num_blocks + 1) * num_kv_heads * block_size;
    if (rows > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PKV_ERR_INVALID;

    const int P = partition_size > 0 ? partition_size : auto_partition_size(num_seqs, max_seq_len);
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

    if (parts > 1) {
        const WorkspaceLayout lay = workspace_layout(num_seqs, num_heads, head_dim, parts);
        if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return PKV_ERR_INVALID;
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        a.part_o = reinterpret_cast<float *>(ws + lay.o_off);
        a.part_m = reinterpret_cast<float *>(ws + lay.m_off);
        a.part_l = reinterpret_cast<float *>(ws + lay.l_off);
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid((unsigned)num_seqs, (unsigned)num_kv_heads, (unsigned)parts);
    pkv_status rc;
    if (dtype == PKV_BF16) {
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

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace (paged_attention_decode_noalloc).
// For callers that cannot allocate device memory, the split-K partials live
// in this array, compiled into the library and resident on every device that
// loads it until the process exits.  Host code must not use the symbol's
// name as a device address (on the host it is only a stand-in); the device
// address is looked up once per device below.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call for that device (with the device current).  nullptr on failure.
static void *noalloc_scratch_address() {
    static std::mutex mu;
    static void *ptrs[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress((void **)&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = p;
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

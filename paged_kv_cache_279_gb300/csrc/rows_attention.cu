// Attention of many query rows against the same paged K/V tiles on the
// 5th-generation tensor cores (tcgen05): the kernel behind
//   * paged_attention_decode_grouped -- beams (or parallel samples) that share
//     the blocks of a prompt prefix ("PagedAttention (vLLM) -- Virtual memory
//     cho AI", section "Copy-on-Write cho Beam Search": branches share the
//     physical blocks of their prefix);
//   * paged_attention_multi_token -- several new tokens of one sequence
//     attending causally over its paged context: chunked prefill and the
//     verification of drafted tokens ("vLLM PagedAttention: Buoc dot pha ...",
//     list of advanced features: "Chunked Prefill", "speculative decoding").
//
// Per KV head the work is a dense contraction: up to 128 query rows (the
// query heads of that KV head for every member of a group, or for every query
// token of a block of queries) against the same 64-token K and V tiles:
//     S = Q K^T (M = 128 rows, N = 64 keys, K = head_dim),
//     O += P V   (M = 128 rows, N = head_dim, K = 64 keys),
// with an online softmax per row in between.  A "context" is one such set of
// rows for one KV head and the tiles it attends:
//   * grouped: the group's prefix tiles (seen by every row), then each
//     member's own tiles (seen only by that member's rows; the others get
//     zero weight) -- so one context yields every member's final result, with
//     no separate merge of prefix and own parts;
//   * multi-token: the tiles up to the block's last query position; row r
//     sees the keys at or before its own position.  When queries span more
//     than one 128-row block (prefill chunks), a context is a pair of
//     consecutive blocks (paired mode): both read every tile once.
// All contexts' tiles are laid end to end, each context behind a few virtual
// tiles that nothing loads (a scheduling charge for its fixed costs), and
// every CTA (one per SM, persistent) takes an equal contiguous share.  A
// context cut by share boundaries is merged inside the kernel: every later
// piece is the first piece of its CTA's share, whose CTA stores a partial
// (o, m, l) per row in its own slot and raises its flag; the CTA holding the
// context's first real tile (its share's last piece) waits for those flags
// and merges.  Every CTA is
// resident at once (cooperative launch), and a CTA never waits for a piece
// later in its own share, so no chain of waits can close.
//
// Warp roles (384 threads):
//   warps 0-3, 4-7  two softmax groups; group g takes the tiles j with
//              j % 2 == g of every piece (two independent chains per SM);
//              in paired mode group g owns block g's rows and takes every
//              tile.  Thread r of a group owns query row r = TMEM lane r.  Reads S
//              from TMEM, keeps the row's running max and sum, writes P (bf16)
//              back into the S columns (P is the A operand of P V, taken from
//              tensor memory), zeroes the V rows of keys past a context's end
//              and, on a piece's last tile, loads the next piece's queries.
//              Each group accumulates its own O; at a piece's end the groups
//              exchange their rows' (max, sum) and each combines the two
//              partial states for half of the columns and writes them
//              (paired: each group writes its own rows).
//   warp 8     paired contexts: issues softmax group 1's Q K^T and P V (one
//              thread); idle otherwise.
//   warp 9     grouped: checks that every member's block table holds the
//              leader's blocks over the prefix.
//   warp 10    producer: walks the share, publishes one descriptor per piece,
//              stages block ids in shared memory (many loads in flight) and
//              issues the K/V TMA boxes (one block per box) into an NS-stage
//              ring, with each tile's key range in a per-stage record.
//   warp 11    MMA: allocates tensor memory; one thread issues Q K^T and P V,
//              each as soon as its inputs are ready (a late tile does not hold
//              up the P V of the one before); paired contexts: group 0's only.
// Every wait is bounded; on a timeout the kernel flags PKV_DEVERR_TIMEOUT,
// waits (bounded) for its own copies in flight, frees its tensor memory and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "pkv_internal.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace rows {

constexpr int kTok = 64;          // keys per tile
constexpr int kRows = tc::kRows;  // query rows per context (the MMA's M)
constexpr int kSG = 2;           // softmax groups (warps 0-3 and 4-7), one chain of tiles each
constexpr int kThreads = 384;
// Warp roles.  Warp 8 issues group 1's MMAs in paired mode.  The producer and MMA warps share the
// schedulers of softmax warps 2, 6 and 3, 7, which have no rows when a context
// has at most 64 (resp. 96) rows.
constexpr int kAuxWarp = 9, kProducerWarp = 10, kMmaWarp = 11;
constexpr int kMma1Warp = 8;  // paired contexts: issues softmax group 1's MMAs
constexpr int kMaxUnits = 1024;   // groups / sequences scanned per launch
constexpr int kMinTiles = 6;      // shares hold >= 6 tiles unless the total is small
// Scheduling charge of a context, in tiles: a context with n tiles is laid out
// as kPieceTiles virtual tiles (never loaded) and then its n real ones, so that
// equal shares of the layout also balance the fixed cost of each piece (its
// queries' load, the wait for its last P V, the combine and the write of its
// rows; about five tiles' streaming time) and not only its tiles.  Below
// kMinTiles, so every share holds a real tile.
constexpr int kPieceTiles = 5;
static_assert(kPieceTiles < kMinTiles, "a share of kMinTiles laid-out tiles holds a real tile");
constexpr int kIdCache = 512;     // block ids staged by the producer
constexpr int kChunkTiles = 128;  // tiles whose keys the producer stages at once
constexpr int kDescs = 8;         // piece descriptors in flight
constexpr int kMergeHeld = 1;     // partials a merger keeps in registers (the rest are re-read)
constexpr float kRescale = 8.f;   // headroom (log2 units) before a row's running max moves
constexpr int kSB = 4;            // S / P buffers in tensor memory: two per softmax group
constexpr uint32_t kOBase = kSB * kTok;  // O of softmax group g at kOBase + g * D
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxCtas = 256;     // partial slots in the workspace: one per CTA

enum { kGrouped = 0, kMulti = 1 };
enum { kWhole = 1, kContinue = 2, kMerger = 4 };

struct Args {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int num_heads, num_kv_heads, group, block_size, max_blocks, num_blocks, max_seq_len;
    float scale_log2;
    unsigned int *err;
    float *part_o;                // [kMaxCtas][kRows][D]
    float *part_ml;               // [kMaxCtas][kRows][2]
    unsigned long long *flags;    // [kMaxCtas]
    unsigned long long tag;
    int mode;
    int unit0, num_units;         // this launch: groups / sequences unit0 .. unit0 + num_units - 1
    int per_ctx;                  // members (grouped) or queries (multi-token) per context: kRows / group
    // grouped
    const int32_t *group_offsets;
    const int32_t *prefix_lens;
    int num_seqs, num_groups, appended;
    // multi-token
    const int32_t *q_starts;
    int num_q_tokens, max_q_len;
};

// One piece of a context: what the MMA and softmax warps need.
struct Piece {
    int ntiles;    // 0: no more pieces
    int row_base;  // first member (grouped) / first query row of q and out (multi-token)
    int rows;      // live rows
    int kvh;
    int pos0;      // multi-token: position of the first query of the block
    int kind;      // kWhole, kContinue or kMerger
    int w0, w1;    // CTAs holding the context's first and last tiles
};

// Per ring stage: the keys of the tile in it.
struct TileInfo {
    int member;    // grouped own tile: member index within the context (rows member*G ..); -1 = every row
    int nvalid;    // keys 0 .. nvalid-1 of the tile exist
    uint32_t bad;  // bit j: block j of the tile had an invalid id (its keys are masked)
    int key0;      // position of the tile's first key
};

// Byte offset rounded up to a multiple of 16 (every region below is accessed
// with up to 16-byte vectors).
constexpr int align16(int x) { return (x + 15) & ~15; }

// Alternating mode: tile j (counted per CTA) belongs to softmax group j % 2;
// each group has two S / P buffers, used by its tiles in turn: buffer
// 2 g + (j / 2) % 2, which completes one phase per use (every fourth tile).
// Paired mode (a context of two query blocks, one per group): both groups
// take every tile; group g's buffer for tile j is 2 g + j % 2, one phase per
// use (every second tile).
template <bool PAIRED>
__device__ __forceinline__ int sbuf(int j, int g) { return PAIRED ? 2 * g + (j & 1) : 2 * (j & 1) + ((j >> 1) & 1); }
template <bool PAIRED>
__device__ __forceinline__ uint32_t sphase(int j) { return (uint32_t)((PAIRED ? j >> 1 : j >> 2) & 1); }
static_assert(kSB == 2 * kSG, "two S / P buffers per softmax group");

template <int D, bool PAIRED>
struct Layout {
    static constexpr int H = D / 64;                      // 128-byte column halves
    static constexpr int kQTile = H * kRows * 128;        // one group's Q: [half][row][128 B]
    static constexpr int kQBytes = (PAIRED ? 2 : 1) * kQTile;
    // K of a tile: [half][token][128 B] (one 2-D box per block and half);
    // V of a tile: [block][half][block row][128 B] (one box per block)
    static constexpr int kKVBytes = H * kTok * 128;
    static constexpr int kStageBytes = 2 * kKVBytes;
    // 160 KB of Q and tiles in flight (paired: the second Q tile takes a stage)
    static constexpr int NS = D == 128 ? (PAIRED ? 4 : 5) : (PAIRED ? 9 : 10);
    static constexpr int q = 0;
    static constexpr int ring = q + kQBytes;
    static constexpr int cum = ring + NS * kStageBytes;               // int [kMaxUnits + 4]
    static constexpr int uval = align16(cum + (kMaxUnits + 4) * 4);   // int [kMaxUnits]: prefix tokens / query count
    static constexpr int ids = align16(uval + kMaxUnits * 4);         // int [kIdCache]
    static constexpr int tkc = align16(ids + kIdCache * 4);           // int4 [kChunkTiles]: keys of the staged tiles
    static constexpr int mo = align16(tkc + kChunkTiles * 16);        // int [kRows + 4]: members' first own tile
    static constexpr int tinfo = align16(mo + (kRows + 4) * 4);       // TileInfo [NS]
    static constexpr int desc = align16(tinfo + NS * 16);             // Piece [kDescs]
    static constexpr int xch = align16(desc + kDescs * 32);           // float2 [2][kRows]: each group's (max, sum) per row
    static constexpr int bars = align16(xch + 2 * kRows * 8);
    // k/v full, kv empty, s/p full, o_done[4], ready, fin, o_free[2], xch full[2]/empty[2], o_last[2], descs
    static constexpr int kBars = 3 * NS + 2 * kSB + 14 + 2 * kDescs;
    static constexpr int misc = align16(bars + kBars * 8);            // TMEM address, scan scratch, counters
    static constexpr int total = misc + 128 + 1024;                   // + alignment slack
    static_assert(sizeof(Piece) == 32 && sizeof(TileInfo) == 16, "descriptor sizes");
    static_assert(ring % 1024 == 0 && kStageBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(tkc % 16 == 0 && tinfo % 16 == 0 && bars % 8 == 0, "vector accesses need aligned regions");
    static_assert(total <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ int clamp_len(int len, int cap) { return len < 0 ? 0 : (len > cap ? cap : len); }

__device__ __forceinline__ void st32u(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// ---------------------------------------------------------------------------
// Units and contexts.  A unit is a group (grouped) or a sequence (multi-
// token).  Its contexts are ordered KV head first, then sub-context: the
// group's member chunks (per_ctx members each) or the sequence's query blocks
// (per_ctx queries each), so that contexts reading the same K/V are adjacent.
// ---------------------------------------------------------------------------
struct Unit {
    int m0, m1;  // grouped: members; multi-token: query rows q0 .. q0 + Q
    int pre;     // grouped: prefix tokens attended by every member (a multiple of 64)
    int Q, L;    // multi-token: queries and context length
    int nsub;    // member chunks / query blocks
};

__device__ __forceinline__ Unit load_unit(const Args &a, const int *uval, int u) {
    Unit x{};
    const int cap = min(a.max_seq_len, a.max_blocks * a.block_size);
    const int gu = a.unit0 + u;
    if (a.mode == kGrouped) {
        int m0 = a.group_offsets[gu], m1 = a.group_offsets[gu + 1];
        if (m0 < 0 || m1 > a.num_seqs || m1 < m0) m0 = m1 = 0;  // flagged by the scan
        x.m0 = m0;
        x.m1 = m1;
        x.pre = uval[u];
        x.nsub = (m1 - m0 + a.per_ctx - 1) / a.per_ctx;
    } else {
        int q0 = a.q_starts[gu], q1 = a.q_starts[gu + 1];
        if (q0 < 0 || q1 < q0 || q1 > a.num_q_tokens) q0 = q1 = 0;  // flagged by the scan
        x.m0 = q0;
        x.Q = uval[u];
        x.m1 = q0 + x.Q;
        x.L = clamp_len(a.seq_lens[gu], cap);
        x.nsub = (x.Q + a.per_ctx - 1) / a.per_ctx;
    }
    return x;
}

__device__ __forceinline__ int own_tiles(const Args &a, int seq, int pre, int cap) {
    const int len = clamp_len(a.seq_lens[seq], cap);
    return len > pre ? (len - pre + kTok - 1) / kTok : 0;
}

// Last query position of query block b (-1 if it sees no key).
__device__ __forceinline__ int block_last_pos(const Unit &x, int b, int per_ctx) {
    return x.L - x.Q + min(x.Q, (b + 1) * per_ctx) - 1;
}

// Real tiles of sub-context `sub` of a unit (for any one KV head).  per_kvh =
// the unit's laid-out tiles per KV head (real and virtual), which gives the
// answer when there is one sub-context.
__device__ __forceinline__ int sub_tiles(const Args &a, const Unit &x, int sub, int per_kvh, int cap) {
    if (x.nsub == 1) return per_kvh > 0 ? per_kvh - kPieceTiles : 0;
    if (a.mode == kGrouped) {
        int n = x.pre / kTok;
        const int c0 = x.m0 + sub * a.per_ctx, c1 = min(x.m1, c0 + a.per_ctx);
        for (int m = c0; m < c1; ++m) n += own_tiles(a, m, x.pre, cap);
        return n;
    }
    const int p = block_last_pos(x, sub, a.per_ctx);
    return p < 0 ? 0 : (p + kTok) / kTok;
}

// Laid-out tiles of a context with n real ones (none when it has none).
__host__ __device__ __forceinline__ int laid_out(int n) { return n > 0 ? n + kPieceTiles : 0; }

// Shares the T laid-out tiles of a launch are cut into: one per CTA, each of
// at least kMinTiles tiles unless the total is small.
__host__ __device__ __forceinline__ int64_t split_parts(int64_t T, int64_t ctas) {
    const int64_t by_size = T / kMinTiles > 1 ? T / kMinTiles : 1;
    return ctas < by_size ? ctas : by_size;
}

// Position in the tile list: context (unit u, kv head, sub-context) with n
// laid-out tiles starting at global tile `start` (its first kPieceTiles are
// virtual).
struct Ctx {
    int u, kvh, sub, n;
    int64_t start;
    int per_kvh;
    Unit x;

    __device__ __forceinline__ bool seek(const Args &a, const int *cum, const int *uval, int64_t t, int cap) {
        int lo = 0, hi = a.num_units;  // largest u with cum[u] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= t) lo = mid; else hi = mid;
        }
        u = lo;
        x = load_unit(a, uval, u);
        per_kvh = (cum[u + 1] - cum[u]) / a.num_kv_heads;
        const int64_t local = t - cum[u];
        kvh = (int)(local / per_kvh);
        int64_t rem = local - (int64_t)kvh * per_kvh;
        start = cum[u] + (int64_t)kvh * per_kvh;
        for (sub = 0; sub < x.nsub; ++sub) {
            n = laid_out(sub_tiles(a, x, sub, per_kvh, cap));
            if (rem < n) return true;
            rem -= n;
            start += n;
        }
        return false;  // the scan and the walk disagree: never expected
    }

    // Next context with at least one tile; false past the launch's last unit.
    __device__ __forceinline__ bool next(const Args &a, const int *cum, const int *uval, int cap) {
        start += n;
        for (;;) {
            if (++sub >= x.nsub) {
                sub = 0;
                if (++kvh == a.num_kv_heads) {
                    kvh = 0;
                    do { ++u; } while (u < a.num_units && cum[u + 1] == cum[u]);
                    if (u >= a.num_units) return false;
                    x = load_unit(a, uval, u);
                    per_kvh = (cum[u + 1] - cum[u]) / a.num_kv_heads;
                }
            }
            n = laid_out(sub_tiles(a, x, sub, per_kvh, cap));
            if (n > 0) return true;
        }
    }

    // Rows of the context: first row of q / out and live rows.
    __device__ __forceinline__ void rows(const Args &a, int &row_base, int &nrows, int &pos0) const {
        if (a.mode == kGrouped) {
            row_base = x.m0 + sub * a.per_ctx;
            nrows = (min(x.m1, row_base + a.per_ctx) - row_base) * a.group;
            pos0 = 0;
        } else {
            row_base = x.m0 + sub * a.per_ctx;
            nrows = (min(x.Q, (sub + 1) * a.per_ctx) - sub * a.per_ctx) * a.group;
            pos0 = x.L - x.Q + sub * a.per_ctx;
        }
    }
};

// Keys of tile i of a context: table row (sequence), first key, valid keys,
// member.  mo[k] = first own tile (relative to the context) of chunk member
// k, k = 0 .. members (grouped contexts only).
struct TileKeys {
    int seq, key0, nvalid, member;
};

__device__ __forceinline__ TileKeys tile_keys(const Args &a, const Ctx &c, const int *mo, int members, int i,
                                              int cap) {
    TileKeys k;
    if (a.mode == kGrouped) {
        const int npt = c.x.pre / kTok;
        const int c0 = c.x.m0 + c.sub * a.per_ctx;
        if (i < npt) {
            k.seq = c.x.m0;  // the leader's blocks
            k.key0 = i * kTok;
            k.nvalid = kTok;
            k.member = -1;
        } else {
            int lo = 0, hi = members;  // largest member with mo[m] <= i - npt
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (mo[mid] <= i - npt) lo = mid; else hi = mid;
            }
            k.member = lo;
            k.seq = c0 + lo;
            k.key0 = c.x.pre + (i - npt - mo[lo]) * kTok;
            k.nvalid = min(kTok, clamp_len(a.seq_lens[k.seq], cap) - k.key0);
        }
    } else {
        k.seq = a.unit0 + c.u;
        k.key0 = i * kTok;
        k.nvalid = min(kTok, block_last_pos(c.x, c.sub, a.per_ctx) + 1 - k.key0);
        k.member = -1;
    }
    return k;
}

__device__ __forceinline__ void ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st8u(uint32_t taddr, const uint32_t *v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// One tile of one row's online softmax over its NC x 16 keys [c0, c0 + 16 NC)
// of the tile: S from tensor memory at sp (scores, 1 column per key), P (bf16
// pairs) back over the first 32 columns at sp -- this row's keys, zero for the
// others.  Keys at or past lim, or in a block whose bit is set in `bad`, get
// zero weight.  The running max moves only when the tile's exceeds it by more
// than 2^kRescale (then `move`, and O is to be scaled by `alpha`).
template <int NC>
__device__ __forceinline__ void softmax_tile(uint32_t sp, int c0, int lim, uint32_t bad, int bshift, float sl2,
                                             float &m_run, float &l, bool &move, float &alpha) {
    constexpr int N = NC * 16;
    float s[N];
    if constexpr (NC == 4) {
        tc::ld32(sp, s);
        tc::ld32(sp + 32, s + 32);
    } else if constexpr (NC == 2) {
        tc::ld32(sp + c0, s);
    } else {
        ld16(sp + c0, s);
    }
    tc::wait_ld();
    // keys of this row: bit k of (lo, hi) = key c0 + k is seen (below lim, in a valid block)
    uint32_t lo = 0u, hi = 0u;
    {
        const int n = lim - c0;
        if (n >= 64) {
            lo = hi = 0xffffffffu;
        } else if (n > 0) {
            lo = n >= 32 ? 0xffffffffu : (1u << n) - 1u;
            hi = n > 32 ? (1u << (n - 32)) - 1u : 0u;
        }
        if (bad) {  // invalid blocks: clear their keys (rare)
            for (int k = 0; k < N; ++k)
                if ((bad >> ((c0 + k) >> bshift)) & 1u) {
                    if (k < 32) lo &= ~(1u << k);
                    else hi &= ~(1u << (k - 32));
                }
        }
    }
    const bool full = (N == 64 ? (lo & hi) : (N == 32 ? lo : (lo & 0xffffu) | ~0xffffu)) == 0xffffffffu;
    if (!full) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const uint32_t w = k < 32 ? lo : hi;
            s[k] = (w >> (k & 31)) & 1u ? s[k] : -INFINITY;
        }
    }
    // Row max of the raw scores, then the log2 scale: sl2 > 0, so the max
    // commutes with the scaling and its rounding.
    float mx[8];  // eight independent chains of three-input maxima over keys q, q + 8, ...
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        mx[q] = s[q];
#pragma unroll
        for (int k = q + 8; k < N; k += 16) mx[q] = k + 8 < N ? fmax3(mx[q], s[k], s[k + 8]) : fmaxf(mx[q], s[k]);
    }
    const float mt = sl2 * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
    float m_new = m_run;
    move = false;
    if (mt != -INFINITY) {
        if (m_run == -INFINITY) {
            m_new = mt;  // nothing accumulated yet: O is zero, nothing to rescale
        } else if (mt > m_run + kRescale) {
            m_new = mt;
            move = true;
        }
    }
    alpha = move ? ex2_approx(m_run - m_new) : 1.f;
    m_run = m_new;
    const float nm = m_run == -INFINITY ? 0.f : -m_run;
    // weights 2^(s sl2 - m): the arguments of two keys from one packed FMA; the
    // denominator sums the fp32 weights (packed adds), P holds them rounded to bf16
    const uint64_t sl2x2 = f32x2(sl2, sl2), nmx2 = f32x2(nm, nm);
    uint32_t pk[N / 2];
    uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
        float a0, a1;
        f32x2_split(fma_f32x2(f32x2(s[2 * k], s[2 * k + 1]), sl2x2, nmx2), a0, a1);
        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
        pk[k] = pack_bf16x2(e0, e1);
        ls[k & 3] = add_f32x2(ls[k & 3], f32x2(e0, e1));
    }
    float sum[2];
    f32x2_split(add_f32x2(add_f32x2(ls[0], ls[1]), add_f32x2(ls[2], ls[3])), sum[0], sum[1]);
    l = l * alpha + (sum[0] + sum[1]);
    // P: 8 columns per 16 keys; this row's groups, then zeros for the others
    const int g0 = c0 >> 4;
    if constexpr (NC == 4) {
        st32u(sp, pk);
    } else {
#pragma unroll
        for (int gg = 0; gg < NC; ++gg) st8u(sp + 8 * (g0 + gg), pk + 8 * gg);
    }
    if (NC < 4) {
        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int g = 0; g < 4; ++g)
            if (g < g0 || g >= g0 + NC) st8u(sp + 8 * g, z);
    }
    tc::wait_st();
}

// A row's 16 output columns (bf16, scaled by f) and 16 partial columns (f32):
// whole 32-byte sectors per store where the address allows (the partial slots
// always do; the caller's output is only promised 16-byte alignment).
__device__ __forceinline__ void store_out16(__nv_bfloat16 *p, const float (&o)[16], float f, bool wide) {
    const uint32_t w0 = pack_bf16x2(o[0] * f, o[1] * f), w1 = pack_bf16x2(o[2] * f, o[3] * f);
    const uint32_t w2 = pack_bf16x2(o[4] * f, o[5] * f), w3 = pack_bf16x2(o[6] * f, o[7] * f);
    const uint32_t w4 = pack_bf16x2(o[8] * f, o[9] * f), w5 = pack_bf16x2(o[10] * f, o[11] * f);
    const uint32_t w6 = pack_bf16x2(o[12] * f, o[13] * f), w7 = pack_bf16x2(o[14] * f, o[15] * f);
    if (wide) {
        st_global_32B(p, w0, w1, w2, w3, w4, w5, w6, w7);
    } else {
        uint4 *d = reinterpret_cast<uint4 *>(p);
        d[0] = make_uint4(w0, w1, w2, w3);
        d[1] = make_uint4(w4, w5, w6, w7);
    }
}
__device__ __forceinline__ void store_part16(float *p, const float (&o)[16]) {
    st_global_32B(p, __float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]),
                  __float_as_uint(o[4]), __float_as_uint(o[5]), __float_as_uint(o[6]), __float_as_uint(o[7]));
    st_global_32B(p + 8, __float_as_uint(o[8]), __float_as_uint(o[9]), __float_as_uint(o[10]), __float_as_uint(o[11]),
                  __float_as_uint(o[12]), __float_as_uint(o[13]), __float_as_uint(o[14]), __float_as_uint(o[15]));
}

// Bounded wait helper: returns false (and flags) once the wait gives up.
__device__ __forceinline__ bool wait_or_flag(uint64_t *bar, uint32_t parity, bool &dead, unsigned int *err) {
    if (dead) return false;
    if (!mbar_wait_bounded(bar, parity)) {
        flag_error(err, PKV_DEVERR_TIMEOUT);
        dead = true;
        return false;
    }
    return true;
}

// Paired contexts: the result of one piece for this thread's row: final rows (whole context), a
// partial in this CTA's slot with its ready flag (a later piece of a context
// begun in an earlier share), or the merge of the other CTAs' partials (the
// context's first piece).  M, Lc: the row's max and sum; load_o(cc, o) gives 16
// unnormalised O columns on the scale of M.  cr: the row within the context
// (and the slot); `last` + 1 warps finish each piece; o_free_bar is arrived
// once O has been read.
template <int D, typename LoadO>
__device__ __forceinline__ void finish_piece(const Args &a, const Piece &pc, float M, float Lc, LoadO &load_o, int cr,
                                             int slot_rows, bool live, bool live_warp, int lane, int w_me, int G,
                                             int last, int *counters, uint64_t *o_free_bar) {
    const int64_t orow = (int64_t)(pc.row_base + (live ? cr / G : 0)) * a.num_heads + pc.kvh * G + cr % G;
    constexpr int kNc = D / 16;  // 16-column chunks of an O row
    // the piece's result: final rows, a partial for the merger, or the merge
    float f = 1.f, e_own = 1.f, Mtr = 0.f;
    bool got = true;
    for (int cc = 0; cc < kNc; ++cc) {
        if (cc == 0) {
            if (pc.kind == kWhole) {
                f = Lc > 0.f ? 1.f / Lc : 0.f;
            } else if (pc.kind == kContinue) {
                if (live)
                    *reinterpret_cast<float2 *>(a.part_ml + ((int64_t)w_me * slot_rows + cr) * 2) = make_float2(M, Lc);
            } else if (live_warp) {
                // merger: this piece holds the context's first tile and is the
                // last piece of this share; CTAs w0 + 1 .. w1 stored the rest
                const int n = pc.w1 - pc.w0;
                got = wait_flags_bounded(a.flags + pc.w0 + 1, n, a.tag, lane);
                if (!got && lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
                float Mt = M;
                if (live)
                    for (int w = pc.w0 + 1; w <= pc.w1; ++w)
                        Mt = fmaxf(Mt, __ldcg(a.part_ml + ((int64_t)w * slot_rows + cr) * 2));
                Mtr = Mt == -INFINITY ? 0.f : Mt;
                e_own = M == -INFINITY ? 0.f : ex2_approx(M - Mtr);
                float Ls = Lc * e_own;
                if (live)
                    for (int w = pc.w0 + 1; w <= pc.w1; ++w) {
                        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + (int64_t)w * slot_rows + cr);
                        if (ml.x != -INFINITY) Ls += ml.y * ex2_approx(ml.x - Mtr);
                    }
                // NaN rows when a piece never came (flagged above)
                f = got ? (Ls > 0.f ? 1.f / Ls : 0.f) : __int_as_float(0x7fc00000);
            }
        }
        if (live_warp) {
            float o[16];
            load_o(cc, o);
            if (live) {
                if (pc.kind == kContinue) {
                    store_part16(a.part_o + ((int64_t)w_me * slot_rows + cr) * D + cc * 16, o);
                } else {
                    if (pc.kind == kMerger) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] *= e_own;
                        for (int w = pc.w0 + 1; w <= pc.w1; ++w) {
                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + (int64_t)w * slot_rows + cr);
                            if (ml.x == -INFINITY) continue;
                            const float e = ex2_approx(ml.x - Mtr);
                            const float4 *src =
                                reinterpret_cast<const float4 *>(a.part_o + ((int64_t)w * slot_rows + cr) * D + cc * 16);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float4 v = __ldcg(src + k);
                                o[4 * k] += e * v.x;
                                o[4 * k + 1] += e * v.y;
                                o[4 * k + 2] += e * v.z;
                                o[4 * k + 3] += e * v.w;
                            }
                        }
                    }
                    store_out16(static_cast<__nv_bfloat16 *>(a.out) + orow * D + cc * 16, o, f,
                                (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0u);
                }
            }
        }
    }
    // O has been read: the next piece's P V may start
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(o_free_bar);
    if (pc.kind == kContinue) {
        // a later piece of a context begun in an earlier share: the partial
        // is stored; the last warp to finish raises the flag
        fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0) {
            fence_acq_rel_gpu();
            if (atomicAdd(&counters[0], 1) == last) {
                counters[0] = 0;
                fence_acq_rel_gpu();
                *reinterpret_cast<volatile unsigned long long *>(a.flags + w_me) = a.tag;
            }
        }
    } else if (pc.kind == kMerger) {
        // the last warp done reading clears the flags (a graph replay reuses the tag)
        __syncwarp();
        if (lane == 0 && atomicAdd(&counters[1], 1) == last) {
            counters[1] = 0;
            for (int k = 0; k < pc.w1 - pc.w0; ++k) a.flags[pc.w0 + 1 + k] = 0ull;
        }
    }
}

template <int D, bool PAIRED>
__global__ void __launch_bounds__(kThreads, 1)
rows_attention_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const Args a) {
    using L = Layout<D, PAIRED>;
    constexpr int H = L::H;
    constexpr int NS = L::NS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int *cum = reinterpret_cast<int *>(smem + L::cum);
    int *uval = reinterpret_cast<int *>(smem + L::uval);
    int *ids = reinterpret_cast<int *>(smem + L::ids);
    int *mo = reinterpret_cast<int *>(smem + L::mo);
    int4 *tkc = reinterpret_cast<int4 *>(smem + L::tkc);
    TileInfo *tinfo = reinterpret_cast<TileInfo *>(smem + L::tinfo);
    Piece *descs = reinterpret_cast<Piece *>(smem + L::desc);
    uint64_t *k_full = reinterpret_cast<uint64_t *>(smem + L::bars);  // a stage's K (and its record) landed
    uint64_t *v_full = k_full + NS;                                    // a stage's V landed
    uint64_t *kv_empty = v_full + NS;
    uint64_t *s_full = kv_empty + NS;
    uint64_t *p_full = s_full + kSB;
    // [4] one phase per completed P V: alternating mode o_done[j % 2] (the tile's
    // group), paired mode o_done[2 g + j % 2]
    uint64_t *o_done = p_full + kSB;
    uint64_t *ready = o_done + 4;     // the next piece's Q is in place
    uint64_t *fin = ready + 1;
    uint64_t *o_free = fin + 1;       // [2] a piece's O has been read: by both groups (alternating) / by group g (paired)
    uint64_t *xch_full = o_free + 2;  // [2] group g's (max, sum) of a piece are in xch[g]
    uint64_t *xch_empty = xch_full + 2;  // [2] the other group has read them
    uint64_t *o_last = xch_empty + 2;    // [2] alternating mode: every P V of a piece has completed (per group)
    uint64_t *desc_full = o_last + 2;
    uint64_t *desc_empty = desc_full + kDescs;
    float2 *xch = reinterpret_cast<float2 *>(smem + L::xch);

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
    int *warp_sums = reinterpret_cast<int *>(smem + L::misc + 16);  // [12] + carry
    int *counters = reinterpret_cast<int *>(smem + L::misc + 96);   // partial-store / merge warp counters
    constexpr int kCarry = kThreads / 32;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = a.num_kv_heads, G = a.group, B = a.block_size;
    const int cap = min(a.max_seq_len, a.max_blocks * B);

    // The prologue reads only this call's inputs (lengths, tables, groups),
    // which no kernel of this library writes; the cache, the queries' rows
    // copied later, the workspace and the outputs are touched after the wait.
    grid_dependency_wait();
    grid_launch_dependents();

    if (threadIdx.x == 0) {
        cum[0] = 0;
        warp_sums[kCarry] = 0;
        counters[0] = counters[1] = 0;
    }
    __syncthreads();

    // ---- scan: tiles of every unit (all its contexts, all KV heads) ----
    for (int base = 0; base < a.num_units; base += kThreads) {
        const int u = base + threadIdx.x;
        int v = 0;
        if (u < a.num_units) {
            const int gu = a.unit0 + u;
            if (a.mode == kGrouped) {
                // loads first: a flag's atomic between them would order them one after another
                int m0 = a.group_offsets[gu], m1 = a.group_offsets[gu + 1];
                const int raw = a.prefix_lens[gu];
                if (m0 < 0 || m1 > a.num_seqs || m1 < m0) {
                    if (blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_PREFIX);
                    m0 = m1 = 0;
                }
                if (blockIdx.x == 0 && (gu == 0 && m0 != 0 || gu + 1 == a.num_groups && m1 != a.num_seqs))
                    flag_error(a.err, PKV_DEVERR_PREFIX);
                const int align = B > 16 ? B : 16;
                if (blockIdx.x == 0 && (raw < 0 || raw % align != 0)) flag_error(a.err, PKV_DEVERR_PREFIX);
                int mn = cap;
                for (int mb = m0; mb < m1; mb += 8) {
                    int raw[8];  // eight members' lengths in flight at once
#pragma unroll
                    for (int k = 0; k < 8; ++k) raw[k] = mb + k < m1 ? a.seq_lens[mb + k] : cap;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (blockIdx.x == 0 && (raw[k] < 0 || raw[k] > cap)) flag_error(a.err, PKV_DEVERR_SEQ_LEN);
                        mn = min(mn, clamp_len(raw[k], cap));
                    }
                }
                // with an append, every member's new token stays in its own part
                int pre = min(raw < 0 ? 0 : raw, mn - (a.appended ? 1 : 0));
                pre = m1 > m0 && pre > 0 ? pre / kTok * kTok : 0;
                uval[u] = pre;
                int tot = 0;  // laid-out tiles of the member chunks (one context each per KV head)
                for (int c0 = m0; c0 < m1; c0 += a.per_ctx) {
                    int n = pre / kTok;
                    for (int m = c0; m < min(m1, c0 + a.per_ctx); ++m) n += own_tiles(a, m, pre, cap);
                    tot += laid_out(n);
                }
                v = Hkv * tot;
            } else {
                // loads first: a flag's atomic between them would order them one after another
                int q0 = a.q_starts[gu], q1 = a.q_starts[gu + 1];
                const int raw_len = a.seq_lens[gu];
                if (q0 < 0 || q1 < q0 || q1 > a.num_q_tokens) {
                    if (blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_SEQ_LEN);
                    q0 = q1 = 0;
                }
                const int Lq = clamp_len(raw_len, cap);
                if (blockIdx.x == 0 && ((raw_len < 0 || raw_len > cap) || q1 - q0 > a.max_q_len || q1 - q0 > Lq))
                    flag_error(a.err, PKV_DEVERR_SEQ_LEN);
                const int Q = min(q1 - q0, a.max_q_len);  // queries past max_q_len are not attended
                uval[u] = Q;
                Unit x{};
                x.Q = Q;
                x.L = Lq;
                const int nb = (Q + a.per_ctx - 1) / a.per_ctx;
                int t = 0;
                for (int b = 0; b < nb; ++b) {
                    const int p = block_last_pos(x, b, a.per_ctx);
                    t += laid_out(p < 0 ? 0 : (p + kTok) / kTok);
                }
                v = Hkv * t;
            }
        }
        int x = v;  // inclusive warp scan
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, sh);
            if (lane >= sh) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        int before = warp_sums[kCarry];
        for (int w = 0; w < warp; ++w) before += warp_sums[w];
        if (u < a.num_units) cum[u + 1] = before + x;
        __syncthreads();
        if (threadIdx.x == kThreads - 1) warp_sums[kCarry] = before + x;
        __syncthreads();
    }
    if (threadIdx.x == 0) cum[a.num_units + 1] = cum[a.num_units] + 1;  // sentinel past the last unit
    __syncthreads();
    const int64_t T = cum[a.num_units];

    // ---- rows whose context has no tile: zero output (CTA c takes units c, c + grid, ...) ----
    for (int u = blockIdx.x; u < a.num_units; u += gridDim.x) {
        const Unit x = load_unit(a, uval, u);
        const int per_kvh = (cum[u + 1] - cum[u]) / Hkv;
        for (int sub = 0; sub < x.nsub; ++sub) {
            if (sub_tiles(a, x, sub, per_kvh, cap) > 0) continue;
            const int r0 = x.m0 + sub * a.per_ctx;
            const int r1 = a.mode == kGrouped ? min(x.m1, r0 + a.per_ctx) : x.m0 + min(x.Q, (sub + 1) * a.per_ctx);
            const int per_row = a.num_heads * D / 8;  // 16-byte chunks of one row of out
            for (int i = threadIdx.x; i < (r1 - r0) * per_row; i += kThreads)
                reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + (int64_t)r0 * a.num_heads * D)[i] =
                    make_uint4(0u, 0u, 0u, 0u);
        }
    }

    const int64_t parts = split_parts(T, gridDim.x);
    if (T == 0 || blockIdx.x >= parts) return;  // before any tensor memory is taken
    const int w_me = blockIdx.x;
    const int64_t s0 = (int64_t)w_me * T / parts, s1 = ((int64_t)w_me + 1) * T / parts;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&kv_empty[i], PAIRED ? 2 : 1);  // paired: each group's P V of the tile
        }
        for (int i = 0; i < kSB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&o_done[i], 1);
        mbar_init(ready, PAIRED ? 8 : 4);
        mbar_init(fin, PAIRED ? 2 : 1);  // one commit per MMA-issuing thread
        for (int i = 0; i < 2; ++i) mbar_init(&o_free[i], PAIRED ? 4 : 4 * kSG);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xch_full[i], 4);
            mbar_init(&xch_empty[i], 4);
            mbar_init(&o_last[i], 1);
        }

        for (int i = 0; i < kDescs; ++i) {
            mbar_init(&desc_full[i], 1);
            mbar_init(&desc_empty[i], 4 * kSG + (PAIRED ? 2 : 1));  // softmax warps and the MMA thread (once per group if paired)
        }
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t q_s = smem_u32(smem + L::q);
    const uint32_t ring_s = smem_u32(smem + L::ring);

    if (warp == kProducerWarp) {
        // ======================= producer =======================
        Ctx c;
        bool dead = !c.seek(a, cum, uval, s0, cap);
        if (dead && lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
        int j = 0;  // tiles issued (32-bit: ring slots and phases are cheap to derive)
        int p = 0;      // pieces published
        const int bpt = kTok / B;  // blocks per tile
        for (int64_t t = s0; t < s1 && !dead;) {
            const int64_t ce = c.start + c.n;
            // the context's real tiles in this share; none when the share ends
            // inside its virtual ones
            const int i0 = max(0, (int)(t - c.start) - kPieceTiles), i1 = (int)(min(s1, ce) - c.start) - kPieceTiles;
            if (i1 <= i0) {
                t = min(s1, ce);
                if (t < s1 && !c.next(a, cum, uval, cap)) {
                    if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
                    dead = true;
                }
                continue;
            }
            int row_base, nrows, pos0;
            c.rows(a, row_base, nrows, pos0);
            // members' first own tiles (grouped): mo[k], k = 0 .. members
            int members = 0;
            if (a.mode == kGrouped) {
                const int c0 = row_base, c1 = min(c.x.m1, c0 + a.per_ctx);
                members = c1 - c0;
                __syncwarp();
                for (int k0 = 0; k0 < members; k0 += 32) {
                    const int k = k0 + lane;
                    int v = k < members ? own_tiles(a, c0 + k, c.x.pre, cap) : 0;
                    int x = v;
#pragma unroll
                    for (int sh = 1; sh < 32; sh <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, x, sh);
                        if (lane >= sh) x += y;
                    }
                    const int carry = k0 == 0 ? 0 : mo[k0];
                    if (k < members) mo[k + 1] = carry + x;
                    if (k0 == 0 && lane == 0) mo[0] = 0;
                    __syncwarp();
                }
                __syncwarp();
            }
            // publish the piece
            if (lane == 0) {
                const int d = p % kDescs;
                if (p >= kDescs) wait_or_flag(&desc_empty[d], (uint32_t)(((p / kDescs) - 1) & 1), dead, a.err);
                Piece pc;
                pc.ntiles = i1 - i0;
                pc.row_base = row_base;
                pc.rows = nrows;
                pc.kvh = c.kvh;
                pc.pos0 = pos0;
                const bool first_here = c.start + kPieceTiles >= s0, last_here = ce <= s1;
                pc.kind = first_here ? (last_here ? kWhole : kMerger) : kContinue;
                pc.w0 = (int)share_owner(c.start + kPieceTiles, T, parts);
                pc.w1 = (int)share_owner(ce - 1, T, parts);
                descs[d] = pc;
                mbar_arrive(&desc_full[d]);
            }
            dead = __shfl_sync(0xffffffffu, dead, 0);
            ++p;
            // tiles of the piece, in chunks: first the chunk's tile keys and block
            // ids are staged in shared memory (all loads in flight together),
            // then each tile is issued from there
            const int cht = min(kChunkTiles, kIdCache / bpt);
            for (int k0 = i0; k0 < i1 && !dead; k0 += cht) {
                const int k1 = min(i1, k0 + cht);
                __syncwarp();
                for (int i = k0 + lane; i < k1; i += 32) {
                    const TileKeys tk = tile_keys(a, c, mo, members, i, cap);
                    tkc[i - k0] = make_int4(tk.key0, tk.nvalid, tk.member, tk.seq);
                }
                __syncwarp();
                for (int e = lane; e < (k1 - k0) * bpt; e += 32) {
                    const int4 tk = tkc[e / bpt];
                    const int jb = e % bpt;
                    ids[e] = jb * B < tk.y ? a.block_tables[(int64_t)tk.w * a.max_blocks + tk.x / B + jb] : INT_MIN;
                }
                __syncwarp();
                for (int i = k0; i < k1; ++i, ++j) {
                    const int st = (int)(j % NS);
                    if (lane == 0 && j >= NS) wait_or_flag(&kv_empty[st], (uint32_t)(((j / NS) - 1) & 1), dead, a.err);
                    dead = __shfl_sync(0xffffffffu, dead, 0);
                    if (dead) break;
                    const int4 tk = tkc[i - k0];
                    const int nblk = (tk.y + B - 1) / B;
                    // lane jb < nblk checks block jb's id (an invalid id is read as block 0, its keys masked)
                    int id = 0;
                    if (lane < nblk) id = ids[(i - k0) * bpt + lane];
                    const bool bad = lane < nblk && (id < 0 || id >= a.num_blocks);
                    const uint32_t badm = __ballot_sync(0xffffffffu, bad);
                    if (lane == 0) {
                        if (badm) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                        TileInfo ti;
                        ti.member = tk.z;
                        ti.nvalid = tk.y;
                        ti.bad = badm;
                        ti.key0 = tk.x;
                        tinfo[st] = ti;
                        mbar_arrive_expect_tx(&k_full[st], (uint32_t)(nblk * H * B * 128));
                        mbar_arrive_expect_tx(&v_full[st], (uint32_t)(nblk * H * B * 128));
                    }
                    __syncwarp();
                    // boxes, one lane each: K by (block, half), then V by block (the
                    // whole (block, kv head) slab, both column halves)
                    for (int bi = lane; bi < nblk * (H + 1); bi += 32) {
                        const bool isv = bi >= nblk * H;
                        const int jb = isv ? bi - nblk * H : bi / H, h = isv ? 0 : bi % H;
                        const int bid = ids[(i - k0) * bpt + jb];
                        const int b2 = (bid < 0 || bid >= a.num_blocks) ? 0 : bid;
                        const int y = (int)(((int64_t)b2 * Hkv + c.kvh) * B);
                        const uint32_t stage = ring_s + st * L::kStageBytes;
                        if (isv)
                            tma_load_3d(stage + L::kKVBytes + jb * (H * B * 128), &tm_v, smem_u32(&v_full[st]), 0, y, 0);
                        else
                            tma_load_2d(stage + h * (kTok * 128) + jb * B * 128, &tm_k, smem_u32(&k_full[st]), h * 64, y);
                    }
                }
            }
            t = min(s1, ce);
            if (t < s1 && !c.next(a, cum, uval, cap)) {
                if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
                dead = true;
            }
        }
        // end of the share: a descriptor with no tiles
        if (lane == 0 && !dead) {
            const int d = p % kDescs;
            if (p >= kDescs) wait_or_flag(&desc_empty[d], (uint32_t)(((p / kDescs) - 1) & 1), dead, a.err);
            Piece pc{};
            pc.ntiles = 0;
            descs[d] = pc;
            mbar_arrive(&desc_full[d]);
        }
        // copies still in flight (only after a timeout) land before the CTA exits
        if (lane == 0 && dead)
            for (int k = max(0, j - NS); k < j; ++k) {
                mbar_wait_bounded(&k_full[k % NS], (uint32_t)((k / NS) & 1));
                mbar_wait_bounded(&v_full[k % NS], (uint32_t)((k / NS) & 1));
            }
    } else if (warp == kMmaWarp || (PAIRED && warp == kMma1Warp)) {
        // ======================= MMA issuer(s) =======================
        if (lane == 0) {
            constexpr uint32_t idesc_pv = tc::instr_desc(D, true);
            constexpr uint32_t idesc_qk = tc::instr_desc(kTok, false);
            // P V: 16 keys per MMA; V's 64-column halves are B rows apart, its
            // 8-row groups 1024 bytes apart inside a block (blocks of 8: a block apart)
            const uint32_t pv_lbo = (uint32_t)(B * 128), pv_sbo = B >= 16 ? 1024u : (uint32_t)(H * B * 128);
            // descriptors advance by (byte offset >> 4) in their start-address field
            uint32_t pv_off[kTok / 16];
#pragma unroll
            for (int k = 0; k < kTok / 16; ++k) pv_off[k] = (uint32_t)((16 * k / B) * (H * B * 128) + (16 * k % B) * 128);
            const uint64_t qd = tc::smem_desc(q_s, 16, 1024);
            if constexpr (PAIRED) {
                // Paired contexts: group g's Q K^T and P V of every tile (Q at q + g *
                // kQTile, S / P in the group's two buffers, O at kOBase + g * D), issued
                // by the group's own thread (warp kMmaWarp: group 0, kMma1Warp: group 1).
                // One thread issuing both groups' instructions next to busy softmax
                // warps was the limit; two threads on two schedulers halve it.
                const int g = warp == kMmaWarp ? 0 : 1;
                const uint64_t qdg = tc::smem_desc(q_s + (uint32_t)g * L::kQTile, 16, 1024);
                const uint32_t ob = kOBase + (uint32_t)g * D;
                int jq = 0, jp = 0;  // next Q K^T tile, next P V tile
                int pq = 0, pp = 0;  // their pieces
                int tq = 0, tp = 0;  // tile within those pieces
                int ntq = -1;
                bool done_q = false, dead = false;
                uint32_t idle = 0;
                for (;;) {
                    bool prog = false;
                    if (jp < jq) {
                        const int sb = sbuf<true>(jp, g);
                        if (mbar_test_wait(&p_full[sb], sphase<true>(jp)) &&
                            mbar_test_wait(&v_full[jp % NS], (uint32_t)((jp / NS) & 1)) &&
                            (tp > 0 || pp == 0 || mbar_test_wait(&o_free[g], (uint32_t)((pp - 1) & 1)))) {
                            tc::fence_after();
                            const uint32_t pa = tmem + (uint32_t)sb * kTok;
                            const uint32_t vb = ring_s + (uint32_t)(jp % NS) * L::kStageBytes + L::kKVBytes;
                            const uint64_t vd = tc::smem_desc(vb, pv_lbo, pv_sbo);
#pragma unroll
                            for (int k = 0; k < kTok / 16; ++k)
                                tc::mma_ts(tmem + ob, pa + 8 * k, vd + (uint64_t)(pv_off[k] >> 4), idesc_pv,
                                           (tp == 0 && k == 0) ? 0u : 1u);
                            tc::commit(&o_done[2 * g + (jp & 1)]);
                            tc::commit(&kv_empty[jp % NS]);
                            ++jp;
                            if (++tp == descs[pp % kDescs].ntiles) {
                                mbar_arrive(&desc_empty[pp % kDescs]);
                                ++pp;
                                tp = 0;
                            }
                            prog = true;
                        }
                    }
                    if (done_q && jp >= jq) break;
                    if (!done_q && jq < jp + 2) {
                        if (ntq < 0 && mbar_test_wait(&desc_full[pq % kDescs], (uint32_t)((pq / kDescs) & 1))) {
                            ntq = descs[pq % kDescs].ntiles;
                            if (ntq == 0) done_q = true;
                            prog = true;
                        }
                        if (ntq > 0 && mbar_test_wait(&k_full[jq % NS], (uint32_t)((jq / NS) & 1)) &&
                            (tq > 0 || mbar_test_wait(ready, (uint32_t)(pq & 1)))) {
                            tc::fence_after();
                            const uint32_t kb = ring_s + (uint32_t)(jq % NS) * L::kStageBytes;
                            const uint64_t kd = tc::smem_desc(kb, 16, 1024);
                            const int sb = sbuf<true>(jq, g);
#pragma unroll
                            for (int k = 0; k < D / 16; ++k)
                                tc::mma(tmem + (uint32_t)sb * kTok,
                                        qdg + (uint64_t)(((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4),
                                        kd + (uint64_t)(((k >> 2) * (kTok * 128) + (k & 3) * 32) >> 4), idesc_qk,
                                        k > 0 ? 1u : 0u);
                            tc::commit(&s_full[sb]);
                            ++jq;
                            if (++tq == ntq) {
                                ++pq;
                                tq = 0;
                                ntq = -1;
                            }
                            prog = true;
                        }
                    }
                    if (prog) {
                        idle = 0;
                    } else if (++idle > kWaitLimit) {
                        flag_error(a.err, PKV_DEVERR_TIMEOUT);
                        dead = true;
                        break;
                    }
                }
                (void)dead;
            } else {
                int jq = 0, jp = 0;           // next Q K^T / P V tile
                int pq = 0, pp = 0;           // their pieces
                int tq = 0, tp = 0;           // tile within those pieces
                int ntq = -1;                 // tiles of piece pq (-1: descriptor not read yet)
                bool done_q = false, dead = false;
                uint32_t idle = 0;
                for (;;) {
                    bool prog = false;
                    if (jp < jq) {
                        // P V of tile jp into its softmax group's O; the first P V of a
                        // piece waits until the previous piece's O has been read
                        const int sb = sbuf<false>(jp, 0);
                        if (mbar_test_wait(&p_full[sb], sphase<false>(jp)) &&
                            mbar_test_wait(&v_full[jp % NS], (uint32_t)((jp / NS) & 1)) &&
                            (tp > 0 || pp == 0 || mbar_test_wait(o_free, (uint32_t)((pp - 1) & 1)))) {
                            tc::fence_after();
                            const uint32_t ob = kOBase + (uint32_t)(jp & 1) * D;
                            const uint32_t pa = tmem + (uint32_t)sb * kTok;  // P in the S columns
                            const uint32_t vb = ring_s + (uint32_t)(jp % NS) * L::kStageBytes + L::kKVBytes;
                            const uint64_t vd = tc::smem_desc(vb, pv_lbo, pv_sbo);
    #pragma unroll
                            for (int k = 0; k < kTok / 16; ++k)
                                tc::mma_ts(tmem + ob, pa + 8 * k, vd + (uint64_t)(pv_off[k] >> 4), idesc_pv,
                                           (tp < kSG && k == 0) ? 0u : 1u);  // a group's first tile of the piece starts O
                            tc::commit(&o_done[jp & 1]);
                            tc::commit(&kv_empty[jp % NS]);
                            ++jp;
                            if (++tp == descs[pp % kDescs].ntiles) {
                                // the piece's P V are all issued: one phase of o_last per
                                // group (its softmax waits for it before reading O)
                                tc::commit(&o_last[0]);
                                tc::commit(&o_last[1]);
                                mbar_arrive(&desc_empty[pp % kDescs]);
                                ++pp;
                                tp = 0;
                            }
                            prog = true;
                        }
                    } else if (done_q) {
                        break;
                    }
                    // Q K^T of tile jq once its S buffer is free: the buffer's last user,
                    // tile jq - kSB, has had its P V issued (the tensor pipe runs in order)
                    if (!done_q && jq < jp + kSB) {
                        if (ntq < 0 && mbar_test_wait(&desc_full[pq % kDescs], (uint32_t)((pq / kDescs) & 1))) {
                            ntq = descs[pq % kDescs].ntiles;
                            if (ntq == 0) done_q = true;
                            prog = true;
                        }
                        if (ntq > 0 && mbar_test_wait(&k_full[jq % NS], (uint32_t)((jq / NS) & 1)) &&
                            (tq > 0 || mbar_test_wait(ready, (uint32_t)(pq & 1)))) {
                            tc::fence_after();
                            const uint32_t kb = ring_s + (uint32_t)(jq % NS) * L::kStageBytes;
                            const uint64_t kd = tc::smem_desc(kb, 16, 1024);
                            const int sb = sbuf<false>(jq, 0);
    #pragma unroll
                            for (int k = 0; k < D / 16; ++k)
                                tc::mma(tmem + (uint32_t)sb * kTok,
                                        qd + (uint64_t)(((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4),
                                        kd + (uint64_t)(((k >> 2) * (kTok * 128) + (k & 3) * 32) >> 4), idesc_qk,
                                        k > 0 ? 1u : 0u);
                            tc::commit(&s_full[sb]);
                            ++jq;
                            if (++tq == ntq) {
                                ++pq;
                                tq = 0;
                                ntq = -1;
                            }
                            prog = true;
                        }
                    }
                    if (prog) {
                        idle = 0;
                    } else if (++idle > kWaitLimit) {
                        flag_error(a.err, PKV_DEVERR_TIMEOUT);
                        dead = true;
                        break;
                    }
                }
            }
            // every MMA (of both issuing threads) has completed before the tensor memory is freed
            tc::commit(fin);
            mbar_wait_bounded(fin, 0u);
        }
    } else if (warp == kAuxWarp) {
        // ======================= members' block tables =======================
        if (a.mode == kGrouped) {
            Ctx c;
            const bool found = c.seek(a, cum, uval, s0, cap);
            const int bpt = kTok / B;
            bool bad = false;
            for (int64_t t = s0; t < s1 && found;) {
                const int64_t ce = c.start + c.n;
                const int i0 = max(0, (int)(t - c.start) - kPieceTiles), i1 = (int)(min(s1, ce) - c.start) - kPieceTiles;
                const int npt = c.x.pre / kTok;
                if (c.kvh == 0 && i0 < npt && i0 < i1) {
                    const int c0 = c.x.m0 + c.sub * a.per_ctx, c1 = min(c.x.m1, c0 + a.per_ctx);
                    const int lb0 = i0 * bpt, nb = (min(i1, npt) - i0) * bpt;
                    const int32_t *lead = a.block_tables + (int64_t)c.x.m0 * a.max_blocks;
                    const int total = (c1 - c0) * nb;
                    for (int k = lane; k < total; k += 32) {
                        const int m = c0 + k / nb, lb = lb0 + k % nb;
                        if (m != c.x.m0 && a.block_tables[(int64_t)m * a.max_blocks + lb] != lead[lb]) bad = true;
                    }
                }
                t = min(s1, ce);
                if (t < s1 && !c.next(a, cum, uval, cap)) break;
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) flag_error(a.err, PKV_DEVERR_PREFIX);
        }
    } else if (warp < 4 * kSG) {
        if constexpr (PAIRED) {
            // ============ softmax, paired contexts: group g owns rows g * 128 .. ============
            // Both groups take every tile of a piece; each keeps its rows' running
            // max and sum and its own O, and writes its rows' result.
            const int g = warp >> 2, wq = warp & 3;
            const int rr = wq * 32 + lane;  // TMEM lane and row of the group's Q tile
            const int cr = g * kRows + rr;  // row of the context
            const uint32_t trow = tmem + ((uint32_t)(wq * 32) << 16);
            bool dead = false;
            int p = 0;
            // P V of the group's tile x has completed: o_done[2 g + x % 2] completes
            // one phase per P V of that parity.  A wait for tile x is only made once
            // S of tile x (or a later one) has landed: the group's MMA thread issued
            // Q K^T of x after P V of x - 2 (that S buffer's previous user), and a
            // commit signals only when every earlier MMA of its thread is done, so
            // the barrier's previous phase (tile x - 2) is complete, and its next one
            // (tile x + 2) cannot be, P V of x + 2 needing P that is not yet out.
            auto wait_pv = [&](int x) {
                if (x >= 0) wait_or_flag(&o_done[2 * g + (x & 1)], (uint32_t)((x >> 1) & 1), dead, a.err);
            };
            auto copy_q = [&](const Piece &pc) {
                const bool live = cr < pc.rows;
                const int row = pc.row_base + (live ? cr / G : 0), head = pc.kvh * G + cr % G;
                const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)row * a.num_heads + head) * D;
#pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    const uint32_t dst = q_s + (uint32_t)g * L::kQTile + (k >> 3) * (kRows * 128) + rr * 128 +
                                         (((k & 7) ^ (rr & 7)) << 4);
                    if (live)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + k * 8) : "memory");
                    else
                        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
            auto q_ready = [&]() {
                asm volatile("cp.async.wait_all;" ::: "memory");
                fence_proxy_async();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ready);
            };
            Piece pc{};
            if (wait_or_flag(&desc_full[0], 0u, dead, a.err)) pc = descs[0];
            if (pc.ntiles > 0) {
                copy_q(pc);
                q_ready();
            }
            int j0 = 0;
            while (pc.ntiles > 0 && !dead) {
                const bool live_warp = g * kRows + wq * 32 < pc.rows;
                const bool live = cr < pc.rows;
                const int my_pos = pc.pos0 + cr / G;  // this row's position
                const int jl = j0 + pc.ntiles - 1;
                float m_run = -INFINITY, l = 0.f;
                Piece nx{};
                bool copied = false;
                for (int j = j0; j <= jl; ++j) {
                    const int st = j % NS, b = sbuf<true>(j, g);
                    wait_or_flag(&k_full[st], (uint32_t)((j / NS) & 1), dead, a.err);
                    const TileInfo ti = tinfo[st];
                    wait_or_flag(&s_full[b], sphase<true>(j), dead, a.err);
                    tc::fence_after();
                    if (dead) break;
                    if (j == jl) {
                        // every Q K^T of this piece has completed: Q may take the next piece's rows
                        const int d = (p + 1) % kDescs;
                        if (wait_or_flag(&desc_full[d], (uint32_t)(((p + 1) / kDescs) & 1), dead, a.err)) nx = descs[d];
                        if (nx.ntiles > 0) {
                            copy_q(nx);
                            copied = true;
                        }
                    }
                    // keys past the context's end or in invalid blocks: their V rows are
                    // zeroed before this group's P is released.  Both groups zero them (the
                    // same rows, the same zeros), so neither group's P V waits on the other.
                    if (ti.nvalid < kTok || ti.bad) {
                        wait_or_flag(&v_full[st], (uint32_t)((j / NS) & 1), dead, a.err);
                        const uint32_t vbase = ring_s + st * L::kStageBytes + L::kKVBytes;
                        for (int e = rr; e < kTok * H * 8; e += kRows) {
                            const int key = (e / 8) % kTok, h = e / (kTok * 8), chk = e % 8;
                            const bool zero = key >= ti.nvalid || ((ti.bad >> (key / B)) & 1u);
                            const uint32_t row = vbase + (key / B) * (H * B * 128) + h * (B * 128) + (key % B) * 128;
                            if (zero) asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(row + chk * 16), "r"(0u) : "memory");
                        }
                        fence_proxy_async();
                    }
                    if (live_warp) {
                        int lim = live ? min(ti.nvalid, my_pos - ti.key0 + 1) : 0;
                        const int bshift = B == 8 ? 3 : (B == 16 ? 4 : 5);
                        bool move = false;
                        float alpha = 1.f;
                        const uint32_t sp = trow + b * kTok;
                        softmax_tile<4>(sp, 0, lim, ti.bad, bshift, a.scale_log2, m_run, l, move, alpha);
                        if (__any_sync(0xffffffffu, move)) {
                            wait_pv(j - 1);
                            tc::fence_after();
                            const uint32_t ob = kOBase + (uint32_t)g * D;
#pragma unroll 1
                            for (int cc = 0; cc < D / 32; ++cc) {
                                float o[32];
                                tc::ld32(trow + ob + cc * 32, o);
                                tc::wait_ld();
#pragma unroll
                                for (int k = 0; k < 32; ++k) o[k] *= alpha;
                                tc::st32(trow + ob + cc * 32, o);
                            }
                            tc::wait_st();
                        }
                    }
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[b]);
                }
                if (dead) break;
                if (copied) q_ready();  // the next piece's Q K^T may start
                wait_pv(jl - 1);  // the group's last P V of each parity, in order
                wait_pv(jl);
                tc::fence_after();
                auto load_o = [&](int cc, float (&o)[16]) {
                    ld16(trow + kOBase + (uint32_t)g * D + cc * 16, o);
                    tc::wait_ld();
                };
                finish_piece<D>(a, pc, m_run, l, load_o, cr, 2 * kRows, live, live_warp, lane, w_me, G, 7, counters,
                                &o_free[g]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&desc_empty[p % kDescs]);
                pc = nx;
                j0 = jl + 1;
                ++p;
            }
            asm volatile("cp.async.wait_all;" ::: "memory");  // no query copy outlives the CTA
        } else {
            // ======================= softmax (two groups of warps 0-3, 4-7) =======================
            // Group g takes the tiles j with j % 2 == g of every piece, with its own
            // running max and sum per row and its own O accumulator in tensor memory
            // (two independent chains per SM).  Thread rr of a group owns query row
            // rr = TMEM lane rr.  At a piece's end the two groups' partial softmax
            // states are combined (as in a split context), each group taking half
            // of the columns.
            const int g = warp >> 2, wq = warp & 3;
            const int rr = wq * 32 + lane;
            const uint32_t trow = tmem + ((uint32_t)(wq * 32) << 16);
            bool dead = false;
            int p = 0;
            // P V of tile x has completed.  o_done[x & 1] completes one phase per P V
            // of that parity (one group's tiles), and a parity wait is only meaningful
            // for the barrier's current or preceding phase.  It is waited for only
            // before a rescale of O, for the group's tile j - 2 once S of its tile j
            // has landed: the MMA thread issued Q K^T of j after P V of j - 4 (the S
            // buffer's previous user), and a commit signals only when every earlier
            // MMA of the thread is done, so the previous phase is complete and the
            // next (P V of j, needing P that is not yet out) is not.  At a piece's
            // end the group waits on o_last instead: one phase per piece.
            auto wait_pv = [&](int x) {
                if (x >= 0) wait_or_flag(&o_done[x & 1], (uint32_t)((x >> 1) & 1), dead, a.err);
            };
            // this thread's query row of a piece into Q (128-byte swizzled, K-major; zero past the live rows)
            auto copy_q = [&](const Piece &pc) {
                const bool live = rr < pc.rows;
                const int row = pc.row_base + (live ? rr / G : 0), head = pc.kvh * G + rr % G;
                const int r = rr;
                const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)row * a.num_heads + head) * D;
    #pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    const uint32_t dst = q_s + (k >> 3) * (kRows * 128) + r * 128 + (((k & 7) ^ (r & 7)) << 4);
                    if (live)
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + k * 8) : "memory");
                    else
                        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
            auto q_ready = [&]() {
                asm volatile("cp.async.wait_all;" ::: "memory");
                fence_proxy_async();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ready);
            };
            Piece pc{};
            if (wait_or_flag(&desc_full[0], 0u, dead, a.err)) pc = descs[0];
            if (g == 0 && pc.ntiles > 0) {
                copy_q(pc);
                q_ready();
            }
            int j0 = 0;  // the piece's first tile
            while (pc.ntiles > 0 && !dead) {
                const bool live_warp = wq * 32 < pc.rows;
                const bool live = rr < pc.rows;
                const int my_member = rr / G;
                const int my_pos = pc.pos0 + rr / G;      // multi-token: this row's position
                const int jl = j0 + pc.ntiles - 1;       // the piece's last tile
                float m_run = -INFINITY, l = 0.f;
                Piece nx{};
                bool have_nx = false, copied = false;
                for (int j = j0 + ((j0 & 1) != g ? 1 : 0); j <= jl; j += kSG) {
                    const int st = j % NS, b = sbuf<false>(j, g);
                    // the stage's record (ordered by the producer's arrive on k_full)
                    wait_or_flag(&k_full[st], (uint32_t)((j / NS) & 1), dead, a.err);
                    const TileInfo ti = tinfo[st];
                    wait_or_flag(&s_full[b], sphase<false>(j), dead, a.err);
                    tc::fence_after();
                    if (dead) break;
                    if (j == jl) {
                        // every Q K^T of this piece has completed: Q may take the next piece's rows
                        const int d = (p + 1) % kDescs;
                        if (wait_or_flag(&desc_full[d], (uint32_t)(((p + 1) / kDescs) & 1), dead, a.err)) nx = descs[d];
                        have_nx = true;
                        if (nx.ntiles > 0) {
                            copy_q(nx);
                            copied = true;
                        }
                    }
                    // keys past the context's end or in invalid blocks: zero their V rows
                    // (stale slots may hold NaN; a zero weight must meet a zero)
                    if (ti.nvalid < kTok || ti.bad) {
                        wait_or_flag(&v_full[st], (uint32_t)((j / NS) & 1), dead, a.err);  // V landed: zero after it
                        const uint32_t vbase = ring_s + st * L::kStageBytes + L::kKVBytes;
                        for (int e = rr; e < kTok * H * 8; e += kRows) {
                            const int key = (e / 8) % kTok, h = e / (kTok * 8), chk = e % 8;
                            const bool zero = key >= ti.nvalid || ((ti.bad >> (key / B)) & 1u);
                            const uint32_t row = vbase + (key / B) * (H * B * 128) + h * (B * 128) + (key % B) * 128;
                            if (zero) asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(row + chk * 16), "r"(0u) : "memory");
                        }
                        fence_proxy_async();
                    }
                    if (live_warp) {
                        // keys this row sees in this tile: [0, lim) minus invalid blocks
                        int lim = ti.nvalid;
                        if (!live) lim = 0;
                        if (ti.member >= 0 && ti.member != my_member) lim = 0;
                        if (a.mode == kMulti) lim = min(lim, my_pos - ti.key0 + 1);
                        const int bshift = B == 8 ? 3 : (B == 16 ? 4 : 5);
                        bool move = false;
                        float alpha = 1.f;
                        const uint32_t sp = trow + b * kTok;
                        softmax_tile<4>(sp, 0, lim, ti.bad, bshift, a.scale_log2, m_run, l, move, alpha);
                        if (__any_sync(0xffffffffu, move)) {
                            // the running max moved: the group's O (which must hold P V of
                            // its previous tile first) is rescaled before this tile's P V
                            wait_pv(j - kSG);
                            tc::fence_after();
                            const uint32_t ob = kOBase + (uint32_t)g * D;
    #pragma unroll 1
                            for (int cc = 0; cc < D / 32; ++cc) {
                                float o[32];
                                tc::ld32(trow + ob + cc * 32, o);
                                tc::wait_ld();
    #pragma unroll
                                for (int k = 0; k < 32; ++k) o[k] *= alpha;
                                tc::st32(trow + ob + cc * 32, o);
                            }
                            tc::wait_st();
                        }
                    }
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[b]);
                }
                if (dead) break;
                if (!have_nx) {
                    const int d = (p + 1) % kDescs;
                    if (wait_or_flag(&desc_full[d], (uint32_t)(((p + 1) / kDescs) & 1), dead, a.err)) nx = descs[d];
                }
                if (copied) q_ready();  // the next piece's Q K^T may start
                // this group's part of the piece: its O (TMEM) with each row's running max and sum
                const bool has0 = pc.ntiles >= kSG || (j0 & 1) == 0, has1 = pc.ntiles >= kSG || (j0 & 1) == 1;
                const bool has_me = g == 0 ? has0 : has1;
                // every P V of the piece has completed (each group waits every piece,
                // so o_last is never more than one phase ahead of its waiter)
                wait_or_flag(&o_last[g], (uint32_t)(p & 1), dead, a.err);
                tc::fence_after();
                // Both groups finish the piece: each hands its rows' (max, sum) to the
                // other, then combines both O parts for its half of the columns (group
                // g: 16-column chunks g * kNc / 2 ..), so neither waits while the other
                // reads tensor memory and writes.
                if (p > 0) wait_or_flag(&xch_empty[g], (uint32_t)((p - 1) & 1), dead, a.err);
                const float2 mine = has_me ? make_float2(m_run, l) : make_float2(-INFINITY, 0.f);
                xch[g * kRows + rr] = mine;
                __syncwarp();
                if (lane == 0) mbar_arrive(&xch_full[g]);
                float2 other = make_float2(-INFINITY, 0.f);
                if (wait_or_flag(&xch_full[1 - g], (uint32_t)(p & 1), dead, a.err)) other = xch[(1 - g) * kRows + rr];
                __syncwarp();
                if (lane == 0) mbar_arrive(&xch_empty[1 - g]);
                tc::fence_after();
                {
                    const float2 x0 = g == 0 ? mine : other, x1 = g == 0 ? other : mine;
                    // both parts on the common max M: o = sum_g O_g 2^(m_g - M), L likewise
                    // (the same arithmetic on the same values in both groups)
                    const float m0 = has0 ? x0.x : -INFINITY, m1 = has1 ? x1.x : -INFINITY;
                    const float Mc = fmaxf(m0, m1);
                    const float Mr = Mc == -INFINITY ? 0.f : Mc;
                    const float f0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - Mr);
                    const float f1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - Mr);
                    const float Lc = (has0 ? x0.y : 0.f) * f0 + (has1 ? x1.y : 0.f) * f1;
                    const float M = Mc;
                    auto load_o = [&](int cc, float (&o)[16]) {
                        // the piece's combined, unnormalised O (16 columns)
                        float o1[16];
                        if (has0) ld16(trow + kOBase + cc * 16, o);
                        if (has1) ld16(trow + kOBase + D + cc * 16, o1);
                        tc::wait_ld();
    #pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = (has0 ? o[k] * f0 : 0.f) + (has1 ? o1[k] * f1 : 0.f);
                    };
                    const int64_t orow = (int64_t)(pc.row_base + (live ? rr / G : 0)) * a.num_heads + pc.kvh * G + rr % G;
                    constexpr int kNc = D / 16;  // 16-column chunks of an O row
                    // the piece's result: final rows, a partial for the merger, or the merge
                    float f = 1.f, e_own = 1.f, Mtr = 0.f;
                    bool got = true;
                    // merger: the first kMergeHeld other pieces' (max, sum) and scale,
                    // read once; later pieces (long contexts only) are re-read per chunk
                    float2 mlh[kMergeHeld];
                    float eh[kMergeHeld];
    #pragma unroll
                    for (int i = 0; i < kMergeHeld; ++i) {
                        mlh[i] = make_float2(-INFINITY, 0.f);
                        eh[i] = 0.f;
                    }
                    if (pc.kind == kWhole) {
                        f = Lc > 0.f ? 1.f / Lc : 0.f;
                    } else if (pc.kind == kContinue) {
                        if (live && g == 0)
                            *reinterpret_cast<float2 *>(a.part_ml + ((int64_t)w_me * kRows + rr) * 2) = make_float2(M, Lc);
                    } else if (live_warp) {
                        // merger: this piece holds the context's first tile and is the
                        // last piece of this share; CTAs w0 + 1 .. w1 stored the rest
                        const int n = pc.w1 - pc.w0;
                        got = wait_flags_bounded(a.flags + pc.w0 + 1, n, a.tag, lane);
                        if (!got && lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
                        float Mt = M;
    #pragma unroll
                        for (int i = 0; i < kMergeHeld; ++i) {
                            if (live && i < n)
                                mlh[i] = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + (int64_t)(pc.w0 + 1 + i) * kRows + rr);
                            Mt = fmaxf(Mt, mlh[i].x);
                        }
                        if (live)
                            for (int w = pc.w0 + 1 + kMergeHeld; w <= pc.w1; ++w)
                                Mt = fmaxf(Mt, __ldcg(a.part_ml + ((int64_t)w * kRows + rr) * 2));
                        Mtr = Mt == -INFINITY ? 0.f : Mt;
                        e_own = M == -INFINITY ? 0.f : ex2_approx(M - Mtr);
                        float Ls = Lc * e_own;
    #pragma unroll
                        for (int i = 0; i < kMergeHeld; ++i)
                            if (mlh[i].x != -INFINITY) {
                                eh[i] = ex2_approx(mlh[i].x - Mtr);
                                Ls += mlh[i].y * eh[i];
                            }
                        if (live)
                            for (int w = pc.w0 + 1 + kMergeHeld; w <= pc.w1; ++w) {
                                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + (int64_t)w * kRows + rr);
                                if (ml.x != -INFINITY) Ls += ml.y * ex2_approx(ml.x - Mtr);
                            }
                        // NaN rows when a piece never came (flagged above)
                        f = got ? (Ls > 0.f ? 1.f / Ls : 0.f) : __int_as_float(0x7fc00000);
                    }
                    for (int cc = g * (kNc / 2); cc < (g + 1) * (kNc / 2); ++cc) {
                        if (live_warp) {
                            // the held partials' 16 columns: in flight with the tensor-memory load
                            float4 ph[kMergeHeld][4];
    #pragma unroll
                            for (int i = 0; i < kMergeHeld; ++i)
                                if (live && pc.kind == kMerger && mlh[i].x != -INFINITY) {
                                    const float4 *src = reinterpret_cast<const float4 *>(
                                        a.part_o + ((int64_t)(pc.w0 + 1 + i) * kRows + rr) * D + cc * 16);
    #pragma unroll
                                    for (int k = 0; k < 4; ++k) ph[i][k] = __ldcg(src + k);
                                }
                            float o[16];
                            load_o(cc, o);
                            if (live) {
                                if (pc.kind == kContinue) {
                                    store_part16(a.part_o + ((int64_t)w_me * kRows + rr) * D + cc * 16, o);
                                } else {
                                    if (pc.kind == kMerger) {
    #pragma unroll
                                        for (int k = 0; k < 16; ++k) o[k] *= e_own;
    #pragma unroll
                                        for (int i = 0; i < kMergeHeld; ++i)
                                            if (mlh[i].x != -INFINITY) {
    #pragma unroll
                                                for (int k = 0; k < 4; ++k) {
                                                    o[4 * k] += eh[i] * ph[i][k].x;
                                                    o[4 * k + 1] += eh[i] * ph[i][k].y;
                                                    o[4 * k + 2] += eh[i] * ph[i][k].z;
                                                    o[4 * k + 3] += eh[i] * ph[i][k].w;
                                                }
                                            }
                                        for (int w = pc.w0 + 1 + kMergeHeld; w <= pc.w1; ++w) {
                                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + (int64_t)w * kRows + rr);
                                            if (ml.x == -INFINITY) continue;
                                            const float e = ex2_approx(ml.x - Mtr);
                                            const float4 *src =
                                                reinterpret_cast<const float4 *>(a.part_o + ((int64_t)w * kRows + rr) * D + cc * 16);
    #pragma unroll
                                            for (int k = 0; k < 4; ++k) {
                                                const float4 v = __ldcg(src + k);
                                                o[4 * k] += e * v.x;
                                                o[4 * k + 1] += e * v.y;
                                                o[4 * k + 2] += e * v.z;
                                                o[4 * k + 3] += e * v.w;
                                            }
                                        }
                                    }
                                    store_out16(static_cast<__nv_bfloat16 *>(a.out) + orow * D + cc * 16, o, f,
                                                (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0u);
                                }
                            }
                        }
                    }
                    // both O parts of this group's columns have been read: once both
                    // groups have, the next piece's P V may start
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(o_free);
                    if (pc.kind == kContinue) {
                        // a later piece of a context begun in an earlier share: the partial
                        // is stored; the last of the eight warps to finish raises the flag
                        fence_acq_rel_gpu();
                        __syncwarp();
                        if (lane == 0) {
                            fence_acq_rel_gpu();
                            if (atomicAdd(&counters[0], 1) == 4 * kSG - 1) {
                                counters[0] = 0;
                                fence_acq_rel_gpu();
                                *reinterpret_cast<volatile unsigned long long *>(a.flags + w_me) = a.tag;
                            }
                        }
                    } else if (pc.kind == kMerger) {
                        // the last warp done reading clears the flags (a graph replay reuses the tag)
                        __syncwarp();
                        if (lane == 0 && atomicAdd(&counters[1], 1) == 4 * kSG - 1) {
                            counters[1] = 0;
                            for (int k = 0; k < pc.w1 - pc.w0; ++k) a.flags[pc.w0 + 1 + k] = 0ull;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&desc_empty[p % kDescs]);
                pc = nx;
                j0 = jl + 1;
                ++p;
            }
            asm volatile("cp.async.wait_all;" ::: "memory");  // no query copy outlives the CTA
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t o_off, ml_off, flags_off, total;
};

// Per CTA slot (at most kMaxCtas): the partial (o, max, sum) of its first
// piece for each of `rows` rows (kRows; 2 kRows for paired contexts), and a
// ready flag.
static WsLayout ws_layout(int D, int rows) {
    WsLayout w;
    w.o_off = 0;
    w.ml_off = round256((size_t)kMaxCtas * rows * D * 4);
    w.flags_off = w.ml_off + round256((size_t)kMaxCtas * rows * 2 * 4);
    w.total = w.flags_off + round256((size_t)kMaxCtas * 8);
    return w;
}

// 3-D view of a bf16 cache for one box per (block, kv head) slab: dims (64
// columns, rows = num_blocks * Hkv * B, D / 64 column halves) with strides
// (D * 2 bytes per row, 128 bytes per half); box (64, B, D / 64), 128-byte
// swizzle.  The slab lands as [half][block row][128 B].
static bool make_slab_map(CUtensorMap *map, const void *base, int64_t rows, int D, int B) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128u};
    cuuint32_t box[3] = {64u, (cuuint32_t)B, (cuuint32_t)(D / 64)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K: the 2-D view (64 columns x B rows per box); V: the slab view.
static bool make_maps(const void *k_cache, const void *v_cache, int64_t rows, int D, int B, CUtensorMap *mk,
                      CUtensorMap *mv) {
    return make_cache_map(mk, k_cache, rows, D, B) && make_slab_map(mv, v_cache, rows, D, B);
}

template <int D, bool PAIRED>
static pkv_status launch(const Args &a, const void *k_cache, const void *v_cache, cudaStream_t st) {
    constexpr int smem = Layout<D, PAIRED>::total;
    static bool done[128] = {};
    auto kern = rows_attention_kernel<D, PAIRED>;
    if (!ensure_smem(kern, smem, done)) return PKV_ERR_CUDA;
    CUtensorMap mk, mv;
    const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * a.block_size;
    if (!make_maps(k_cache, v_cache, rows, D, a.block_size, &mk, &mv)) return PKV_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return PKV_ERR_CUDA;
    const int grid = std::min(sms, kMaxCtas);
    // every CTA resident at once: the in-kernel merge waits on other CTAs
    static std::atomic<int> mode{-1};
    return launch_resident(mode, kern, dim3((unsigned)grid), dim3(kThreads), smem, st, mk, mv, a);
}

static pkv_status run(Args a, int D, bool paired, int total_units, const void *k_cache, const void *v_cache,
                      cudaStream_t st) {
    for (int u0 = 0; u0 < total_units; u0 += kMaxUnits) {
        a.unit0 = u0;
        a.num_units = std::min(kMaxUnits, total_units - u0);
        a.tag = next_call_tag();
        const pkv_status rc = paired ? (D == 128 ? launch<128, true>(a, k_cache, v_cache, st)
                                                 : launch<64, true>(a, k_cache, v_cache, st))
                                     : (D == 128 ? launch<128, false>(a, k_cache, v_cache, st)
                                                 : launch<64, false>(a, k_cache, v_cache, st));
        if (rc != PKV_OK) return rc;
    }
    return PKV_OK;
}

}  // namespace rows

// The store of each sequence's new token at position seq_lens[s] - 1 (defined
// with the decode kernels).
pkv_status append_new_tokens(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int num_kv_heads,
                             int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, int max_seq_len,
                             int dtype, cudaStream_t st);

}  // namespace pkv

using namespace pkv;

// Diagnostics of the rows kernel's split (host only), for host-side tests.
PKV_API int pkv_rows_context_tiles(int tiles) { return tiles < 0 ? -1 : rows::laid_out(tiles); }

PKV_API int64_t pkv_rows_split_parts(int64_t total_tiles, int64_t ctas) {
    if (total_tiles < 0 || ctas < 1) return -1;
    return total_tiles == 0 ? 0 : rows::split_parts(total_tiles, ctas);
}

PKV_API size_t paged_attention_grouped_workspace_size(int num_seqs, int num_heads, int head_dim, int max_seq_len) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    return rows::ws_layout(head_dim, rows::kRows).total;
}

PKV_API size_t paged_attention_multi_token_workspace_size(int num_q_tokens, int num_heads, int head_dim,
                                                          int max_seq_len) {
    if (num_q_tokens <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    return rows::ws_layout(head_dim, 2 * rows::kRows).total;  // room for paired contexts
}

static bool fill_common(rows::Args &a, void *out, const void *q, const int32_t *block_tables, const int32_t *seq_lens,
                        int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                        int num_blocks, int max_seq_len, float scale, void *workspace, size_t workspace_bytes,
                        int slot_rows) {
    const rows::WsLayout lay = rows::ws_layout(head_dim, slot_rows);
    if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return false;
    a.out = out;
    a.q = q;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_heads / num_kv_heads;
    a.block_size = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.err = device_error_word();
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.part_o = reinterpret_cast<float *>(ws + lay.o_off);
    a.part_ml = reinterpret_cast<float *>(ws + lay.ml_off);
    a.flags = reinterpret_cast<unsigned long long *>(ws + lay.flags_off);
    a.per_ctx = slot_rows / a.group;
    return true;
}

PKV_API pkv_status paged_attention_decode_grouped(
    void *out, const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
    const int32_t *block_tables, const int32_t *seq_lens, const int32_t *group_offsets,
    const int32_t *prefix_lens, int num_groups, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int max_blocks_per_seq, int num_blocks, int max_seq_len, float scale, void *workspace,
    size_t workspace_bytes, int dtype, void *stream) {
    if (num_seqs < 0 || num_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        max_seq_len < 0 || !std::isfinite(scale) || num_groups < 1)
        return PKV_ERR_INVALID;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
    if (dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_seq_len == 0) return PKV_OK;
    if (num_groups > num_seqs) return PKV_ERR_INVALID;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !group_offsets || !prefix_lens)
        return PKV_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID;
    if (((int64_t)num_blocks + 1) * num_kv_heads * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PKV_ERR_INVALID;
    // tile counts of a launch's groups are summed in 32-bit integers
    if ((int64_t)num_seqs * num_kv_heads * ((max_seq_len + rows::kTok - 1) / rows::kTok + 1 + rows::kPieceTiles) >
        INT32_MAX / 2)
        return PKV_ERR_UNSUPPORTED;
    rows::Args a{};
    if (!fill_common(a, out, q, block_tables, seq_lens, num_heads, num_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_seq_len, scale, workspace, workspace_bytes, rows::kRows))
        return PKV_ERR_INVALID;
    a.mode = rows::kGrouped;
    a.group_offsets = group_offsets;
    a.prefix_lens = prefix_lens;
    a.num_seqs = num_seqs;
    a.num_groups = num_groups;
    a.appended = k_new ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (k_new) {
        // each member's new token goes to its slot first; the attention reads it from there
        const pkv_status rc = append_new_tokens(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                                num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                                                max_seq_len, PKV_BF16, st);
        if (rc != PKV_OK) return rc;
    }
    return rows::run(a, head_dim, false, num_groups, k_cache, v_cache, st);
}

PKV_API pkv_status paged_attention_multi_token(void *out, const void *q, const void *k_cache, const void *v_cache,
                                               const int32_t *block_tables, const int32_t *seq_lens,
                                               const int32_t *q_starts, int num_seqs, int num_q_tokens,
                                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                                               int max_blocks_per_seq, int num_blocks, int max_q_len,
                                               int max_seq_len, float scale, void *workspace,
                                               size_t workspace_bytes, void *stream) {
    if (num_seqs < 0 || num_q_tokens < 0 || num_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 ||
        num_blocks < 1 || max_seq_len < 0 || max_q_len < 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_q_tokens == 0) return PKV_OK;
    if (max_q_len < 1 || max_seq_len < 1) return PKV_ERR_INVALID;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_starts) return PKV_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID;
    if (((int64_t)num_blocks + 1) * num_kv_heads * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PKV_ERR_INVALID;
    // tiles of a launch's sequences (every query block of every KV head) in 32-bit integers
    const int64_t per_seq = ((int64_t)max_q_len * (num_heads / num_kv_heads) + rows::kRows - 1) / rows::kRows *
                            ((max_seq_len + rows::kTok - 1) / rows::kTok + rows::kPieceTiles);
    if (std::min<int64_t>(num_seqs, rows::kMaxUnits) * num_kv_heads * per_seq > INT32_MAX / 2)
        return PKV_ERR_UNSUPPORTED;
    // Paired contexts (two 128-row query blocks sharing every tile, one per
    // softmax group) when a sequence may have more than one block of queries
    const bool paired = (int64_t)max_q_len * (num_heads / num_kv_heads) > rows::kRows;
    rows::Args a{};
    if (!fill_common(a, out, q, block_tables, seq_lens, num_heads, num_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_seq_len, scale, workspace, workspace_bytes,
                     paired ? 2 * rows::kRows : rows::kRows))
        return PKV_ERR_INVALID;
    a.mode = rows::kMulti;
    a.q_starts = q_starts;
    a.num_q_tokens = num_q_tokens;
    a.max_q_len = max_q_len;
    return rows::run(a, head_dim, paired, num_seqs, k_cache, v_cache, static_cast<cudaStream_t>(stream));
}

/*
 * pkv.h -- C ABI of the paged KV-cache library (GB300, sm_103a).
 *
 * The method ("PagedAttention (vLLM) -- Virtual memory cho AI", sections
 * "Co che Block Table", "Copy-on-Write cho Beam Search" and "Tai sao no hoat
 * dong"): the KV cache is cut into fixed-size blocks (typically 16 tokens)
 * that sit anywhere in a physical pool; each sequence owns a block table from
 * logical block i (tokens iB .. iB+B-1) to a physical block; blocks are handed
 * out only when a token needs one; branches of beam search share prefix blocks
 * and copy a block only when they diverge inside it; the attention kernel
 * receives the block table and gathers K/V from the scattered blocks.
 *
 * Conventions for every call below
 *   - Pointers marked "device" are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or retains device memory.  Pointers
 *     marked "host" are ordinary host memory, only read during the call.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Device work is enqueued on it; no call synchronises the device, except
 *     pkv_read_device_errors, which waits for the stream.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the previous kernel on the stream finishes if that kernel
 *     triggers its dependents early (griddepcontrol.launch_dependents), and
 *     waits for it before touching its results.  The decode kernels read their
 *     inputs (queries, block tables, lengths) before that wait, so a kernel of
 *     the caller that triggers early must not write those inputs after its
 *     trigger.  Kernels that do not trigger early (the usual case) are waited
 *     for in full, as without programmatic launch.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns PKV_ERR_INVALID (or PKV_ERR_UNSUPPORTED for a valid but
 *     unsupported shape) and enqueues nothing.  A failed launch returns
 *     PKV_ERR_CUDA.  No call raises, exits, traps or asserts on the device.
 *   - Index data that lives on the device (slot mappings, block tables,
 *     sequence lengths, copy pairs) cannot be checked before launch.  Kernels
 *     check every such index before using it: an out-of-range value is never
 *     dereferenced, the affected token, block or pair is skipped, and a bit is
 *     set in a device-side error word read by pkv_read_device_errors.
 *
 * KV cache layout (one K and one V tensor per layer):
 *   [num_blocks][num_kv_heads][block_size][head_dim], row-major, element type
 *   dtype.  One (block, kv head) is a contiguous block_size x head_dim slab
 *   (4 KiB for bf16, block 16, head_dim 128).  Base addresses must be 16-byte
 *   aligned.
 *
 * Supported shapes: head_dim in {64, 128}; block_size in {8, 16, 32};
 *   num_heads a multiple of num_kv_heads with at most 8 query heads per KV head;
 *   dtype PKV_F32 or PKV_BF16.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_EXPORT __attribute__((visibility("default")))
#else
#define PKV_EXPORT
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,     /* bad argument (null pointer, size, sequence id) */
    PKV_ERR_OOM = 2,         /* the allocator has no free block; nothing changed */
    PKV_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    PKV_ERR_UNSUPPORTED = 4, /* valid shape outside the supported set */
    PKV_ERR_TIMEOUT = 5,     /* reserved: a bounded device wait gave up */
    PKV_ERR_TOO_LARGE = 6    /* needs more than the library's built-in scratch */
} pkv_status;

typedef enum pkv_dtype {
    PKV_F32 = 0,  /* float32 in, float32 math, float32 out (no TF32, no bf16) */
    PKV_BF16 = 1  /* bfloat16 storage, float32 accumulation, bf16 output (RNE) */
} pkv_dtype;

/* Bits of the device-side error word (see pkv_read_device_errors). */
#define PKV_DEVERR_BLOCK_ID 1u  /* block-table entry outside [0, num_blocks) */
#define PKV_DEVERR_SEQ_LEN 2u   /* seq_len < 0 or above max_seq_len / table capacity */
#define PKV_DEVERR_SLOT 4u      /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_COPY_PAIR 8u /* block_copy pair outside [0, num_blocks) or src == dst */
#define PKV_DEVERR_TIMEOUT 16u  /* a bounded wait inside a kernel ran out; the rows of a
                                   merge that gave up are NaN.  A piece that arrives after
                                   its merger gave up may leave its ready flag set: zero
                                   the call's workspace before reusing it (a CUDA graph
                                   replays the same flag tag) */
#define PKV_DEVERR_PREFIX 32u   /* grouped decode: bad group offsets or prefix length, or a
                                   member whose blocks differ from the leader's in the prefix */

/* Human-readable name of a status code; never NULL. */
PKV_EXPORT const char *pkv_status_string(int status);

/* Version of this ABI (incremented on any signature change). */
PKV_EXPORT int pkv_abi_version(void);

/*
 * kv_cache_write -- store the K/V of new tokens in their cache slots.
 *
 * Source: "PagedAttention (vLLM) -- Virtual memory cho AI", section "Co che
 * Block Table" (a token lives in physical block table[pos / B] at offset
 * pos % B; blocks are filled as tokens are produced) and "KV cache &
 * PagedAttention -- vi sao chatbot AI ton bo nho" (aiwiki.vn), third
 * paragraph (keys/values are stored for reuse in later steps).
 *
 *   k_new, v_new   device, [num_tokens][num_kv_heads][head_dim], dtype, contiguous
 *   k_cache, v_cache  device, cache layout above, written in place
 *   slot_mapping   device int64 [num_tokens]: slot = physical_block * block_size
 *                  + offset.  slot < 0: the token is skipped (padding).
 *                  slot >= num_blocks * block_size: skipped, PKV_DEVERR_SLOT set.
 * Two tokens mapped to the same slot race (one of them wins).  The copy is
 * bit-exact.  num_tokens == 0 enqueues nothing and returns PKV_OK.
 */
PKV_EXPORT pkv_status kv_cache_write(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, int dtype,
                          void *stream);

/*
 * paged_attention_workspace_size -- bytes of device scratch that
 * paged_attention_decode needs for the same (num_seqs, num_heads, head_dim,
 * max_seq_len, partition_size).  With partition_size > 0 it is 0 when a
 * single pass suffices (every sequence fits one partition).  The scratch holds
 * one partial result per (sequence, query head, piece of context): running
 * max, running sum and an unnormalised output row, all float32; with
 * partition_size == 0 also one 8-byte ready flag per partial.
 */
PKV_EXPORT size_t paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim,
                                      int max_seq_len, int partition_size);

/*
 * paged_attention_decode -- attention of one new query per sequence over its
 * paged KV cache.
 *
 * Source: aiwiki.vn page above, second paragraph (the current query against
 * the keys of the visible positions; the weights combine the values);
 * troisinh page, section "Tai sao no hoat dong", item "Kernel scatter-gather"
 * (the kernel takes the block table and gathers K/V from scattered blocks into
 * on-chip memory before the softmax).  For sequence s, query head h, kv head
 * g = h / (num_heads / num_kv_heads):
 *     out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K[s,t,g,:]) * V[s,t,g,:]
 * over t < seq_lens[s], where token t of sequence s is read from physical block
 * block_tables[s][t / block_size] at offset t % block_size.  The new token must
 * already be in the cache (call kv_cache_write first).  seq_lens[s] == 0 gives
 * an all-zero output row.
 *
 *   out            device [num_seqs][num_heads][head_dim], dtype
 *   q              device [num_seqs][num_heads][head_dim], dtype
 *   k_cache, v_cache  device, cache layout above
 *   block_tables   device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(seq_lens[s] / block_size) are never read
 *   seq_lens       device int32 [num_seqs], each in [0, max_seq_len] and
 *                  <= max_blocks_per_seq * block_size (larger values are
 *                  clamped and flagged with PKV_DEVERR_SEQ_LEN)
 *   scale          multiplies every q.k score (typically 1/sqrt(head_dim))
 *   partition_size a positive multiple of 16: contexts longer than one
 *                  partition are split into partitions of that many tokens,
 *                  each attended independently, and a reduction kernel merges
 *                  the partials (max-rescaled sums), all on `stream`.
 *                  0 = balanced split (bf16): all (sequence, kv head) contexts
 *                  are laid end to end and cut into equal shares of at least
 *                  256 tokens, one per resident warp; a context cut by share
 *                  boundaries is merged inside the attention kernel by the
 *                  warp holding its first tokens, once the other pieces have
 *                  flagged their partials (one kernel per call).  Its warps
 *                  wait on one another, so it is launched cooperatively: a
 *                  grid that cannot be resident at once fails at launch
 *                  (PKV_ERR_CUDA) instead of waiting.  fp32 (or more than
 *                  8192 sequences) uses 512-token partitions and a reduction
 *                  kernel.
 *   workspace      device scratch of at least paged_attention_workspace_size()
 *                  bytes for the same arguments (may be NULL when that is 0),
 *                  256-byte aligned.  Contents need no initialisation (the
 *                  balanced split's ready flags carry a per-call 64-bit tag and
 *                  are cleared after use, so CUDA graph replays of one call
 *                  work too); calls that share a workspace must be ordered on
 *                  the device.
 * Results do not depend on which physical blocks hold the tokens: the order of
 * arithmetic depends only on logical positions, so any permutation of the pool
 * gives bit-identical outputs.
 */
PKV_EXPORT pkv_status paged_attention_decode(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *seq_lens, int num_seqs, int num_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                  float scale, int partition_size, void *workspace,
                                  size_t workspace_bytes, int dtype, void *stream);

/*
 * FP8 (E4M3) KV cache -- kv_cache_write_fp8 and paged_attention_decode_fp8.
 *
 * Source: aiwiki.vn page above, the paragraph on quantisation and offloading:
 * a quantised KV cache stores keys and values in a lower-precision
 * representation to cut the bytes per element, at a conversion cost and a
 * risk of numerical error.  The page fixes no format; this library uses the
 * OCP FP8 E4M3 encoding (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals, no infinities, S.1111.111 = NaN, largest value 448) with
 * one float32 scale per tensor (k_scale for K, v_scale for V):
 *     code(x)  = the E4M3 value nearest to the float32 quotient x / scale
 *                (ties to the even code; beyond +-448, infinities included,
 *                saturate to +-448; NaN gives a NaN code)
 *     value(c) = e4m3(c) * scale
 * FP8 cache layout (one byte per element; base addresses 16-byte aligned):
 *     K: [num_blocks][num_kv_heads][block_size][head_dim]  (as the bf16 cache)
 *     V: [num_blocks][num_kv_heads][head_dim][block_size]  (transposed per
 *        block, so the attention kernel reads runs of consecutive tokens)
 * block_copy copies FP8 blocks unchanged (block_bytes = Hkv * B * D).
 * Supported: head_dim 128, block_size 16 or 32, bf16 new K/V, queries and
 * outputs, at most 8 query heads per KV head, at most 8192 sequences.
 *
 * kv_cache_write_fp8 -- quantise and store the K/V of new tokens.
 *   k_new, v_new   device bf16 [num_tokens][num_kv_heads][head_dim]
 *   k_cache, v_cache  device uint8, FP8 layout above, written in place
 *   slot_mapping   device int64 [num_tokens], as for kv_cache_write
 *   k_scale, v_scale  positive finite float32 scales (else PKV_ERR_INVALID)
 * The codes are bit-exact functions of the inputs (code() above).
 *
 * paged_attention_decode_fp8 -- paged_attention_decode over an FP8 cache:
 *     out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K'[s,t,g,:]) * V'[s,t,g,:]
 * with K' = value(K codes, k_scale), V' = value(V codes, v_scale), g the KV
 * head of h, and the same block-table lookup, length rules, zero rows for
 * empty contexts and device error bits as paged_attention_decode.  q and out
 * are bf16 [num_seqs][num_heads][head_dim].  Always the balanced split: the
 * workspace is paged_attention_workspace_size(num_seqs, num_heads, head_dim,
 * max_seq_len, 0) bytes, 256-byte aligned (may be NULL when max_seq_len is 0).
 * Results do not depend on which physical blocks hold the tokens.
 */
PKV_EXPORT pkv_status kv_cache_write_fp8(const void *k_new, const void *v_new, void *k_cache,
                                         void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int num_blocks, float k_scale, float v_scale, void *stream);

/*
 * paged_attention_decode_append_fp8 -- one FP8 decode step in one call:
 * equivalent to kv_cache_write_fp8 of k_new[s] / v_new[s] (bf16
 * [num_seqs][num_kv_heads][head_dim]) at position seq_lens[s] - 1 of sequence
 * s (the slot its block table gives for that position), followed by
 * paged_attention_decode_fp8.  The codes are stored inside the attention
 * kernel, before any load of their tile.  Every seq_lens[s] must be >= 1 (a
 * sequence of length 0 stores nothing and gets a zero row); a block-table
 * entry outside the pool skips the store and is flagged as in the decode.
 */
PKV_EXPORT pkv_status paged_attention_decode_append_fp8(void *out, const void *q, const void *k_new,
                                                        const void *v_new, void *k_cache, void *v_cache,
                                                        const int32_t *block_tables, const int32_t *seq_lens,
                                                        int num_seqs, int num_heads, int num_kv_heads,
                                                        int head_dim, int block_size, int max_blocks_per_seq,
                                                        int num_blocks, int max_seq_len, float scale,
                                                        float k_scale, float v_scale, void *workspace,
                                                        size_t workspace_bytes, void *stream);

PKV_EXPORT pkv_status paged_attention_decode_fp8(void *out, const void *q, const void *k_cache,
                                                 const void *v_cache, const int32_t *block_tables,
                                                 const int32_t *seq_lens, int num_seqs, int num_heads,
                                                 int num_kv_heads, int head_dim, int block_size,
                                                 int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                                 float scale, float k_scale, float v_scale,
                                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attention_multi_token -- attention of several new tokens per sequence
 * (chunked prefill, verification of drafted tokens) over the paged cache.
 *
 * Source: "vLLM PagedAttention: Buoc dot pha ve thong luong suy luan LLM"
 * (vi.news.hada.io), the advanced features built on PagedAttention (chunked
 * prefill; speculative decoding with drafted tokens), with the causal reading
 * of the aiwiki.vn page's attention (a position attends to the positions it
 * may see).  Sequence s carries Q_s = q_starts[s+1] - q_starts[s] query
 * tokens, the last Q_s positions of its context of L_s = seq_lens[s] tokens
 * (their K/V already written, e.g. by kv_cache_write); query i sits at
 * position p = L_s - Q_s + i and
 *     out[q_starts[s]+i, h, :] = sum_{t <= p} softmax_t(scale * q[q_starts[s]+i, h, :] . K[s,t,g,:]) V[s,t,g,:]
 * with g the KV head of h.  Q_s = 1 is the decode step.
 *
 *   q, out         device bf16 [num_q_tokens][num_heads][head_dim]
 *   k_cache, v_cache, block_tables, seq_lens  as for paged_attention_decode (bf16)
 *   q_starts       device int32 [num_seqs + 1], q_starts[0] = 0, non-decreasing,
 *                  q_starts[num_seqs] = num_q_tokens; inconsistent entries are
 *                  flagged (PKV_DEVERR_SEQ_LEN) and the sequence is skipped
 *   max_q_len      >= every Q_s (queries past it are not attended, their rows
 *                  are left unwritten, and PKV_DEVERR_SEQ_LEN is set); a
 *                  sequence with Q_s > L_s is flagged too and its queries that
 *                  see no token get zero rows
 *   workspace      paged_attention_multi_token_workspace_size() bytes,
 *                  256-byte aligned (about 34 MB for head_dim 128, whatever
 *                  the number of tokens: one partial slot of 256 rows per
 *                  CTA).  Contents need no initialisation; calls that share a
 *                  workspace must be ordered on the device.
 * The attention runs on the tensor cores (tcgen05): per KV head, the query
 * heads of up to 128 / (num_heads / num_kv_heads) queries form the 128 rows
 * of one query block, attended against 64-token tiles of K and V (Q K^T and
 * P V with fp32 accumulators in tensor memory, the causal limit applied per
 * row).  When max_q_len spans more than one block (a prefill chunk), two
 * consecutive blocks form one context: each tile is read once for both.
 * All contexts' tiles are cut into equal shares, one per SM; a context cut by
 * share boundaries is merged inside the kernel.  The CTAs wait on one another,
 * so the kernel is launched cooperatively: a grid that cannot be resident at
 * once fails at launch (PKV_ERR_CUDA) instead of waiting.
 * Supported: bf16; head_dim 64 or 128; block_size 8, 16 or 32; at most 8
 * query heads per KV head.  Results do not depend on which physical blocks
 * hold the tokens.
 */
PKV_EXPORT size_t paged_attention_multi_token_workspace_size(int num_q_tokens, int num_heads, int head_dim,
                                                             int max_seq_len);
PKV_EXPORT pkv_status paged_attention_multi_token(void *out, const void *q, const void *k_cache,
                                                  const void *v_cache, const int32_t *block_tables,
                                                  const int32_t *seq_lens, const int32_t *q_starts,
                                                  int num_seqs, int num_q_tokens, int num_heads,
                                                  int num_kv_heads, int head_dim, int block_size,
                                                  int max_blocks_per_seq, int num_blocks, int max_q_len,
                                                  int max_seq_len, float scale, void *workspace,
                                                  size_t workspace_bytes, void *stream);

/*
 * block_copy -- copy whole physical blocks, in every layer, for K and V.
 *
 * Source: troisinh page, section "Copy-on-Write cho Beam Search": sequences
 * share the physical blocks of a common prefix and a block is split (copied)
 * only when their tokens start to differ.  block_allocator_append_slot reports
 * the (src, dst) pair to copy.
 *
 *   k_caches, v_caches  host arrays of num_layers device pointers (one cache
 *                       tensor per layer, cache layout above)
 *   block_pairs    device int64 [num_pairs][2] = (src, dst) physical block ids.
 *                  A pair outside [0, num_blocks), or with src == dst, is
 *                  skipped and flags PKV_DEVERR_COPY_PAIR.  A dst must not be
 *                  the src or dst of another pair in the same call.
 *   block_bytes    bytes of one physical block of one layer's K (or V) tensor:
 *                  num_kv_heads * block_size * head_dim * element size; a
 *                  positive multiple of 16.
 * The copy is bit-exact.  num_pairs == 0 or num_layers == 0 returns PKV_OK.
 */
PKV_EXPORT pkv_status block_copy(void *const *k_caches, void *const *v_caches, int num_layers,
                      const int64_t *block_pairs, int num_pairs, int num_blocks,
                      size_t block_bytes, void *stream);

/*
 * paged_attention_decode_append -- one decode step in one call: store each
 * sequence's new token, then attend.
 *
 * Source: the same passages as kv_cache_write and paged_attention_decode; the
 * new token is produced, stored in its block (troisinh page, "Co che Block
 * Table") and attended together with the cached ones (aiwiki.vn page,
 * second and third paragraphs).
 *
 * Equivalent to kv_cache_write of k_new[s] / v_new[s] at position
 * seq_lens[s] - 1 of sequence s (the slot its block table gives for that
 * position; sequences with seq_lens[s] == 0 store nothing) followed by
 * paged_attention_decode with the same arguments.
 *   k_new, v_new   device [num_seqs][num_kv_heads][head_dim], dtype, 16-byte aligned
 *   k_cache, v_cache  written (the new token) and read
 * With partition_size == 0 and bf16 the store happens inside the attention
 * kernel, by the warp that attends the tile holding that position, just
 * before it loads the tile; otherwise a store kernel runs first.  The result
 * is the same either way.
 */
PKV_EXPORT pkv_status paged_attention_decode_append(void *out, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache,
                                  const int32_t *block_tables, const int32_t *seq_lens,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_blocks_per_seq, int num_blocks,
                                  int max_seq_len, float scale, int partition_size,
                                  void *workspace, size_t workspace_bytes, int dtype, void *stream);

/*
 * paged_attention_decode_grouped -- decode for batches whose sequences share
 * prefix blocks (beam search, parallel sampling), each shared block read once.
 *
 * Source: troisinh page, section "Copy-on-Write cho Beam Search" (branches
 * of beam search / parallel sampling share the physical blocks of their common
 * prefix) and aiwiki.vn page, paging paragraphs (blocks shared between
 * branches instead of duplicated).  Same result as paged_attention_decode
 * (or, with k_new/v_new, as paged_attention_decode_append).
 *
 *   group_offsets  device int32 [num_groups + 1]: group g is sequences
 *                  group_offsets[g] .. group_offsets[g+1]-1; 0 = first entry,
 *                  num_seqs = last; every sequence belongs to one group
 *   prefix_lens    device int32 [num_groups]: tokens at the start of every
 *                  member's context stored in the same physical blocks as the
 *                  group's first member (its block-table entries are equal).
 *                  A multiple of max(16, block_size); it is cut to the shortest
 *                  member (minus one token when appending).  0 = no sharing.
 *   k_new, v_new   device [num_seqs][num_kv_heads][head_dim] or both NULL: as
 *                  in paged_attention_decode_append
 *   workspace      at least paged_attention_grouped_workspace_size() bytes
 *                  (as for paged_attention_multi_token), 256-byte aligned, no
 *                  initialisation needed
 * Per KV head, a group (up to 128 / (num_heads / num_kv_heads) members at a
 * time) is one context of members x query heads rows on the tensor cores
 * (tcgen05, fp32 accumulators in tensor memory): the shared part, cut to whole
 * 64-token tiles, is read once and seen by every row; then each member's own
 * tiles, seen by that member's rows only.  One context gives every member's
 * final result; a context cut by the kernel's equal per-SM shares is merged
 * inside the kernel (cooperative launch, as for paged_attention_multi_token).
 * With k_new/v_new a small kernel stores the new tokens first.  A launch
 * scans at most 1024 groups; more groups take several launches.
 * A bad group description (offsets out of order or not covering 0..num_seqs,
 * a prefix length that is not a multiple of max(16, block_size)) flags
 * PKV_DEVERR_PREFIX.  A member whose prefix blocks differ from the first
 * member's also flags PKV_DEVERR_PREFIX; that member's result is then
 * unspecified (finite).  bf16 only, num_seqs <= 8192 (else
 * PKV_ERR_UNSUPPORTED).
 */
PKV_EXPORT size_t paged_attention_grouped_workspace_size(int num_seqs, int num_heads, int head_dim,
                                              int max_seq_len);
PKV_EXPORT pkv_status paged_attention_decode_grouped(void *out, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache,
                                  const int32_t *block_tables, const int32_t *seq_lens,
                                  const int32_t *group_offsets, const int32_t *prefix_lens,
                                  int num_groups, int num_seqs, int num_heads, int num_kv_heads,
                                  int head_dim, int block_size, int max_blocks_per_seq,
                                  int num_blocks, int max_seq_len, float scale, void *workspace,
                                  size_t workspace_bytes, int dtype, void *stream);

/*
 * paged_attention_decode_noalloc -- paged_attention_decode for callers that
 * cannot allocate device memory.  No passage of the pages has a counterpart:
 * this entry point exists for the caller, not for the method.
 *
 * Some callers have no way to hand the library a scratch buffer: code that
 * runs where cudaMalloc is forbidden or unavailable (inside a custom memory
 * pool that owns all device memory, a plugin host that only passes tensors
 * in and out, a runtime that must not allocate on its decode path).  This
 * variant takes the same inputs and outputs as paged_attention_decode minus
 * the workspace; the split-K partials live instead in a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library, which every
 * GPU that loads the library keeps until the process exits.
 *
 *   partition_size 0 = 512-token partitions; otherwise as for
 *                  paged_attention_decode.  The split always uses fixed
 *                  partitions plus the merge kernel.
 *   Returns PKV_ERR_TOO_LARGE, with nothing enqueued, when the partials for
 *   (num_seqs, num_heads, head_dim, max_seq_len, partition_size) need more
 *   than PKV_NOALLOC_SCRATCH_BYTES (see paged_attention_workspace_size).
 *   Every other argument and error behaves as in paged_attention_decode.
 *
 * The first call on a device looks up that device's address of the array
 * (cudaGetSymbolAddress) with the device current; make that first call before
 * any stream capture.  The address is cached per device together with the
 * CUDA context it was taken in; a call from another context (a context the
 * caller created, or a primary context created anew after cudaDeviceReset)
 * looks it up again, so make such a call outside stream capture too.  Every call on a device shares the one array and leaves
 * its partials there: nothing in it has to start at zero (each call writes
 * every partial it later reads), but calls whose work overlaps on the GPU --
 * two streams, or two host threads -- race on it and must be serialised by
 * the caller.  The call itself allocates nothing.
 */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
PKV_EXPORT pkv_status paged_attention_decode_noalloc(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *seq_lens, int num_seqs, int num_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                  float scale, int partition_size, int dtype, void *stream);

/*
 * pkv_read_device_errors -- wait for `stream`, then return in *flags_out the
 * PKV_DEVERR_* bits set by kernels of this library on the current device since
 * the last clear; clear != 0 resets the word afterwards.
 */
PKV_EXPORT pkv_status pkv_read_device_errors(uint32_t *flags_out, int clear, void *stream);

/*
 * pkv_bounded_wait_check -- failure-detection check of the two bounded waits
 * the attention kernels use, so that a test can make each run out without a
 * GPU fault.  One warp runs, on `stream`:
 *   1. the merger's flag wait: polls the n_flags 8-byte words at `flags`
 *      (device memory, read only; skipped when n_flags == 0) until all hold
 *      `tag`, at most `polls` rounds;
 *   2. the mbarrier wait: waits for phase 0 of a fresh shared-memory mbarrier
 *      of one arrival, at most `polls` polls; the warp arrives first only when
 *      arrive != 0.
 * A wait that runs out sets PKV_DEVERR_TIMEOUT in the device error word
 * (pkv_read_device_errors) and the kernel goes on and returns; the context
 * stays usable.  The attention kernels run the same two waits with a limit of
 * 2^22 polls.  PKV_ERR_INVALID for n_flags < 0, a null `flags` with
 * n_flags > 0, or polls == 0.
 */
PKV_EXPORT pkv_status pkv_bounded_wait_check(const uint64_t *flags, int n_flags, uint64_t tag, int arrive,
                                             uint32_t polls, void *stream);

/* ------------------------------------------------------------------------
 * Host block allocator.
 *
 * Source: troisinh page, sections "Co che Block Table" (fixed blocks, a
 * per-sequence table, a block only when a token needs it; 100 tokens -> 7
 * blocks of 16; freed blocks reused at once without defragmentation) and
 * "Copy-on-Write cho Beam Search"; aiwiki.vn page, paging paragraphs (blocks
 * added on demand, waste concentrated in each sequence's last block, prefix
 * blocks shared between branches).
 *
 * Policy: free blocks form a LIFO stack that first hands out 0, 1, 2, ...; a
 * freed sequence pushes its blocks in table order.  Every operation is
 * all-or-nothing: PKV_ERR_OOM / PKV_ERR_INVALID leave the state unchanged.
 * A handle is not thread-safe; it owns host memory only.
 * ---------------------------------------------------------------------- */
typedef struct pkv_allocator pkv_allocator;

/* NULL on bad arguments (num_blocks < 1, block_size < 1) or out of memory. */
PKV_EXPORT pkv_allocator *block_allocator_create(int num_blocks, int block_size);
PKV_EXPORT void block_allocator_destroy(pkv_allocator *a);

/* New sequence `seq` holding num_tokens tokens (a prompt): ceil(n/B) blocks. */
PKV_EXPORT pkv_status block_allocator_add_seq(pkv_allocator *a, int64_t seq, int64_t num_tokens);

/* Room for one more token of `seq`.  *slot_out receives its slot.  If the last
 * block is full (or absent) a fresh block is taken.  If the last block is
 * partially filled and shared (reference count > 1), a fresh block replaces it
 * in this sequence's table, the shared block loses one reference and
 * (*cow_src_out, *cow_dst_out) name the pair to copy with block_copy before the
 * token is written; otherwise both are -1.  Output pointers may be NULL. */
PKV_EXPORT pkv_status block_allocator_append_slot(pkv_allocator *a, int64_t seq, int64_t *slot_out,
                                       int32_t *cow_src_out, int32_t *cow_dst_out);

/* One decode step's worth of append_slot for n distinct sequences, in order.
 * slots_out: host int64 [n]; cow_pairs_out: host int64 [n][2] receives the
 * (src, dst) pairs to copy, *n_cow_out of them (ready for block_copy).  All or
 * nothing: PKV_ERR_OOM if the free stack cannot serve every sequence,
 * PKV_ERR_INVALID for an unknown or repeated id; then nothing changes. */
PKV_EXPORT pkv_status block_allocator_append_slots(pkv_allocator *a, const int64_t *seqs, int n,
                                        int64_t *slots_out, int64_t *cow_pairs_out,
                                        int *n_cow_out);

/* append_slots plus the incremental update of the caller's dense block
 * tables, for a serving loop that keeps them between steps: tables is host
 * int32 [n][cap] (row i belongs to seqs[i], as block_allocator_block_tables
 * wrote it) and seq_lens host int32 [n].  Per sequence, only the entry of the
 * block holding the new token is written (the fresh block, the CoW
 * destination, or the same id again) and seq_lens[i] becomes the new token
 * count; nothing else in the row changes, so a row that block_tables wrote
 * before stays equal to what it would write now.  PKV_ERR_INVALID (nothing
 * changed) also when a new token's block index would be >= cap. */
PKV_EXPORT pkv_status block_allocator_append_step(pkv_allocator *a, const int64_t *seqs, int n,
                                                  int32_t *tables, int cap, int32_t *seq_lens,
                                                  int64_t *slots_out, int64_t *cow_pairs_out, int *n_cow_out);

/* `child` starts as a copy of `parent` that shares every block (refcount + 1). */
PKV_EXPORT pkv_status block_allocator_fork(pkv_allocator *a, int64_t parent, int64_t child);

/* Drop `seq`; blocks whose reference count reaches 0 return to the free stack. */
PKV_EXPORT pkv_status block_allocator_free_seq(pkv_allocator *a, int64_t seq);

/* Copy the block table of `seq` into out[0 .. cap); *n_out = its length.
 * PKV_ERR_INVALID if the table is longer than cap (nothing written). */
PKV_EXPORT pkv_status block_allocator_block_table(const pkv_allocator *a, int64_t seq, int32_t *out,
                                       int cap, int *n_out);

/* Dense tables for n sequences: out is host int32 [n][cap], rows padded with
 * `pad`; seq_lens_out (host int32 [n], may be NULL) receives token counts. */
PKV_EXPORT pkv_status block_allocator_block_tables(const pkv_allocator *a, const int64_t *seqs, int n,
                                        int32_t *out, int cap, int32_t pad,
                                        int32_t *seq_lens_out);

/* Groups for paged_attention_decode_grouped: the given sequences, in order,
 * are cut into runs whose block tables start with the same physical blocks
 * (beams forked from one prompt).  group_offsets_out: host int32 [n + 1];
 * prefix_lens_out: host int32 [n] (tokens in the shared full blocks, rounded
 * down to a multiple of max(16, block_size); 0 for a single sequence);
 * *num_groups_out = number of runs. */
PKV_EXPORT pkv_status block_allocator_prefix_groups(const pkv_allocator *a, const int64_t *seqs, int n,
                                         int32_t *group_offsets_out, int32_t *prefix_lens_out,
                                         int *num_groups_out);

/*
 * block_allocator_extend -- room for `count` more tokens of `seq` at once (a
 * prefill chunk, drafted tokens): writes slots_out[count] (host int64) for
 * positions len .. len+count-1, exactly as `count` calls of
 * block_allocator_append_slot would, but all or nothing (PKV_ERR_OOM changes
 * nothing).  At most one copy-on-write pair can arise (a shared, partially
 * filled last block); it is reported in *cow_src_out / *cow_dst_out (-1 if
 * none) and must be copied (block_copy) before the new tokens are written.
 */
PKV_EXPORT pkv_status block_allocator_extend(pkv_allocator *a, int64_t seq, int64_t count, int64_t *slots_out,
                                             int32_t *cow_src_out, int32_t *cow_dst_out);

/*
 * block_allocator_truncate -- keep the first num_tokens tokens of `seq`
 * (0 <= num_tokens <= its length, else PKV_ERR_INVALID), e.g. to roll back
 * drafted tokens that verification rejected ("vLLM PagedAttention: Buoc dot
 * pha ...", speculative decoding).  Blocks wholly past the new end lose this
 * sequence's reference (freed, or parked as evictable if registered in the
 * prefix cache); a shared last block is copied on the next append as usual; a
 * registered block that becomes the partially filled last block of its only
 * holder is unregistered (the next append writes into it).  Device data is
 * not touched.
 */
PKV_EXPORT pkv_status block_allocator_truncate(pkv_allocator *a, int64_t seq, int64_t num_tokens);

/*
 * block_allocator_add_seq_cached -- block_allocator_add_seq for a prompt
 * whose token ids are known, reusing the K/V of earlier prompts that start
 * with the same tokens (prefix caching).
 *
 * Source: "vLLM PagedAttention: Buoc dot pha ve thong luong suy luan LLM",
 * list of advanced features, "Prefix caching" (the KV cache of a prompt
 * prefix shared by several requests is reused instead of recomputed); and
 * "PagedAttention (vLLM) -- Virtual memory cho AI", related posts ("Prefix
 * Caching" for system prompts reused many times).  The pages give no
 * mechanism; this one: every full block of a prompt added here is registered
 * under a 64-bit hash of its whole token prefix (FNV-1a over the parent's
 * hash and the block's token ids).  A later prompt whose leading full blocks
 * have registered prefixes with equal token ids (compared exactly) shares
 * those blocks (reference count + 1) instead of taking new ones; the first
 * block that does not match, and everything after it, is allocated as usual
 * (a partially filled last block is never shared this way).
 *
 *   tokens              host int32 [num_tokens]: the prompt's token ids
 *   cached_tokens_out   tokens at the start of the prompt whose K and V are
 *                       already in the pool (a multiple of block_size); the
 *                       caller writes K/V for positions cached_tokens_out ..
 *                       num_tokens - 1 only.  A registered block holds valid
 *                       K/V once the prompt that registered it has been
 *                       written.
 * A registered block whose last holder is freed stays registered and is kept
 * (evictable) until the free stack runs dry: then the one released longest
 * ago is handed out and unregistered (a freed prompt's blocks are released
 * last block first, so a prefix loses its tail before its head).
 * block_allocator_num_free counts free and evictable blocks.  All-or-nothing:
 * PKV_ERR_OOM and PKV_ERR_INVALID change nothing.
 */
PKV_EXPORT pkv_status block_allocator_add_seq_cached(pkv_allocator *a, int64_t seq, const int32_t *tokens,
                                          int64_t num_tokens, int64_t *cached_tokens_out);

/* Prefix cache counters: full blocks found (hits) and not found (misses) by
 * block_allocator_add_seq_cached so far, blocks registered now, and how many
 * of those are evictable (no holder).  Any output may be NULL. */
PKV_EXPORT pkv_status block_allocator_cache_stats(const pkv_allocator *a, int64_t *hits, int64_t *misses,
                                       int *cached_blocks, int *evictable_blocks);

/* Empty the prefix cache: evictable blocks return to the free stack (released
 * longest ago first); blocks still held keep their holders but are no longer
 * found by block_allocator_add_seq_cached. */
PKV_EXPORT pkv_status block_allocator_cache_clear(pkv_allocator *a);

/* Slots of token positions start .. start+count-1 of `seq` (all must exist). */
PKV_EXPORT pkv_status block_allocator_slots(const pkv_allocator *a, int64_t seq, int64_t start,
                                 int64_t count, int64_t *out);

/* Token count of `seq`, or -1 if it does not exist. */
PKV_EXPORT int64_t block_allocator_num_tokens(const pkv_allocator *a, int64_t seq);
PKV_EXPORT int block_allocator_num_free(const pkv_allocator *a);
/* Reference count of a physical block, -1 if the id is out of range. */
PKV_EXPORT int block_allocator_refcount(const pkv_allocator *a, int32_t block);

/* Occupied slots and allocated slots over all live sequences, each physical
 * block counted once however many sequences share it.  Waste fraction =
 * 1 - used / allocated. */
PKV_EXPORT pkv_status block_allocator_waste(const pkv_allocator *a, int64_t *used_tokens,
                                 int64_t *allocated_slots);

/*
 * Diagnostics of the balanced split (host only, no device work).  They expose
 * the arithmetic the balanced decode kernel runs, so that host-side tests can
 * check the invariants its in-kernel merge relies on against the kernel's own
 * code rather than a copy.  Not part of the method: the pages say nothing
 * about how a kernel divides its work.
 *
 * pkv_balanced_segment_tiles: the tiles a (sequence, kv head) segment of
 *   `tiles` real tiles takes in the kernel's tile list: the real ones after
 *   a fixed number of empty lead tiles (a scheduling charge for the piece's
 *   fixed costs and the merge), 0 for an empty segment; -1 if tiles < 0.
 *   Shares, slots and ownership below count these laid-out tiles.
 * pkv_balanced_slots: partial slots per (sequence, query head) that the
 *   workspace of a balanced call holds for contexts of up to max_seq_len
 *   tokens (ceil(max_seq_len / 256) + 1); -1 if max_seq_len < 0.
 * pkv_balanced_split_parts: number of equal shares the kernel cuts
 *   total_tiles tiles into, when the longest (sequence, kv head) segment has
 *   max_segment_tiles tiles and at most `warps` warps take shares; 0 when
 *   there is no tile, -1 for a negative argument or warps < 1.
 * pkv_balanced_share_owner: the share (0 .. parts-1) holding tile `tile` of
 *   the total_tiles tiles cut into `parts` shares [floor(c T / parts),
 *   floor((c + 1) T / parts)); -1 for arguments out of range.
 */
PKV_EXPORT int pkv_balanced_segment_tiles(int tiles);

/*
 * Diagnostics of the rows kernel's split (grouped decode, multi-token
 * attention; host only, no device work), for host-side tests:
 * pkv_rows_context_tiles: the tiles a context of `tiles` real 64-key tiles
 *   takes in the kernel's tile list (its real tiles after a fixed number of
 *   virtual ones, a scheduling charge), 0 for none; -1 if tiles < 0.
 * pkv_rows_split_parts: the shares (one per CTA) that total_tiles laid-out
 *   tiles are cut into with `ctas` CTAs, share c = [floor(c T / parts),
 *   floor((c + 1) T / parts)); 0 for no tile, -1 for bad arguments.
 */
PKV_EXPORT int pkv_rows_context_tiles(int tiles);
PKV_EXPORT int64_t pkv_rows_split_parts(int64_t total_tiles, int64_t ctas);
PKV_EXPORT int pkv_balanced_slots(int max_seq_len);
PKV_EXPORT int64_t pkv_balanced_split_parts(int64_t total_tiles, int max_segment_tiles, int max_seq_len,
                                            int64_t warps);
PKV_EXPORT int64_t pkv_balanced_share_owner(int64_t tile, int64_t total_tiles, int64_t parts);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */

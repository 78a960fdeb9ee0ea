// Cache write (slot-mapped scatter of new K/V), copy-on-write block copy, the
// device error word and the status strings.
//
// kv_cache_write: "PagedAttention (vLLM) -- Virtual memory cho AI", section
// "Co che Block Table" -- a token lives in physical block table[pos / B] at
// offset pos % B, and blocks are filled as tokens are produced.
// block_copy: same page, section "Copy-on-Write cho Beam Search" -- a shared
// block is copied when the branches sharing it start to differ.
//
// Both kernels move 16-byte vectors: consecutive threads own consecutive
// 16-byte chunks of a K/V row (or of a whole physical block), so every warp
// reads and writes fully coalesced 512-byte spans.
#include <cmath>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

__device__ unsigned int g_error_word = 0;

unsigned int *device_error_word() {
    static std::mutex mu;
    static unsigned int *ptrs[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned int *>(p);
    }
    return ptrs[dev];
}

// One thread per 16-byte chunk of one (token, kv head) row of K and of V.
__global__ void __launch_bounds__(256)
kv_cache_write_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                      uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                      const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                      int num_kv_heads, int chunks_per_row, int block_size,
                      int64_t num_slots, unsigned int *err) {
    // a dependent decode kernel may start its launch while this one runs; it
    // waits for this grid before reading the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t per_token = (int64_t)num_kv_heads * chunks_per_row;
    const int64_t total = num_tokens * per_token;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;
        const int64_t h = r / chunks_per_row;
        const int64_t c = r - h * chunks_per_row;
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (r == 0) flag_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        k_cache[dst] = k_new[i];
        v_cache[dst] = v_new[i];
    }
}

// FP8 (E4M3) cache write.  One thread per 16 head_dim entries of one (token,
// kv head): the K codes go out as one 16-byte row chunk; the V codes go to
// the transposed V block ([D][block_size] per (block, kv head)), one byte per
// head_dim row.  Codes from quantize16 (pkv_internal.cuh).
__global__ void __launch_bounds__(256)
kv_cache_write_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                          unsigned char *__restrict__ k_cache, unsigned char *__restrict__ v_cache,
                          const int64_t *__restrict__ slot_mapping, int64_t num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int64_t num_slots, float k_scale, float v_scale,
                          unsigned int *err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int chunks = head_dim / 16;
    const int64_t per_token = (int64_t)num_kv_heads * chunks;
    const int64_t total = num_tokens * per_token;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;
        const int64_t h = r / chunks;
        const int c = (int)(r - h * chunks);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (r == 0) flag_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
        const int64_t bh = blk * num_kv_heads + h;
        uint4 kx[2] = {k_new[2 * i], k_new[2 * i + 1]};
        uint4 vx[2] = {v_new[2 * i], v_new[2 * i + 1]};
        uint32_t kw[4], vw[4];
        quantize16(kx, k_scale, kw);
        quantize16(vx, v_scale, vw);
        *reinterpret_cast<uint4 *>(k_cache + (bh * block_size + off) * head_dim + 16 * c) =
            make_uint4(kw[0], kw[1], kw[2], kw[3]);
        unsigned char *vcol = v_cache + (bh * head_dim + 16 * c) * block_size + off;
#pragma unroll
        for (int j = 0; j < 16; ++j) vcol[(int64_t)j * block_size] = (unsigned char)(vw[j >> 2] >> (8 * (j & 3)));
    }
}

constexpr int kMaxCopyLayers = 64;
struct CopyPtrs {
    uint4 *k[kMaxCopyLayers];
    uint4 *v[kMaxCopyLayers];
};

// grid = (pair, layer, K or V); each CTA copies one physical block.
__global__ void __launch_bounds__(256)
block_copy_kernel(CopyPtrs p, const int64_t *__restrict__ pairs, int num_blocks,
                  int64_t vec_per_block, unsigned int *err) {
    const int pair = blockIdx.x;
    const int layer = blockIdx.y;
    const int64_t src = pairs[2 * (int64_t)pair];
    const int64_t dst = pairs[2 * (int64_t)pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst) {
        if (threadIdx.x == 0 && layer == 0 && blockIdx.z == 0) flag_error(err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    uint4 *base = blockIdx.z ? p.v[layer] : p.k[layer];
    const uint4 *s = base + src * vec_per_block;
    uint4 *d = base + dst * vec_per_block;
    for (int64_t i = threadIdx.x; i < vec_per_block; i += blockDim.x) d[i] = s[i];
}

}  // namespace pkv

using namespace pkv;

PKV_API const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID: return "invalid argument";
        case PKV_ERR_OOM: return "out of KV blocks";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PKV_ERR_TIMEOUT: return "device wait timed out";
        case PKV_ERR_TOO_LARGE: return "needs more scratch than the library's built-in array";
        default: return "unknown status";
    }
}

PKV_API int pkv_abi_version(void) { return 1; }

PKV_API pkv_status kv_cache_write(const void *k_new, const void *v_new, void *k_cache,
                                  void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                  int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                  int dtype, void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1)
        return PKV_ERR_INVALID;
    if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID;
    const int elt = dtype == PKV_F32 ? 4 : 2;
    const int chunks = head_dim * elt / 16;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * chunks;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    const unsigned grid = (unsigned)(blocks < 1048576 ? blocks : 1048576);
    kv_cache_write_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, (uint4 *)k_cache, (uint4 *)v_cache,
        slot_mapping, num_tokens, num_kv_heads, chunks, block_size,
        (int64_t)num_blocks * block_size, device_error_word());
    return launch_status();
}

PKV_API pkv_status kv_cache_write_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                      const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks, float k_scale,
                                      float v_scale, void *stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1)
        return PKV_ERR_INVALID;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID;
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * (head_dim / 16);
    const int64_t blocks = (total + 255) / 256;
    const unsigned grid = (unsigned)(blocks < 1048576 ? blocks : 1048576);
    kv_cache_write_fp8_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_new, (const uint4 *)v_new, (unsigned char *)k_cache, (unsigned char *)v_cache,
        slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, (int64_t)num_blocks * block_size,
        k_scale, v_scale, device_error_word());
    return launch_status();
}

PKV_API pkv_status block_copy(void *const *k_caches, void *const *v_caches, int num_layers,
                              const int64_t *block_pairs, int num_pairs, int num_blocks,
                              size_t block_bytes, void *stream) {
    if (num_layers < 0 || num_pairs < 0 || num_blocks < 1) return PKV_ERR_INVALID;
    if (num_layers == 0 || num_pairs == 0) return PKV_OK;
    if (!k_caches || !v_caches || !block_pairs || block_bytes == 0 || block_bytes % 16 != 0)
        return PKV_ERR_INVALID;
    if (num_pairs > 65535 * 1024) return PKV_ERR_INVALID;
    for (int l = 0; l < num_layers; ++l)
        if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
            return PKV_ERR_INVALID;
    unsigned int *err = device_error_word();
    const int64_t vec = (int64_t)(block_bytes / 16);
    for (int l0 = 0; l0 < num_layers; l0 += kMaxCopyLayers) {
        const int nl = num_layers - l0 < kMaxCopyLayers ? num_layers - l0 : kMaxCopyLayers;
        CopyPtrs p{};
        for (int i = 0; i < nl; ++i) {
            p.k[i] = (uint4 *)k_caches[l0 + i];
            p.v[i] = (uint4 *)v_caches[l0 + i];
        }
        dim3 grid((unsigned)num_pairs, (unsigned)nl, 2);
        block_copy_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(p, block_pairs, num_blocks, vec, err);
        if (launch_status() != PKV_OK) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

PKV_API pkv_status pkv_read_device_errors(uint32_t *flags_out, int clear, void *stream) {
    if (!flags_out) return PKV_ERR_INVALID;
    unsigned int *w = device_error_word();
    if (!w) return PKV_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, w, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (clear && cudaMemsetAsync(w, 0, sizeof(unsigned int), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    *flags_out = host;
    return PKV_OK;
}

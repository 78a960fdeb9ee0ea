// Internal helpers shared by the library's CUDA translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <unistd.h>

#include <atomic>
#include <chrono>
#include <mutex>

#include "pkv.h"

#define PKV_API extern "C" __attribute__((visibility("default")))

namespace pkv {

// Device address of the library's error word on the current device (set up
// on first use per device).  nullptr if CUDA is unusable.
unsigned int *device_error_word();

inline pkv_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A 64-bit tag per balanced call, never 0 (the value of a cleared flag): flags
// left by other calls, or never written, hold another value.  The sequence
// starts at a value drawn from the clock, the process and an address, so
// separate processes start far apart.
inline unsigned long long next_call_tag() {
    static std::atomic<unsigned long long> count{0};
    static const unsigned long long base = [] {
        unsigned long long x = (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
        x ^= (unsigned long long)getpid() * 0x9E3779B97F4A7C15ull;
        x ^= (unsigned long long)reinterpret_cast<uintptr_t>(&count);
        x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
        x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
        return x ^ (x >> 31);
    }();
    unsigned long long t;
    do {
        t = base + count.fetch_add(1, std::memory_order_relaxed);
    } while (t == 0);
    return t;
}

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
inline bool make_cache_map(CUtensorMap *map, const void *base, int64_t rows, int D, int boxh) {
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

// Opt a kernel in to the dynamic shared memory it may need (once per device).
template <typename K>
inline bool ensure_smem(K kernel, int bytes, bool (&done)[128]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return false;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

inline int sm_count() {
    static int counts[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream drains; it waits (griddepcontrol.wait)
// before touching memory, so stream order is preserved.
// With `cooperative`, the launch also asks for every CTA of the grid to be
// resident at once (cudaLaunchAttributeCooperative): a grid that cannot be is
// refused at launch (PKV_ERR_CUDA) instead of running in waves.  Kernels whose
// CTAs wait on one another (the in-kernel merges) rely on that.
template <typename... KArgs, typename... Args>
inline pkv_status launch_pdl_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                bool cooperative, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? launch_status() : PKV_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
inline pkv_status launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
    return launch_pdl_ex(kern, grid, block, smem, st, false, args...);
}

// Cooperative launch without programmatic serialization.
template <typename... KArgs, typename... Args>
inline pkv_status launch_coop(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? launch_status() : PKV_ERR_CUDA;
}

// Launch of a kernel whose CTAs wait on one another: cooperative (every CTA
// resident at once, else the launch is refused) together with programmatic
// serialization where the driver takes both, else cooperative alone.  `mode`
// keeps, per kernel, the first combination that launched (-1: not tried yet,
// 0: both attributes, 1: cooperative only).
template <typename... KArgs, typename... Args>
inline pkv_status launch_resident(std::atomic<int> &mode, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t st, Args... args) {
    int m = mode.load();
    if (m >= 0)
        return m == 0 ? launch_pdl_ex(kern, grid, block, smem, st, true, args...)
                      : launch_coop(kern, grid, block, smem, st, args...);
    if (launch_pdl_ex(kern, grid, block, smem, st, true, args...) == PKV_OK) {
        mode.store(0);
        return PKV_OK;
    }
    (void)cudaGetLastError();  // the refused combination's error, before the next attempt
    const pkv_status rc = launch_coop(kern, grid, block, smem, st, args...);
    if (rc == PKV_OK) mode.store(1);
    return rc;
}

__device__ __forceinline__ void flag_error(unsigned int *err, unsigned int bits) {
    if (err) atomicOr(err, bits);
}

// FP8 (E4M3) quantisation shared by the cache write and the fused append:
// code = the E4M3 value nearest to the float32 quotient x / scale (IEEE
// division), ties to even, saturating at +-448 (cvt ... satfinite).
// Two codes, low byte = lo.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 1 / scale when scale is a positive power of two whose reciprocal is a normal
// float, else 0.  Then x * (1 / scale) is the same real number as x / scale,
// rounded once, so its codes are the division's, bit for bit.
__device__ __forceinline__ float pow2_reciprocal(float scale) {
    const uint32_t b = __float_as_uint(scale);
    const uint32_t ex = (b >> 23) & 0xffu;
    return (b & 0x807fffffu) == 0u && ex >= 1u && ex <= 253u ? __uint_as_float((254u - ex) << 23) : 0.f;
}

__device__ __forceinline__ void quantize16(const uint4 (&x)[2], float scale, uint32_t (&w)[4]) {
    const uint32_t *e = reinterpret_cast<const uint32_t *>(x);
    const float inv = pow2_reciprocal(scale);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bf16 pairs (4 values) -> 4 codes, low byte first
        const uint32_t p0 = e[2 * i], p1 = e[2 * i + 1];
        const float x0 = __uint_as_float(p0 << 16), x1 = __uint_as_float(p0 & 0xffff0000u);
        const float x2 = __uint_as_float(p1 << 16), x3 = __uint_as_float(p1 & 0xffff0000u);
        float f0, f1, f2, f3;
        if (inv != 0.f) {  // a power-of-two scale: one multiply each
            f0 = __fmul_rn(x0, inv);
            f1 = __fmul_rn(x1, inv);
            f2 = __fmul_rn(x2, inv);
            f3 = __fmul_rn(x3, inv);
        } else {
            f0 = __fdiv_rn(x0, scale);
            f1 = __fdiv_rn(x1, scale);
            f2 = __fdiv_rn(x2, scale);
            f3 = __fdiv_rn(x3, scale);
        }
        w[i] = e4m3x2(f0, f1) | (e4m3x2(f2, f3) << 16);
    }
}

// Balanced split of the decode kernel: T tiles of all (sequence, kv head)
// segments laid end to end, cut into `parts` equal contiguous shares, share c
// = [floor(c T / parts), floor((c + 1) T / parts)).  A segment of n tiles
// meets at most ceil(n / share) + 1 shares and has `slots` partial slots, so
// shares hold at least ceil(seg_max / (slots - 1)) tiles; at most `warps`
// shares.  The kernel and the host diagnostic hooks share this code.
__host__ __device__ __forceinline__ int64_t balanced_parts(int64_t T, int seg_max, int slots, int64_t warps) {
    const int64_t min_share = slots > 1 ? ((seg_max + slots - 2) / (slots - 1) > 1 ? (seg_max + slots - 2) / (slots - 1) : 1)
                                        : (T > 1 ? T : 1);
    int64_t parts = T / min_share;
    if (parts < 1) parts = 1;
    if (parts > warps) parts = warps;
    return parts;
}

// Share that holds tile t.
__host__ __device__ __forceinline__ int64_t share_owner(int64_t t, int64_t T, int64_t parts) {
    return ((t + 1) * parts + T - 1) / T - 1;
}

}  // namespace pkv

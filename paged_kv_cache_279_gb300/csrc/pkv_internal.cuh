// Internal helpers shared by the library's CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

__device__ __forceinline__ void quantize16(const uint4 (&x)[2], float scale, uint32_t (&w)[4]) {
    const uint32_t *e = reinterpret_cast<const uint32_t *>(x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bf16 pairs (4 values) -> 4 codes, low byte first
        const uint32_t p0 = e[2 * i], p1 = e[2 * i + 1];
        const float f0 = __fdiv_rn(__uint_as_float(p0 << 16), scale);
        const float f1 = __fdiv_rn(__uint_as_float(p0 & 0xffff0000u), scale);
        const float f2 = __fdiv_rn(__uint_as_float(p1 << 16), scale);
        const float f3 = __fdiv_rn(__uint_as_float(p1 & 0xffff0000u), scale);
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

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

}  // namespace pkv

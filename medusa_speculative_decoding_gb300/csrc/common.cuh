// common.cuh -- shared helpers of libmedusa_gb300 (status handling, device
// properties, bf16 decoding, warp reductions, streaming loads).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "medusa.h"

namespace medusa {

// Records a message for medusa_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
// Checks the launch that was just enqueued; returns MEDUSA_OK or MEDUSA_ERR_CUDA.
int check_launch(const char* what);
// Number of SMs of the current device (cached per device).
int sm_count();
// Opt-in maximum dynamic shared memory per block of the current device.
int max_smem_optin();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16-byte load that bypasses L1 (weights and caches are streamed once per step).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// (value, index) order used by every top-k and argmax here: larger value
// first, lower index first among equal values.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

}  // namespace medusa

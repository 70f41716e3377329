// common.cuh -- small device helpers shared by the kernels of this library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace m2 {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the hardware exponent unit (PTX ex2.approx.ftz.f32).  Every caller
// passes x <= 0 (a masked log2-space decay), so results lie in [0, 1] and an
// underflow to 0 is the intended limit.
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Element loads/stores for the two I/O types.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

__device__ __forceinline__ void record_error(int32_t* err, int32_t bits) {
    if (err) atomicOr(err, bits);
}

}  // namespace m2

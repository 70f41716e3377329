// common.cuh -- small device helpers shared by the kernels of this library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace m2 {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the hardware exponent unit (PTX ex2.approx.ftz.f32).  Callers pass
// x <= 0 (a masked log2-space decay: results in [0, 1], an underflow to 0 is
// the intended limit), except stage 4's diagonal-block reference factor,
// whose argument is at most 14.
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

// Programmatic dependent launch.  A kernel launched with it may start while the
// previous kernel of the stream is still running: grid_dep_wait() blocks until
// that kernel has completed and its writes are visible (a no-op for a kernel
// launched without it); grid_dep_launch() lets the next kernel of the stream
// start launching once every CTA of this grid has issued it or exited.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch k<<<grid, block, smem, st>>>(args...), with programmatic dependent
// launch allowed when pdl is set.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace m2

// internal.h -- launchers shared between the C-ABI layer (api.cu) and the kernels.
// Not part of the public interface (include/mamba2_ssd.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace m2 {

// Problem dimensions of one call, after validation.
struct Dims {
    int64_t b, T, H, P, N, G, L, nc;
    int dtype;   // 0 = f32, 1 = bf16 (element type of x, B, C, y, Sprev)
};

// Element counts and byte sizes of the intermediates.
inline int64_t n_cum(const Dims& d) { return d.b * d.H * d.T; }
inline int64_t n_state(const Dims& d) { return d.b * d.nc * d.H * d.P * d.N; }
inline int64_t esize(const Dims& d) { return d.dtype == 1 ? 2 : 4; }

// Stage 1: chunk-local log2-scaled cumsum + [b,h,t] transpose of dt.
cudaError_t launch_chunk_cumsum(const Dims& d, const float* dt, const float* A, float* cum2,
                                float* dtT, int32_t* err, cudaStream_t st);

// Stage 2: chunk states.  CUDA-core variant (any supported shape / dtype).
cudaError_t launch_chunk_state_simt(const Dims& d, const void* x, const void* B,
                                    const float* cum2, const float* dtT, float* dS,
                                    int32_t* err, cudaStream_t st);
// Stage 2: tcgen05 variant (bf16, shapes accepted by tc_supported()).
cudaError_t launch_chunk_state_tc(const Dims& d, const void* x, const void* B,
                                  const float* cum2, const float* dtT, float* dS,
                                  int32_t* err, cudaStream_t st);

// Stage 3: sequential state pass over chunks.
cudaError_t launch_state_pass(const Dims& d, const float* dS, const float* cum2,
                              const float* init, void* Sprev, float* final_state,
                              int32_t* err, cudaStream_t st);

// Stage 4: fused output.  CUDA-core variant.
cudaError_t launch_chunk_out_simt(const Dims& d, const void* x, const void* B, const void* C,
                                  const float* cum2, const float* dtT, const void* Sprev,
                                  const float* D, void* y, int32_t* err, cudaStream_t st);
// Stage 4: tcgen05 variant.
cudaError_t launch_chunk_out_tc(const Dims& d, const void* x, const void* B, const void* C,
                                const float* cum2, const float* dtT, const void* Sprev,
                                const float* D, void* y, int32_t* err, cudaStream_t st);

// True when the tcgen05 kernels handle this shape.
bool tc_supported(const Dims& d);

// Device-side error bits (OR-ed into the library's error word).
enum : int32_t {
    kErrTimeoutK2 = 1 << 0,    // a bounded wait ran out in the tcgen05 chunk-state kernel
    kErrTimeoutK4 = 1 << 1,    // ... in the tcgen05 chunk-output kernel
    kErrLaunchCfg = 1 << 2,    // a kernel saw a launch configuration it does not support
};

}  // namespace m2

// fwd_noalloc.cu -- mamba2_ssd_fwd_noalloc: the forward pass without any
// allocation, for callers that cannot allocate device memory themselves (a
// host framework that owns every allocation, a plug-in that may not call the
// CUDA allocator, a hot path that must not allocate).  The workspace comes
// from a fixed device array compiled into this library; everything else is
// mamba2_ssd_fwd unchanged.
#include <cuda_runtime.h>

#include <mutex>

#include "mamba2_ssd.h"

namespace {

// The shared scratch.  In host code this name is only a host-side stand-in:
// its device address is obtained with cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MAMBA2_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device; looked up once per
// device (the first call on a device), with that device current.  The cached
// address belongs to the device's primary context, the one the CUDA runtime
// uses; it stays valid for the life of the process unless that context is
// destroyed (cudaDeviceReset).
mamba2_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();   // leave no error pending for the caller's next call
        return MAMBA2_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MAMBA2_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();   // the failed lookup must not surface in a later launch check
            return MAMBA2_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MAMBA2_OK;
}

}  // namespace

extern "C" mamba2_status mamba2_ssd_fwd_noalloc(const mamba2_ssd_shape* shape, const void* x,
                                                const float* dt, const float* A, const void* B,
                                                const void* C, const float* D,
                                                const float* initial_state, void* y,
                                                float* final_state, void* stream) {
    mamba2_status st = mamba2_ssd_check_shape(shape);
    if (st != MAMBA2_OK) return st;
    // Too large for the fixed scratch: reject before touching the GPU.
    if (mamba2_ssd_workspace_size(shape) > MAMBA2_NOALLOC_SCRATCH_BYTES) return MAMBA2_ERR_WORKSPACE;
    void* ws = nullptr;
    st = scratch_address(&ws);
    if (st != MAMBA2_OK) return st;
    return mamba2_ssd_fwd(shape, x, dt, A, B, C, D, initial_state, y, final_state, ws,
                          MAMBA2_NOALLOC_SCRATCH_BYTES, stream);
}

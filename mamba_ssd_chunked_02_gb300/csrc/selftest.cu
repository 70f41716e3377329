// selftest.cu -- make the library's bounded waits run out, on purpose, safely.
//
// One CTA waits on an mbarrier that nothing arrives at (mbar_wait_or_abort, the
// wait every tensor-core kernel uses between its roles) and on a global flag word
// that nothing sets (wait_flag, the wait of the fused stage 2+3 kernel), each for
// at most `limit_ns`.  Both must give up and report: the kernel then sets
// kErrSelfTest in the device error word and returns normally, so the context
// stays usable.  Nothing faults, traps or hangs.
#include "common.cuh"
#include "internal.h"
#include "tc5.cuh"

namespace m2 {
namespace {

__device__ int32_t g_never_set;   // zero-initialised and never written

__global__ void __launch_bounds__(64) wait_timeout_kernel(uint64_t limit_ns, int32_t* err) {
    using namespace tc;
    __shared__ uint64_t bar;
    __shared__ int abort_mb, abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        abort_mb = 0;
        abort_flag = 0;
    }
    __syncthreads();
    bool got = true;
    if (threadIdx.x == 0) got = mbar_wait_or_abort(&bar, 0, &abort_mb, limit_ns);
    if (threadIdx.x == 32) got = wait_flag(&g_never_set, &abort_flag, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0 && !got && abort_mb) record_error(err, kErrSelfTest);
    if (threadIdx.x == 32 && !got && abort_flag) record_error(err, kErrSelfTest);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int32_t* err, cudaStream_t st) {
    wait_timeout_kernel<<<1, 64, 0, st>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace m2

// tc_stub.cu -- placeholder until the tcgen05 kernels land: no shape takes the
// tensor-core path.
#include "internal.h"

namespace m2 {
bool tc_supported(const Dims&) { return false; }
cudaError_t launch_chunk_state_tc(const Dims&, const void*, const void*, const float*,
                                  const float*, float*, int32_t*, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_chunk_out_tc(const Dims&, const void*, const void*, const void*, const float*,
                                const float*, const void*, const float*, void*, int32_t*,
                                cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace m2

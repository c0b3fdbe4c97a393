// Tensor-core kernel placeholder.
#include "pq_internal.h"

namespace pqk {
unsigned tc_wait_timeouts(bool) { return 0; }
bool tc_supported(int, int64_t, int64_t, int) { return false; }
cudaError_t launch_gemv_tc(int, const uint8_t *, int64_t, int64_t, const float *, int, float *,
                           int64_t, cudaStream_t, const DeviceInfo &) {
    return cudaErrorNotSupported;
}
}  // namespace pqk

// Streaming kernel placeholder (filled in below by the bulk-copy ring kernel).
#include "pq_internal.h"

namespace pqk {
bool stream_supported(int, int64_t, int64_t, int) { return false; }
cudaError_t launch_gemv_stream(int, const uint8_t *, int64_t, int64_t, const float *, int, float *,
                               int64_t, cudaStream_t, const DeviceInfo &) {
    return cudaErrorNotSupported;
}
}  // namespace pqk

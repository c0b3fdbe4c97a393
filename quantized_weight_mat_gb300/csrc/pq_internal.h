// Internal interface between the C ABI (pq_api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "pq.h"

namespace pqk {

constexpr int kMaxDeviceIds = 64;   // device ordinals served by the per-device state below

// A set-up step that must run once on every device a kernel is launched on
// (function attributes are per device): thread-safe, and a failed step keeps
// its status, so every later call on that device returns it.
class PerDeviceOnce {
public:
    template <class F> cudaError_t run(F step) {
        int dev = 0;
        const cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDeviceIds) return cudaErrorInvalidDevice;
        std::call_once(flag_[dev], [&] { status_[dev] = step(); });
        return status_[dev];
    }

private:
    std::once_flag flag_[kMaxDeviceIds];
    cudaError_t status_[kMaxDeviceIds] = {};
};

constexpr int kNumFmts = 8;                                       // pq_fmt values 0..7
constexpr int kQK[kNumFmts] = {32, 256, 256, 1, 256, 256, 256, 2};  // weights per block
constexpr int kBlockBytes[kNumFmts] = {34, 144, 210, 1, 176, 110, 84, 1};   // bytes per block

// Byte offset of the f32 scales of a per-row int8 matrix.
inline int64_t i8row_scale_offset(int64_t n_out, int64_t k) { return (n_out * k + 15) / 16 * 16; }
// Byte offset of the f32 scales of a per-row int4 matrix (k even).
inline int64_t i4row_scale_offset(int64_t n_out, int64_t k) { return (n_out * (k / 2) + 15) / 16 * 16; }

struct DeviceInfo {
    int sm_count;
    int major, minor;
    size_t smem_optin;   // max dynamic shared memory per block (opt-in)
    int l2_bytes;
};

// Cached per-device properties of the current device; nullptr on failure.
const DeviceInfo *device_info();

// Library-owned stream-ordered memory pool of the current device (scratch
// memory taken with cudaMallocFromPoolAsync, kept for reuse); null on failure.
cudaMemPool_t scratch_pool();

// Epilogue applied to the mat-vec outputs before they are stored.
//   kEpiBias:   y[b][r] = (W x_b)[r] + bias[r]
//   kEpiSwiGLU: W is a fused gate+up matrix of n_out = 2 * n_ff rows (gate
//               rows first); h[b][j] = silu((W x_b)[j]) * (W x_b)[n_ff + j],
//               stored as [batch][n_ff]
constexpr int kEpiNone = 0, kEpiBias = 1, kEpiSwiGLU = 2;
struct Epilogue {
    int kind = kEpiNone;
    const float *bias = nullptr;
};

// Launchers: arguments already validated; return cudaError_t of the launch.
cudaError_t launch_dequant(int fmt, const uint8_t *w, int64_t n_out, int64_t k, float *out,
                           cudaStream_t s);

cudaError_t launch_gemv_generic(int fmt, const uint8_t *w, int64_t n_out, int64_t k,
                                const float *x, int batch, float *y, int64_t ldy,
                                cudaStream_t s, int sm_count);

// Streaming kernel (bulk-copy ring).  `supported` reports whether it can run
// this case; the launcher handles batch <= 4, and batch <= 8 where
// `stream_mma_takes` (the register-operand whole-row kernel: Q4_K and Q6_K at
// k = 4096, batch 3-8) holds.
bool stream_supported(int fmt, int64_t n_out, int64_t k, int batch);
bool stream_mma_takes(int fmt, int64_t n_out, int64_t k, int batch);
cudaError_t launch_gemv_stream(int fmt, const uint8_t *w, int64_t n_out, int64_t k,
                               const float *x, int batch, float *y, int64_t ldy,
                               cudaStream_t s, const DeviceInfo &dev);
// The batch-1 whole-row kernel (every format with a whole-row policy) and
// the register-operand whole-row kernel (batch 2-8) with the epilogue fused
// into their stores; `stream_epilogue_fused` says whether one takes the case.
// y has leading dimension ldy (for SwiGLU: n_out / 2 outputs per column).
bool stream_epilogue_fused(int fmt, int64_t n_out, int64_t k, int batch, int kind);
cudaError_t launch_gemv_stream_epi(int fmt, const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch,
                                   float *y, int64_t ldy, cudaStream_t s, const DeviceInfo &dev, const Epilogue &epi);

// Tensor-core kernel (tcgen05): Q4_K, batch chunks of 8 or 16.
bool tc_supported(int fmt, int64_t n_out, int64_t k, int batch);
// The epilogue is fused: the bias is added at the final store, SwiGLU pairs
// gate and up tiles in the finishing kernel (y is then h, [batch][n_out / 2]
// with row stride ldy).
cudaError_t launch_gemv_tc(int fmt, const uint8_t *w, int64_t n_out, int64_t k,
                           const float *x, int batch, float *y, int64_t ldy,
                           cudaStream_t s, const DeviceInfo &dev, const Epilogue &epi = Epilogue{});

// Allocation-free variant of the tensor-core kernel: the x image lives in a
// fixed device array instead of pool memory (k <= noalloc_max_k(), batch <= 16).
int noalloc_max_k();
cudaError_t launch_gemv_tc_noalloc(const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch,
                                   float *y, int64_t ldy, cudaStream_t s, const DeviceInfo &dev);

// Stand-alone epilogue kernels (epilogue.cu) for kernels without a fused one:
// y[b][r] += bias[r]; h[b][j] = silu(g[b][j]) * g[b][n_ff + j] with g
// [batch][2 n_ff].
cudaError_t launch_add_bias(float *y, const float *bias, int64_t n_out, int64_t ldy, int batch, cudaStream_t s);
cudaError_t launch_swiglu_rows(const float *g, int64_t n_ff, int batch, float *h, int64_t ldh, cudaStream_t s);

// Process-wide: may kernels read weights before the preceding kernel on the
// stream has finished (set by pq_set_weight_prefetch)?
int weight_prefetch();

// Bounded waits that ran out in each kernel file since the last reset.
unsigned stream_wait_timeouts(bool reset);
unsigned tc_wait_timeouts(bool reset);
unsigned selftest_wait_timeouts(bool reset);
// Bounded-wait self-test: 1 if the wait ran out and the kernel returned, 0 if
// it completed, -1 on a CUDA error.  Synchronises `s`.
int run_selftest_wait(unsigned long long limit_ns, cudaStream_t s);

}  // namespace pqk

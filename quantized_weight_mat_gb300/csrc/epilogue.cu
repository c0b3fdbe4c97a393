// Epilogues as their own small kernels, for the cases whose mat-vec kernel
// has none fused (batch 2-4 on the CUDA-core kernels, the generic kernel).
// The batch-1 whole-row kernel and the tensor-core kernel fuse them into
// their stores instead.  The operations (PESTI README, "Conformance"): the
// QKV projections carry a bias; the MLP multiplies silu of the gate
// projection by the up projection.

#include "pq_internal.h"

namespace pqk {
namespace {

// y[b][r] += bias[r]
__global__ void __launch_bounds__(256) add_bias(float *__restrict__ y, const float *__restrict__ bias,
                                                long long n_out, long long ldy, int batch) {
    const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_out) return;
    const float bv = bias[r];
    for (int b = 0; b < batch; ++b) y[(size_t)b * ldy + r] += bv;
}

// silu(z) = z / (1 + e^-z) with CUDA's expf
__device__ __forceinline__ float silu_epi(float z) { return z / (1.0f + expf(-z)); }

// h[b][j] = silu(g[b][j]) * g[b][n_ff + j], g = [batch][2 n_ff]
__global__ void __launch_bounds__(256) swiglu_rows(const float *__restrict__ g, long long n_ff, int batch,
                                                   float *__restrict__ h, long long ldh) {
    const long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n_ff) return;
    for (int b = 0; b < batch; ++b) {
        const float *gb = g + (size_t)b * 2 * n_ff;
        h[(size_t)b * ldh + j] = silu_epi(gb[j]) * gb[n_ff + j];
    }
}

}  // namespace

cudaError_t launch_add_bias(float *y, const float *bias, int64_t n_out, int64_t ldy, int batch, cudaStream_t s) {
    add_bias<<<(unsigned)((n_out + 255) / 256), 256, 0, s>>>(y, bias, n_out, ldy, batch);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_rows(const float *g, int64_t n_ff, int batch, float *h, int64_t ldh, cudaStream_t s) {
    swiglu_rows<<<(unsigned)((n_ff + 255) / 256), 256, 0, s>>>(g, n_ff, batch, h, ldh);
    return cudaGetLastError();
}

}  // namespace pqk

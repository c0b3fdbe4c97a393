// Self-test of the failure detection the kernels rely on: every mbarrier
// wait is bounded in time, and a wait that runs out is counted and ends the
// wait instead of hanging the GPU.  This kernel waits on a barrier that
// nothing completes, with a short limit, and reports what happened.

#include "pq_internal.h"
#include "pq_ptx.cuh"

namespace pqk {
namespace {

__device__ int g_selftest_status;

__global__ void selftest_wait(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    // nothing arrives on `bar`: the bounded wait must run out and return false
    const bool completed = mbar_wait_for(&bar, 0u, limit_ns);
    g_selftest_status = completed ? 0 : 1;
}

}  // namespace

unsigned selftest_wait_timeouts(bool reset) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) return 0;
    if (reset) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_wait_timeouts, &z, sizeof(z));
    }
    return v;
}

int run_selftest_wait(unsigned long long limit_ns, cudaStream_t s) {
    const int minus_one = -1;
    if (cudaMemcpyToSymbolAsync(g_selftest_status, &minus_one, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return -1;
    selftest_wait<<<1, 32, 0, s>>>(limit_ns);
    if (cudaGetLastError() != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    int status = -1;
    if (cudaMemcpyFromSymbol(&status, g_selftest_status, sizeof(int)) != cudaSuccess) return -1;
    return status;
}

}  // namespace pqk

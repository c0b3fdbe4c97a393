// C ABI of the library: argument checks, kernel choice, launches.
//
// Every check runs on the host before any launch, so a rejected call never
// touches the GPU.  The state kept here: a per-device record of properties,
// filled once per device, and a per-device scratch memory pool.

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "pq_internal.h"

namespace pqk {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];
bool g_ok[kMaxDevices];

void fill_info(int dev) {
    DeviceInfo &d = g_info[dev];
    int v = 0;
    g_ok[dev] = false;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return;
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return;
    if (cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return;
    d.smem_optin = (size_t)v;
    if (cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return;
    g_ok[dev] = true;
}
}  // namespace

namespace {
std::atomic<int> g_weight_prefetch{0};
}

int weight_prefetch() { return g_weight_prefetch.load(std::memory_order_relaxed); }

const DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_once[dev], fill_info, dev);
    return g_ok[dev] ? &g_info[dev] : nullptr;
}

// Stream-ordered scratch for kernels that need some (x images, partial
// sums): a library-owned memory pool per device that keeps freed memory for
// reuse.
cudaMemPool_t scratch_pool() {
    static cudaMemPool_t pools[64] = {};
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::call_once(once[dev], [dev] {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
            uint64_t keep = ~0ull;
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
            pools[dev] = pool;
        }
    });
    return pools[dev];
}

}  // namespace pqk

using namespace pqk;

namespace {

bool valid_fmt(int fmt) { return fmt >= 0 && fmt < kNumFmts; }

// Bytes of W, or -1 when the shape is invalid / overflows.
int64_t weight_bytes64(int fmt, int64_t n_out, int64_t k) {
    if (!valid_fmt(fmt) || n_out <= 0 || k <= 0) return -1;
    if (k % kQK[fmt]) return -1;
    if (n_out > (INT64_C(1) << 40) / k) return -1;   // n_out*k <= 2^40 weights
    if (fmt == PQ_I8_ROW) return i8row_scale_offset(n_out, k) + 4 * n_out;
    if (fmt == PQ_I4_ROW) return i4row_scale_offset(n_out, k) + 4 * n_out;
    return n_out * (k / kQK[fmt]) * kBlockBytes[fmt];
}

bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

int check_common(int fmt, const void *w, int n_out, int k) {
    if (!valid_fmt(fmt)) return PQ_ERR_FMT;
    if (!w || n_out <= 0 || k <= 0) return PQ_ERR_ARG;
    if (k % kQK[fmt]) return PQ_ERR_K;
    if (weight_bytes64(fmt, n_out, k) < 0) return PQ_ERR_SIZE;
    if ((uintptr_t)w % 16) return PQ_ERR_ALIGN;
    return PQ_OK;
}

int check_device(const DeviceInfo **out) {
    const DeviceInfo *dev = device_info();
    if (!dev || dev->major != 10 || dev->minor != 3) return PQ_ERR_DEVICE;
    *out = dev;
    return PQ_OK;
}

int check_gemv(int fmt, const void *w, int n_out, int k, const float *x, int batch,
               const float *y) {
    int st = check_common(fmt, w, n_out, k);
    if (st) return st;
    if (!x || !y || batch <= 0) return PQ_ERR_ARG;
    if ((int64_t)batch * n_out > (INT64_C(1) << 40) || (int64_t)batch * k > (INT64_C(1) << 40))
        return PQ_ERR_SIZE;
    if ((uintptr_t)x % 16 || (uintptr_t)y % 4) return PQ_ERR_ALIGN;
    const int64_t ybytes = 4 * (int64_t)batch * n_out;
    if (overlaps(y, ybytes, w, weight_bytes64(fmt, n_out, k)) ||
        overlaps(y, ybytes, x, 4 * (int64_t)batch * k))
        return PQ_ERR_ARG;
    return PQ_OK;
}

// Kernel for one chunk of `nb` batch columns.  The tensor-core kernel costs
// about the same at any batch up to 16, so it also takes batch 3-4 where the
// CUDA-core kernels are slower: long rows (k >= 8192), and at batch 4 large
// matrices (>= 2^25 weights); measured on 4096x14336, 14336x4096, 28672x4096.
int choose(int fmt, int64_t n_out, int64_t k, int nb) {
    // Q4_K / Q6_K at k = 4096, batch 3-8: the register-operand whole-row kernel
    // (14336x4096 batch 4: 12.1 us against 17.4 for the tensor-core kernel)
    if (nb <= 8 && stream_mma_takes(fmt, n_out, k, nb)) return PQ_KERNEL_STREAM;
    const bool tc_pays = nb >= 5 || (nb >= 3 && k >= 8192) || (nb == 4 && n_out * k >= (INT64_C(1) << 25));
    if (tc_pays && tc_supported(fmt, n_out, k, nb)) return PQ_KERNEL_TC;
    if (nb <= 4 && stream_supported(fmt, n_out, k, nb)) return PQ_KERNEL_STREAM;
    // Q8_0, per-row int8 and the rest of the K family have a streaming kernel
    // for one column only (Q6_K for 1-4); one launch per column still beats
    // the generic kernel (Q6_K LM head 128256x4096, one column at a time:
    // 2 x 65 us against 301 us at batch 2)
    if (fmt != PQ_Q4_K && stream_supported(fmt, n_out, k, 1)) return PQ_KERNEL_STREAM;
    return PQ_KERNEL_GENERIC;
}

// Chunking of the batch: chunks of up to 32 columns (the tensor-core kernel
// takes 1-32: one pass over W for a 32-row prompt); a chunk that no
// tensor-core kernel takes is split further into chunks of up to 4, and into
// single columns for a streaming kernel that only takes one.
template <class F>
int for_each_chunk(int fmt, int64_t n_out, int64_t k, int batch, int forced, F &&f) {
    for (int b0 = 0; b0 < batch;) {
        int nb = batch - b0 < 32 ? batch - b0 : 32;
        int kern = forced >= 0 ? forced : choose(fmt, n_out, k, nb);
        if (kern != PQ_KERNEL_TC && nb > 4 && !(kern == PQ_KERNEL_STREAM && stream_mma_takes(fmt, n_out, k, nb < 8 ? nb : 8)))
            nb = 4;
        if (kern == PQ_KERNEL_STREAM && nb > 8) nb = 8;
        // a streaming kernel that takes one column at a time runs column by column
        if (kern == PQ_KERNEL_STREAM && nb > 1 && !stream_supported(fmt, n_out, k, nb) &&
            stream_supported(fmt, n_out, k, 1))
            nb = 1;
        if (kern == PQ_KERNEL_STREAM && !stream_supported(fmt, n_out, k, nb)) return PQ_ERR_KERNEL;
        if (kern == PQ_KERNEL_TC && !tc_supported(fmt, n_out, k, nb)) return PQ_ERR_KERNEL;
        int st = f(kern, b0, nb);
        if (st) return st;
        b0 += nb;
    }
    return PQ_OK;
}

// Mat-vec with an optional epilogue.  The kernel choice is pq_gemv's for the
// n_out x k matrix (for SwiGLU the fused 2 * n_ff-row matrix); the batch-1
// whole-row kernel, the register-operand kernel (Q4_K and Q6_K at k = 4096,
// batch 2-8) and the tensor-core kernels fuse the epilogue into their
// stores, the others run it as a small kernel afterwards (SwiGLU through a
// pool buffer of batch x n_out outputs).
int gemv_epi_impl(int fmt, const void *w_blocks, int n_out, int k, const float *x, int batch, float *y,
                  cudaStream_t stream, const Epilogue &epi) {
    const DeviceInfo *dev = nullptr;
    int st = check_device(&dev);
    if (st) return st;
    const bool sw = epi.kind == kEpiSwiGLU;
    const int64_t ldy = sw ? n_out / 2 : n_out;
    const uint8_t *w = static_cast<const uint8_t *>(w_blocks);
    st = for_each_chunk(fmt, n_out, k, batch, PQ_KERNEL_AUTO, [](int, int, int) { return PQ_OK; });
    if (st) return st;
    return for_each_chunk(fmt, n_out, k, batch, PQ_KERNEL_AUTO, [&](int kern, int b0, int nb) {
        const float *xb = x + (int64_t)b0 * k;
        float *yb = y + (int64_t)b0 * ldy;
        cudaError_t e;
        if (kern == PQ_KERNEL_TC) {
            e = launch_gemv_tc(fmt, w, n_out, k, xb, nb, yb, ldy, stream, *dev, epi);
        } else if (kern == PQ_KERNEL_STREAM && stream_epilogue_fused(fmt, n_out, k, nb, epi.kind)) {
            e = launch_gemv_stream_epi(fmt, w, n_out, k, xb, nb, yb, ldy, stream, *dev, epi);
        } else {
            // plain mat-vec, then the epilogue kernel
            float *out = yb;
            void *tmp = nullptr;
            if (sw) {
                cudaMemPool_t pool = scratch_pool();
                if (!pool) return PQ_ERR_LAUNCH;
                if (cudaMallocFromPoolAsync(&tmp, (size_t)nb * n_out * 4, pool, stream) != cudaSuccess)
                    return PQ_ERR_LAUNCH;
                out = static_cast<float *>(tmp);
            }
            if (kern == PQ_KERNEL_STREAM)
                e = launch_gemv_stream(fmt, w, n_out, k, xb, nb, out, n_out, stream, *dev);
            else
                e = launch_gemv_generic(fmt, w, n_out, k, xb, nb, out, n_out, stream, dev->sm_count);
            if (e == cudaSuccess)
                e = sw ? launch_swiglu_rows(out, n_out / 2, nb, yb, ldy, stream)
                       : launch_add_bias(yb, epi.bias, n_out, ldy, nb, stream);
            if (tmp) {
                const cudaError_t f = cudaFreeAsync(tmp, stream);
                if (e == cudaSuccess) e = f;
            }
        }
        return e == cudaSuccess ? PQ_OK : PQ_ERR_LAUNCH;
    });
}

int gemv_impl(int fmt, const void *w_blocks, int n_out, int k, const float *x, int batch,
              float *y, cudaStream_t stream, int kernel) {
    int st = check_gemv(fmt, w_blocks, n_out, k, x, batch, y);
    if (st) return st;
    if (kernel < PQ_KERNEL_AUTO || kernel > PQ_KERNEL_TC) return PQ_ERR_KERNEL;
    const DeviceInfo *dev = nullptr;
    if ((st = check_device(&dev))) return st;
    const uint8_t *w = static_cast<const uint8_t *>(w_blocks);
    // validate every chunk before the first launch
    st = for_each_chunk(fmt, n_out, k, batch, kernel, [](int, int, int) { return PQ_OK; });
    if (st) return st;
    return for_each_chunk(fmt, n_out, k, batch, kernel, [&](int kern, int b0, int nb) {
        const float *xb = x + (int64_t)b0 * k;
        float *yb = y + (int64_t)b0 * n_out;
        cudaError_t e;
        if (kern == PQ_KERNEL_TC)
            e = launch_gemv_tc(fmt, w, n_out, k, xb, nb, yb, n_out, stream, *dev);
        else if (kern == PQ_KERNEL_STREAM)
            e = launch_gemv_stream(fmt, w, n_out, k, xb, nb, yb, n_out, stream, *dev);
        else
            e = launch_gemv_generic(fmt, w, n_out, k, xb, nb, yb, n_out, stream, dev->sm_count);
        return e == cudaSuccess ? PQ_OK : PQ_ERR_LAUNCH;
    });
}

}  // namespace

extern "C" {

size_t pq_weight_bytes(pq_fmt fmt, int n_out, int k) {
    const int64_t n = weight_bytes64((int)fmt, n_out, k);
    return n < 0 ? 0 : (size_t)n;
}

const char *pq_strerror(int status) {
    switch (status) {
    case PQ_OK: return "ok";
    case PQ_ERR_ARG: return "invalid argument (null pointer, non-positive size, or overlapping output)";
    case PQ_ERR_FMT: return "unknown quantization format";
    case PQ_ERR_K: return "k is not a multiple of the format's block size";
    case PQ_ERR_ALIGN: return "misaligned pointer (w and x need 16 bytes, y and out need 4 or 16)";
    case PQ_ERR_SIZE: return "sizes overflow";
    case PQ_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103)";
    case PQ_ERR_LAUNCH: return "CUDA kernel launch failed";
    case PQ_ERR_KERNEL: return "the requested kernel does not support this case";
    }
    return "unknown status";
}

int pq_gemv(pq_fmt fmt, const void *w_blocks, int n_out, int k, const float *x, int batch,
            float *y, struct CUstream_st *stream) {
    return gemv_impl((int)fmt, w_blocks, n_out, k, x, batch, y, stream, PQ_KERNEL_AUTO);
}

int pq_gemv_kernel(pq_fmt fmt, const void *w_blocks, int n_out, int k, const float *x,
                   int batch, float *y, struct CUstream_st *stream, int kernel) {
    return gemv_impl((int)fmt, w_blocks, n_out, k, x, batch, y, stream, kernel);
}

int pq_gemv_bias(pq_fmt fmt, const void *w_blocks, int n_out, int k, const float *x, int batch,
                 const float *bias, float *y, struct CUstream_st *stream) {
    int st = check_gemv((int)fmt, w_blocks, n_out, k, x, batch, y);
    if (st) return st;
    if (!bias) return PQ_ERR_ARG;
    if ((uintptr_t)bias % 4) return PQ_ERR_ALIGN;
    if (overlaps(y, 4 * (int64_t)batch * n_out, bias, 4 * (int64_t)n_out)) return PQ_ERR_ARG;
    Epilogue epi;
    epi.kind = kEpiBias;
    epi.bias = bias;
    return gemv_epi_impl((int)fmt, w_blocks, n_out, k, x, batch, y, stream, epi);
}

int pq_gemv_swiglu(pq_fmt fmt, const void *w_blocks, int n_ff, int k, const float *x, int batch, float *h,
                   struct CUstream_st *stream) {
    if (!valid_fmt((int)fmt)) return PQ_ERR_FMT;
    if (!w_blocks || !x || !h || n_ff <= 0 || k <= 0 || batch <= 0) return PQ_ERR_ARG;
    if (n_ff > 0x3fffffff) return PQ_ERR_SIZE;
    const int n_out = 2 * n_ff;
    int st = check_common((int)fmt, w_blocks, n_out, k);
    if (st) return st;
    if ((int64_t)batch * n_out > (INT64_C(1) << 40) || (int64_t)batch * k > (INT64_C(1) << 40)) return PQ_ERR_SIZE;
    if ((uintptr_t)x % 16 || (uintptr_t)h % 4) return PQ_ERR_ALIGN;
    const int64_t hbytes = 4 * (int64_t)batch * n_ff;
    if (overlaps(h, hbytes, w_blocks, weight_bytes64((int)fmt, n_out, k)) ||
        overlaps(h, hbytes, x, 4 * (int64_t)batch * k))
        return PQ_ERR_ARG;
    Epilogue epi;
    epi.kind = kEpiSwiGLU;
    return gemv_epi_impl((int)fmt, w_blocks, n_out, k, x, batch, h, stream, epi);
}

int pq_gemv_choice(pq_fmt fmt, int n_out, int k, int batch) {
    int st = check_common((int)fmt, (const void *)16, n_out, k);
    if (st) return st;
    if (batch <= 0) return PQ_ERR_ARG;
    return choose((int)fmt, n_out, k, batch < 32 ? batch : 32);
}

int pq_gemv_launches(pq_fmt fmt, int n_out, int k, int batch) {
    int st = check_common((int)fmt, (const void *)16, n_out, k);
    if (st) return st;
    if (batch <= 0) return PQ_ERR_ARG;
    int launches = 0;
    st = for_each_chunk((int)fmt, n_out, k, batch, PQ_KERNEL_AUTO, [&](int, int, int) {
        ++launches;
        return PQ_OK;
    });
    return st ? st : launches;
}

int pq_set_weight_prefetch(int enable) {
    return g_weight_prefetch.exchange(enable ? 1 : 0);
}

int pq_wait_timeouts(int reset) {
    const DeviceInfo *dev = nullptr;
    if (check_device(&dev)) return PQ_ERR_DEVICE;
    const unsigned n =
        stream_wait_timeouts(reset != 0) + tc_wait_timeouts(reset != 0) + selftest_wait_timeouts(reset != 0);
    return n > 0x7fffffffu ? 0x7fffffff : (int)n;
}

// Failure-detection self-test (see pq.h).
int pq_selftest_wait_timeout(unsigned limit_us, struct CUstream_st *stream) {
    if (limit_us < 1 || limit_us > 1000000) return PQ_ERR_ARG;
    const DeviceInfo *dev = nullptr;
    if (check_device(&dev)) return PQ_ERR_DEVICE;
    const int r = run_selftest_wait(1000ull * limit_us, stream);
    return r < 0 ? PQ_ERR_LAUNCH : r;
}

// Allocation-free mat-vec (tensor-core kernel with fixed scratch).  Checks as
// pq_gemv, then: Q4_K only (PQ_ERR_KERNEL otherwise), k <= noalloc_max_k()
// (PQ_ERR_SIZE otherwise).  Batches above 16 run in chunks of 16, one after
// another on `stream`, each reusing the scratch.
int pq_gemv_noalloc(pq_fmt fmt, const void *w_blocks, int n_out, int k, const float *x, int batch,
                    float *y, struct CUstream_st *stream) {
    int st = check_gemv((int)fmt, w_blocks, n_out, k, x, batch, y);
    if (st) return st;
    if (fmt != PQ_Q4_K) return PQ_ERR_KERNEL;
    if (k > noalloc_max_k()) return PQ_ERR_SIZE;
    const DeviceInfo *dev = nullptr;
    if ((st = check_device(&dev))) return st;
    for (int b0 = 0; b0 < batch; b0 += 16) {
        const int nb = batch - b0 < 16 ? batch - b0 : 16;
        cudaError_t e = launch_gemv_tc_noalloc(static_cast<const uint8_t *>(w_blocks), n_out, k,
                                               x + (int64_t)b0 * k, nb, y + (int64_t)b0 * n_out, n_out,
                                               stream, *dev);
        if (e != cudaSuccess) return PQ_ERR_LAUNCH;
    }
    return PQ_OK;
}

int pq_dequant(pq_fmt fmt, const void *w_blocks, int n_out, int k, float *out,
               struct CUstream_st *stream) {
    int st = check_common((int)fmt, w_blocks, n_out, k);
    if (st) return st;
    if (!out) return PQ_ERR_ARG;
    if ((uintptr_t)out % 16) return PQ_ERR_ALIGN;
    if (overlaps(out, 4 * (int64_t)n_out * k, w_blocks, weight_bytes64((int)fmt, n_out, k)))
        return PQ_ERR_ARG;
    const DeviceInfo *dev = nullptr;
    if ((st = check_device(&dev))) return st;
    cudaError_t e = launch_dequant((int)fmt, static_cast<const uint8_t *>(w_blocks), n_out, k, out,
                                   stream);
    return e == cudaSuccess ? PQ_OK : PQ_ERR_LAUNCH;
}

}  // extern "C"

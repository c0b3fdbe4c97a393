// Generic fused dequant + mat-vec: one warp per output row, any format,
// any shape, batch processed in chunks of up to 4 columns.
//
// This is the plain form of the operation (ember pull request, quant.rs
// description: decoding fused into the mat-vec, no f32 copy of W): the
// warp walks its row's blocks, each lane decodes 8 weights per Q4_K / Q6_K
// super-block (or per Q8_0 block group) to f32 in registers, multiplies by
// x (read through the read-only cache; x is small and shared by every warp
// of the SM) and accumulates in f32; a shuffle tree reduces the 32 lanes.
// It serves every case the specialised kernels do not, and is their
// reference point in the tests.

#include "pq_device.cuh"
#include "pq_internal.h"

namespace pqk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Launched with programmatic dependent launch when the whole grid is resident
// at once (at most one block per SM): the block may start while the previous
// kernel on the stream finishes and waits for it before reading anything.
// The next kernel is released only after that wait: these blocks hold no
// shared memory, so releasing it at the start let the blocks of a dozen
// launches ahead become resident at once (36-60 us before their turn, in a
// CUDA graph of back-to-back calls) and compete for the memory system with
// the launch that runs (Q8_0 896x896 3.65 -> 3.44 us with the order below).
// Without that launch attribute both instructions do nothing.
__device__ __forceinline__ void dependent_launch_prologue() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
}

template <int NB>
__device__ __forceinline__ void fma8(float (&acc)[NB], const float (&wv)[8], const float *x,
                                     int64_t k, int64_t i0, bool split4) {
    // weights i0..i0+7, or (split4) i0..i0+3 and i0+32..i0+35
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float *xb = x + b * k + i0;
        const float4 a = ldg_f4(xb);
        const float4 c = ldg_f4(xb + (split4 ? 32 : 4));
        acc[b] = fmaf(wv[0], a.x, acc[b]);
        acc[b] = fmaf(wv[1], a.y, acc[b]);
        acc[b] = fmaf(wv[2], a.z, acc[b]);
        acc[b] = fmaf(wv[3], a.w, acc[b]);
        acc[b] = fmaf(wv[4], c.x, acc[b]);
        acc[b] = fmaf(wv[5], c.y, acc[b]);
        acc[b] = fmaf(wv[6], c.z, acc[b]);
        acc[b] = fmaf(wv[7], c.w, acc[b]);
    }
}

template <int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_generic_q4_k(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                      float *__restrict__ y, int64_t ldy) {
    dependent_launch_prologue();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= n_out) return;
    const int nb = k / 256;
    const uint8_t *wr = w + (int64_t)row * nb * 144;
    const int c = lane >> 3, p0 = (lane & 7) * 4;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll 2
    for (int blk = 0; blk < nb; ++blk) {
        const uint8_t *bp = wr + (int64_t)blk * 144;
        const uint32_t dd = ldg_u32(bp);
        const uint32_t s0 = ldg_u32(bp + 4), s1 = ldg_u32(bp + 8), s2 = ldg_u32(bp + 12);
        const uint32_t qs = ldg_u32(bp + 16 + 4 * lane);
        const float d = h2f(dd), dmin = h2f(dd >> 16);
        int sc0, m0, sc1, m1;
        q4k_scale_min(s0, s1, s2, 2 * c, sc0, m0);
        q4k_scale_min(s0, s1, s2, 2 * c + 1, sc1, m1);
        const float dl0 = d * (float)sc0, ml0 = dmin * (float)m0;
        const float dl1 = d * (float)sc1, ml1 = dmin * (float)m1;
        float wv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t byte = (qs >> (8 * i)) & 0xff;
            wv[i] = dl0 * (float)(byte & 15) - ml0;
            wv[4 + i] = dl1 * (float)(byte >> 4) - ml1;
        }
        fma8<NB>(acc, wv, x, k, (int64_t)blk * 256 + 64 * c + p0, true);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) y[b * ldy + row] = v;
    }
}

template <int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_generic_q6_k(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                      float *__restrict__ y, int64_t ldy) {
    dependent_launch_prologue();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= n_out) return;
    const int nb = k / 256;
    const uint8_t *wr = w + (int64_t)row * nb * 210;
    const int h = lane >> 4, t = (lane & 15) >> 2, l0 = 8 * (lane & 3);
    const int ql_off = 64 * h + l0 + 32 * (t & 1), qh_off = 128 + 32 * h + l0;
    const int nib = (t >= 2) ? 4 : 0, hsh = 2 * t;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll 2
    for (int blk = 0; blk < nb; ++blk) {
        const uint8_t *bp = wr + (int64_t)blk * 210;
        const float d = h2f(ldg_u16(bp + 208));
        const float ds = d * (float)(int)(int8_t)__ldg(bp + 192 + (lane >> 1));
        float wv[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t ql = ldg_u16(bp + ql_off + i), qh = ldg_u16(bp + qh_off + i);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int lo4 = (ql >> (8 * e + nib)) & 15;
                const int hi2 = (qh >> (8 * e + hsh)) & 3;
                wv[i + e] = ds * (float)((lo4 | (hi2 << 4)) - 32);
            }
        }
        fma8<NB>(acc, wv, x, k, (int64_t)blk * 256 + 8 * lane, false);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) y[b * ldy + row] = v;
    }
}

template <int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_generic_q8_0(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                      float *__restrict__ y, int64_t ldy) {
    dependent_launch_prologue();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= n_out) return;
    const int nb = k / 32;
    const uint8_t *wr = w + (int64_t)row * nb * 34;
    const int part = lane & 3;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int g = 0; g < nb; g += 8) {
        const int blk = g + (lane >> 2);
        if (blk < nb) {
            const uint8_t *bp = wr + (int64_t)blk * 34;
            const float d = h2f(ldg_u16(bp));
            float wv[8];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const uint32_t q2 = ldg_u16(bp + 2 + 8 * part + i);
                wv[i] = d * (float)(int8_t)(q2 & 0xff);
                wv[i + 1] = d * (float)(int8_t)(q2 >> 8);
            }
            fma8<NB>(acc, wv, x, k, (int64_t)blk * 32 + 8 * part, false);
        }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) y[b * ldy + row] = v;
    }
}

// Q8_0 rows of at most 32 blocks, k a multiple of 128 (rows then start on
// 8-byte boundaries), with the weights declared static (pq_set_weight_prefetch):
// a call this small is bound by latency.  Each warp reads its row with
// coalesced 8-byte loads before the wait for the previous kernel and parks it
// in shared memory; after the wait only x (an L2 hit) is loaded, lane l takes
// block l (scale and 32 codes) and x's 32 values per column.  The next kernel
// is released after the wait, so exactly one launch ahead is fetching its
// weights while this one computes (released at the start, the blocks of many
// launches ahead fetched theirs at once and the running launch's x loads
// queued behind them: 6.8 us per call).  Q8_0 896x896, CUDA graph of
// back-to-back calls: 3.65 -> 2.39 us.
constexpr int kShortRowBytes = 32 * 34;   // 1088: 32 blocks
template <int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_q8_0_short(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                    float *__restrict__ y, int64_t ldy) {
    __shared__ __align__(16) uint8_t rows[kWarps][kShortRowBytes + 64];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kWarps + warp;
    const int nb = k / 32;
    const int rowbytes = nb * 34;              // a multiple of 8 (nb % 4 == 0)
    if (row < n_out) {
        const uint8_t *wr = w + (int64_t)row * rowbytes;
        uint64_t v[5];
#pragma unroll
        for (int m = 0; m < 5; ++m) {
            const int off = 8 * lane + 256 * m;
            v[m] = off < rowbytes ? __ldg(reinterpret_cast<const unsigned long long *>(wr + off)) : 0ull;
        }
#pragma unroll
        for (int m = 0; m < 5; ++m) {
            const int off = 8 * lane + 256 * m;
            if (off < rowbytes) *reinterpret_cast<uint64_t *>(&rows[warp][off]) = v[m];
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // x may be the previous kernel's output
    asm volatile("griddepcontrol.launch_dependents;");
    if (row >= n_out) return;   // whole warps
    __syncwarp();
    const bool live = lane < nb;
    const uint16_t *blk = reinterpret_cast<const uint16_t *>(&rows[warp][34 * lane]);
    uint32_t dq[17];   // scale bits, then codes 2i, 2i+1 in the two bytes of dq[1 + i]
#pragma unroll
    for (int i = 0; i < 17; ++i) dq[i] = live ? blk[i] : 0u;
    const float d = h2f(dq[0]);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float acc = 0.f;
        if (live) {
            const float *xb = x + (int64_t)b * k + 32 * lane;
            float4 xv[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) xv[m] = ldg_f4(xb + 4 * m);
            const float *xf = reinterpret_cast<const float *>(xv);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                acc = fmaf((float)(int8_t)(dq[1 + i] & 0xffu), xf[2 * i], acc);
                acc = fmaf((float)(int8_t)(dq[1 + i] >> 8), xf[2 * i + 1], acc);
            }
            acc *= d;
        }
        const float v = warp_sum(acc);
        if (lane == 0) y[b * ldy + row] = v;
    }
}

// Q5_K / Q3_K / Q2_K: lane l decodes weights 8l..8l+7 of each super-block
// of the row (pq_kfamily.cuh) and multiplies them by x.
template <int FMT, int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_generic_kfamily(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                         float *__restrict__ y, int64_t ldy) {
    dependent_launch_prologue();
    constexpr int BB = kBlockBytes[FMT];
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= n_out) return;
    const int nb = k / 256;
    const uint8_t *wr = w + (int64_t)row * nb * BB;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll 2
    for (int blk = 0; blk < nb; ++blk) {
        float wv[8];
        kfamily_lane<FMT>(wr + (int64_t)blk * BB, lane, wv);
        fma8<NB>(acc, wv, x, k, (int64_t)blk * 256 + 8 * lane, false);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) y[b * ldy + row] = v;
    }
}

// Per-row int8: lanes stride the row 4 codes at a time when k % 4 == 0
// (row starts are then 4-byte aligned), else one code at a time.
template <int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_generic_i8_row(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                        float *__restrict__ y, int64_t ldy, int64_t soff) {
    dependent_launch_prologue();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= n_out) return;
    const uint8_t *wr = w + (int64_t)row * k;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    if ((k & 3) == 0) {
        for (int i = 4 * lane; i < k; i += 128) {
            const uint32_t q = ldg_u32(wr + i);
            const float q0 = (float)(int8_t)(q & 0xff), q1 = (float)(int8_t)((q >> 8) & 0xff);
            const float q2 = (float)(int8_t)((q >> 16) & 0xff), q3 = (float)(int8_t)(q >> 24);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float4 a = ldg_f4(x + (int64_t)b * k + i);
                acc[b] = fmaf(q0, a.x, acc[b]);
                acc[b] = fmaf(q1, a.y, acc[b]);
                acc[b] = fmaf(q2, a.z, acc[b]);
                acc[b] = fmaf(q3, a.w, acc[b]);
            }
        }
    } else {
        for (int i = lane; i < k; i += 32) {
            const float q = (float)(int8_t)__ldg(wr + i);
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = fmaf(q, __ldg(x + (int64_t)b * k + i), acc[b]);
        }
    }
    const float s = __ldg(reinterpret_cast<const float *>(w + soff) + row);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) y[b * ldy + row] = s * v;
    }
}

// Per-row int4: lanes stride the row 8 codes (one 32-bit word) at a time when
// k % 8 == 0 (row starts are then 4-byte aligned), else 2 codes (one byte).
template <int NB>
__global__ void __launch_bounds__(kThreads)
    gemv_generic_i4_row(const uint8_t *__restrict__ w, int n_out, int k, const float *__restrict__ x,
                        float *__restrict__ y, int64_t ldy, int64_t soff) {
    dependent_launch_prologue();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= n_out) return;
    const uint8_t *wr = w + (int64_t)row * (k / 2);
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    if ((k & 7) == 0) {
        for (int i = 8 * lane; i < k; i += 256) {
            const uint32_t q = ldg_u32(wr + i / 2);
            float wv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) wv[e] = i4_value((q >> (4 * e)) & 15u);
            fma8<NB>(acc, wv, x, k, i, false);
        }
    } else {
        for (int i = 2 * lane; i < k; i += 64) {
            const uint32_t b8 = __ldg(wr + i / 2);
            const float q0 = i4_value(b8 & 15u), q1 = i4_value(b8 >> 4);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                acc[b] = fmaf(q0, __ldg(x + (int64_t)b * k + i), acc[b]);
                acc[b] = fmaf(q1, __ldg(x + (int64_t)b * k + i + 1), acc[b]);
            }
        }
    }
    const float s = __ldg(reinterpret_cast<const float *>(w + soff) + row);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0) y[b * ldy + row] = s * v;
    }
}

template <int NB>
cudaError_t launch_nb(int fmt, const uint8_t *w, int64_t n_out, int64_t k, const float *x,
                      float *y, int64_t ldy, cudaStream_t s, int sm_count) {
    const int grid = (int)((n_out + kWarps - 1) / kWarps);
    const int n = (int)n_out, kk = (int)k;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // overlap with the previous kernel only when every block is resident at
    // once; a larger grid's later blocks would compete with the next kernel's
    // early ones (measured slower: Q8_0 4096 x 4096, 12.4 -> 16.4 us)
    cfg.attrs = attr;
    cfg.numAttrs = grid <= sm_count ? 1 : 0;
    cudaError_t e;
    switch (fmt) {
    case PQ_Q4_K: e = cudaLaunchKernelEx(&cfg, gemv_generic_q4_k<NB>, w, n, kk, x, y, ldy); break;
    case PQ_Q6_K: e = cudaLaunchKernelEx(&cfg, gemv_generic_q6_k<NB>, w, n, kk, x, y, ldy); break;
    case PQ_Q8_0:
        // the short-row kernel reads W before its dependency wait: only for
        // weights declared static, and only as part of a one-wave PDL launch
        e = cfg.numAttrs && weight_prefetch() && kk <= 1024 && kk % 128 == 0 && ((uintptr_t)w & 7) == 0
                ? cudaLaunchKernelEx(&cfg, gemv_q8_0_short<NB>, w, n, kk, x, y, ldy)
                : cudaLaunchKernelEx(&cfg, gemv_generic_q8_0<NB>, w, n, kk, x, y, ldy);
        break;
    case PQ_Q5_K: e = cudaLaunchKernelEx(&cfg, gemv_generic_kfamily<PQ_Q5_K, NB>, w, n, kk, x, y, ldy); break;
    case PQ_Q3_K: e = cudaLaunchKernelEx(&cfg, gemv_generic_kfamily<PQ_Q3_K, NB>, w, n, kk, x, y, ldy); break;
    case PQ_Q2_K: e = cudaLaunchKernelEx(&cfg, gemv_generic_kfamily<PQ_Q2_K, NB>, w, n, kk, x, y, ldy); break;
    case PQ_I8_ROW:
        e = cudaLaunchKernelEx(&cfg, gemv_generic_i8_row<NB>, w, n, kk, x, y, ldy, (int64_t)i8row_scale_offset(n_out, k));
        break;
    case PQ_I4_ROW:
        e = cudaLaunchKernelEx(&cfg, gemv_generic_i4_row<NB>, w, n, kk, x, y, ldy, (int64_t)i4row_scale_offset(n_out, k));
        break;
    default: return cudaErrorInvalidValue;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// x is [batch][k], y is [batch][ldy]; columns are processed 4 at a time.
cudaError_t launch_gemv_generic(int fmt, const uint8_t *w, int64_t n_out, int64_t k,
                                const float *x, int batch, float *y, int64_t ldy,
                                cudaStream_t s, int sm_count) {
    for (int b0 = 0; b0 < batch; b0 += 4) {
        const int nb = batch - b0 < 4 ? batch - b0 : 4;
        const float *xb = x + (int64_t)b0 * k;
        float *yb = y + (int64_t)b0 * ldy;
        cudaError_t e;
        switch (nb) {
        case 1: e = launch_nb<1>(fmt, w, n_out, k, xb, yb, ldy, s, sm_count); break;
        case 2: e = launch_nb<2>(fmt, w, n_out, k, xb, yb, ldy, s, sm_count); break;
        case 3: e = launch_nb<3>(fmt, w, n_out, k, xb, yb, ldy, s, sm_count); break;
        default: e = launch_nb<4>(fmt, w, n_out, k, xb, yb, ldy, s, sm_count); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pqk

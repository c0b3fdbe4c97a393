// pq_dequant kernels: decode every block of W to f32, bit-exact to the
// layout rules (GGUF-style Q8_0 / Q4_K / Q6_K / Q5_K / Q3_K / Q2_K blocks, the
// formats the PESTI README decodes, "What This Is"; per-row int8 and int4 of
// the ember pull request's quant.rs description).
//
// Write-bound: 4 B of output per weight against 0.56-1.06 B read.  One warp
// decodes one super-block (Q4_K, Q6_K) or eight Q8_0 blocks per step, each
// lane producing 8 consecutive weights stored as two 16-byte vectors.  Block
// index gb of the flattened matrix maps to output offset gb*QK because rows
// are contiguous.  All index arithmetic is 64-bit (the 128256 x 4096 head is
// 525 M outputs).
//
// Rounding: every product below is exact in f32 (fp16 d has an 11-bit
// significand, the 6-bit scales/mins and 4/6/8-bit codes are small
// integers); the only rounded step is Q4_K's final subtraction and the
// per-row int8 product, done with explicit _rn intrinsics, so FMA
// contraction cannot change a bit.

#include "pq_device.cuh"
#include "pq_internal.h"

namespace pqk {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void store8(float *o, const float (&v)[8]) {
    reinterpret_cast<float4 *>(o)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(o)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__global__ void __launch_bounds__(kThreads) dequant_q4_k(const uint8_t *__restrict__ w,
                                                         int64_t nblk, float *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    const int c = lane >> 3, p0 = (lane & 7) * 4;
    for (int64_t gb = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); gb < nblk;
         gb += warps) {
        const uint8_t *blk = w + gb * 144;
        const uint32_t dd = ldg_u32(blk);
        const uint32_t s0 = ldg_u32(blk + 4), s1 = ldg_u32(blk + 8), s2 = ldg_u32(blk + 12);
        const uint32_t qs = ldg_u32(blk + 16 + 4 * lane);
        const float d = h2f(dd), dmin = h2f(dd >> 16);
        int sc0, m0, sc1, m1;
        q4k_scale_min(s0, s1, s2, 2 * c, sc0, m0);
        q4k_scale_min(s0, s1, s2, 2 * c + 1, sc1, m1);
        const float dl0 = __fmul_rn(d, (float)sc0), ml0 = __fmul_rn(dmin, (float)m0);
        const float dl1 = __fmul_rn(d, (float)sc1), ml1 = __fmul_rn(dmin, (float)m1);
        float lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t byte = (qs >> (8 * i)) & 0xff;
            lo[i] = __fsub_rn(__fmul_rn(dl0, (float)(byte & 15)), ml0);
            hi[i] = __fsub_rn(__fmul_rn(dl1, (float)(byte >> 4)), ml1);
        }
        float *o = out + gb * 256 + 64 * c + p0;
        reinterpret_cast<float4 *>(o)[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
        reinterpret_cast<float4 *>(o + 32)[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
    }
}

__global__ void __launch_bounds__(kThreads) dequant_q6_k(const uint8_t *__restrict__ w,
                                                         int64_t nblk, float *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    // lane -> weights 8*lane .. 8*lane+7: half h, quarter t, column offset l0
    const int h = lane >> 4, t = (lane & 15) >> 2, l0 = 8 * (lane & 3);
    const int ql_off = 64 * h + l0 + 32 * (t & 1), qh_off = 128 + 32 * h + l0;
    const int nib = (t >= 2) ? 4 : 0, hsh = 2 * t;
    for (int64_t gb = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); gb < nblk;
         gb += warps) {
        const uint8_t *blk = w + gb * 210;
        const float d = h2f(ldg_u16(blk + 208));
        const int sc = (int)(int8_t)__ldg(blk + 192 + (lane >> 1));
        const float ds = __fmul_rn(d, (float)sc);
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t ql = ldg_u16(blk + ql_off + i), qh = ldg_u16(blk + qh_off + i);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int lo4 = (ql >> (8 * e + nib)) & 15;
                const int hi2 = (qh >> (8 * e + hsh)) & 3;
                v[i + e] = __fmul_rn(ds, (float)((lo4 | (hi2 << 4)) - 32));
            }
        }
        store8(out + gb * 256 + 8 * lane, v);
    }
}

__global__ void __launch_bounds__(kThreads) dequant_q8_0(const uint8_t *__restrict__ w,
                                                         int64_t nblk, float *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t groups = (int64_t)gridDim.x * (kThreads / 32);
    const int part = lane & 3;
    for (int64_t g = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); g * 8 < nblk;
         g += groups) {
        const int64_t gb = g * 8 + (lane >> 2);
        if (gb >= nblk) continue;
        const uint8_t *blk = w + gb * 34;
        const float d = h2f(ldg_u16(blk));
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t q2 = ldg_u16(blk + 2 + 8 * part + i);
            v[i] = __fmul_rn(d, (float)(int8_t)(q2 & 0xff));
            v[i + 1] = __fmul_rn(d, (float)(int8_t)(q2 >> 8));
        }
        store8(out + gb * 32 + 8 * part, v);
    }
}

// Q5_K / Q3_K / Q2_K: one warp per super-block, lane l writes weights
// 8l..8l+7 (pq_kfamily.cuh).
template <int FMT>
__global__ void __launch_bounds__(kThreads) dequant_kfamily(const uint8_t *__restrict__ w,
                                                            int64_t nblk, float *__restrict__ out) {
    constexpr int BB = kBlockBytes[FMT];
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t gb = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); gb < nblk;
         gb += warps) {
        float v[8];
        kfamily_lane<FMT>(w + gb * BB, lane, v);
        store8(out + gb * 256 + 8 * lane, v);
    }
}

// Per-row int8, four outputs per thread when k % 4 == 0.
__global__ void __launch_bounds__(kThreads) dequant_i8_row_v4(const uint8_t *__restrict__ w,
                                                              int64_t n_out, int64_t k,
                                                              int64_t soff, float *__restrict__ out) {
    const int64_t n4 = n_out * k / 4;
    const float *scale = reinterpret_cast<const float *>(w + soff);
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < n4;
         t += (int64_t)gridDim.x * kThreads) {
        const int64_t i0 = 4 * t;
        const float s = __ldg(scale + i0 / k);
        const uint32_t q = ldg_u32(w + i0);
        float4 o;
        o.x = __fmul_rn(s, (float)(int8_t)(q & 0xff));
        o.y = __fmul_rn(s, (float)(int8_t)((q >> 8) & 0xff));
        o.z = __fmul_rn(s, (float)(int8_t)((q >> 16) & 0xff));
        o.w = __fmul_rn(s, (float)(int8_t)(q >> 24));
        reinterpret_cast<float4 *>(out)[t] = o;
    }
}

__global__ void __launch_bounds__(kThreads) dequant_i8_row_v1(const uint8_t *__restrict__ w,
                                                              int64_t n_out, int64_t k,
                                                              int64_t soff, float *__restrict__ out) {
    const int64_t n = n_out * k;
    const float *scale = reinterpret_cast<const float *>(w + soff);
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kThreads)
        out[i] = __fmul_rn(__ldg(scale + i / k), (float)(int8_t)__ldg(w + i));
}

// Per-row int4: eight outputs per thread from one 32-bit word when k % 8 == 0
// (rows then start 4-byte aligned and a word never crosses a row), else two
// outputs from one byte (k is even, so a byte never crosses a row).  Weight e
// of a word is its nibble e.
__global__ void __launch_bounds__(kThreads) dequant_i4_row_v8(const uint8_t *__restrict__ w,
                                                              int64_t n_out, int64_t k,
                                                              int64_t soff, float *__restrict__ out) {
    const int64_t n8 = n_out * k / 8;
    const float *scale = reinterpret_cast<const float *>(w + soff);
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < n8;
         t += (int64_t)gridDim.x * kThreads) {
        const int64_t i0 = 8 * t;
        const float s = __ldg(scale + i0 / k);
        const uint32_t q = ldg_u32(w + 4 * t);
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(s, i4_value((q >> (4 * e)) & 15u));
        store8(out + i0, v);
    }
}

__global__ void __launch_bounds__(kThreads) dequant_i4_row_v2(const uint8_t *__restrict__ w,
                                                              int64_t n_out, int64_t k,
                                                              int64_t soff, float *__restrict__ out) {
    const int64_t nq = n_out * k / 2;
    const float *scale = reinterpret_cast<const float *>(w + soff);
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < nq;
         t += (int64_t)gridDim.x * kThreads) {
        const float s = __ldg(scale + 2 * t / k);
        const uint32_t b = __ldg(w + t);
        reinterpret_cast<float2 *>(out)[t] =
            make_float2(__fmul_rn(s, i4_value(b & 15u)), __fmul_rn(s, i4_value(b >> 4)));
    }
}

int grid_for(int64_t work_items, int per_block) {
    int64_t g = (work_items + per_block - 1) / per_block;
    const DeviceInfo *dev = device_info();
    const int64_t cap = (int64_t)(dev ? dev->sm_count : 148) * 16;   // grid-stride beyond this
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_dequant(int fmt, const uint8_t *w, int64_t n_out, int64_t k, float *out,
                           cudaStream_t s) {
    const int wpb = kThreads / 32;
    switch (fmt) {
    case PQ_Q4_K: {
        const int64_t nblk = n_out * (k / 256);
        dequant_q4_k<<<grid_for(nblk, wpb), kThreads, 0, s>>>(w, nblk, out);
        break;
    }
    case PQ_Q6_K: {
        const int64_t nblk = n_out * (k / 256);
        dequant_q6_k<<<grid_for(nblk, wpb), kThreads, 0, s>>>(w, nblk, out);
        break;
    }
    case PQ_Q8_0: {
        const int64_t nblk = n_out * (k / 32);
        dequant_q8_0<<<grid_for((nblk + 7) / 8, wpb), kThreads, 0, s>>>(w, nblk, out);
        break;
    }
    case PQ_Q5_K:
    case PQ_Q3_K:
    case PQ_Q2_K: {
        const int64_t nblk = n_out * (k / 256);
        const int grid = grid_for(nblk, wpb);
        if (fmt == PQ_Q5_K)
            dequant_kfamily<PQ_Q5_K><<<grid, kThreads, 0, s>>>(w, nblk, out);
        else if (fmt == PQ_Q3_K)
            dequant_kfamily<PQ_Q3_K><<<grid, kThreads, 0, s>>>(w, nblk, out);
        else
            dequant_kfamily<PQ_Q2_K><<<grid, kThreads, 0, s>>>(w, nblk, out);
        break;
    }
    case PQ_I4_ROW: {
        const int64_t soff = i4row_scale_offset(n_out, k);
        if (k % 8 == 0)
            dequant_i4_row_v8<<<grid_for(n_out * k / 8, kThreads), kThreads, 0, s>>>(w, n_out, k,
                                                                                    soff, out);
        else
            dequant_i4_row_v2<<<grid_for(n_out * k / 2, kThreads), kThreads, 0, s>>>(w, n_out, k,
                                                                                    soff, out);
        break;
    }
    case PQ_I8_ROW: {
        const int64_t soff = i8row_scale_offset(n_out, k);
        if (k % 4 == 0)
            dequant_i8_row_v4<<<grid_for(n_out * k / 4, kThreads), kThreads, 0, s>>>(w, n_out, k,
                                                                                    soff, out);
        else
            dequant_i8_row_v1<<<grid_for(n_out * k, kThreads), kThreads, 0, s>>>(w, n_out, k,
                                                                                soff, out);
        break;
    }
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pqk

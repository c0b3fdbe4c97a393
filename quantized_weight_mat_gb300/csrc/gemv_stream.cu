// Weight-streaming fused dequant + mat-vec for batch 1..4 on CUDA cores.
//
// The operation is the ember pull request's mat-vec with the decoding of W
// fused into it, so that no f32 copy of W is made (quant.rs description),
// for GGUF-style Q4_K and Q6_K super-blocks (the K family that the PESTI
// README decodes, "What This Is").  At batch 1 it moves 0.5625 B (Q4_K) per weight and does 2
// flops per weight: it is bound by HBM bandwidth, and the design goal is to
// keep HBM busy while spending as few issue slots per weight as possible.
//
// Common structure (one persistent CTA per SM, each owning a contiguous,
// balanced range of rows):
//   * a producer warp streams the CTA's rows through a ring of shared-memory
//     stages with bulk asynchronous copies (cp.async.bulk; completion counted
//     in bytes on an mbarrier per stage, slots handed back on a second one);
//   * x is converted once per CTA into two int8 limbs per element with one
//     scale per 256 values: x ~= u * (254*xh + xl), |error| <= max|x|/64516,
//     so each sub-block's dot product sum_i q_i*x_i becomes dp4a integer dot
//     products (exact);
//   * per super-block the scales and mins are applied in 32-bit integers
//     (H = sum_j sc_j*dot_j over both limbs, M = sum_j m_j*sum X_i), then a
//     few f32 operations: y += u*(d*(254*H + L) - dmin*M) for Q4_K;
//   * partial sums are reduced with warp shuffles (and, for long rows split
//     over several warps, in shared memory in a fixed order).
// No atomics, fixed summation order: results are deterministic.
//
// Three kernels share that structure:
//   rowk::gemv_rows<Q4K|Q6K>  batch 1: a stage is a run of whole rows fetched
//                      with ONE contiguous bulk copy; each lane owns 128
//                      weights (half a super-block) of a fixed k range and
//                      keeps that range of x in registers for the whole kernel;
//   rowsnb::gemv_rows_nb<2>   batch 2, long rows: the same with a lane owning
//                      64 weights, x for both columns in registers, x made
//                      once per call by a small kernel;
//   gemv_stream_q4_k<NB>      batch 1..4, any k: a stage is 32 rows x 8
//                      super-blocks (one copy per row segment), x read from
//                      the shared image per stage and reused across a warp's
//                      rows.
//
// Every mbarrier wait is bounded in time (pq_ptx.cuh); on timeout the
// kernel records it and the warp stops.

#include "pq_device.cuh"
#include "pq_internal.h"
#include "pq_ptx.cuh"

namespace pqk {

namespace {

#ifndef PQ_STREAM_CW
#define PQ_STREAM_CW 8
#endif
#ifndef PQ_STREAM_RPW
#define PQ_STREAM_RPW 4
#endif
constexpr int CW = PQ_STREAM_CW;             // consumer warps
constexpr int RPW = PQ_STREAM_RPW;           // rows per consumer warp per stage
constexpr int TR = CW * RPW;                 // rows per tile (<= 32: one copy per producer lane)
constexpr int KB = 8;                        // super-blocks per row segment
constexpr int SEG = KB * 144;                // bytes per row segment
constexpr int STAGE = TR * SEG;              // bytes per stage
constexpr int MAX_STAGES = 8;
constexpr int THREADS = (CW + 1) * 32;
constexpr int kSmemBudget = 227 * 1024;      // sm_103 opt-in shared memory per block
constexpr int kStaticSmem = 2 * MAX_STAGES * 8;

static_assert(TR <= 32, "one producer lane per row of a tile");
static_assert(SEG % 16 == 0 && STAGE % 128 == 0, "bulk-copy alignment");

struct Params {
    const uint8_t *w;
    const float *x;
    float *y;
    long long ldy;
    int n_out;
    int k;
    int nstages;
};

// Bytes of the per-CTA x image for `nb_cols` columns: two int8 limbs per
// element plus 16 B of metadata per 64-weight slice.
inline int x_image_bytes(int64_t k, int nb_cols) { return (int)(nb_cols * (2 * k + (k / 64) * 16)); }

int plan_stages(int64_t k, int nb_cols) {
    const int64_t avail = kSmemBudget - kStaticSmem - x_image_bytes(k, nb_cols);
    int64_t s = avail / STAGE;
    return (int)(s > MAX_STAGES ? MAX_STAGES : s);
}

// x -> limbs.  Warp per 256-value block q; lane l holds values 8l..8l+7, which
// lie in sub-block j = l/4.  Layout of one column's image (S = k/64 slices,
// slice s = 4q + c covers sub-blocks 2c and 2c+1 of block q):
//   group g (0..7) of slice s at byte (g*S + s)*16:
//     g0,g1: xh of sub-block 2c (values 0-15, 16-31)   g2,g3: xh of sub-block 2c+1
//     g4..g7: the same for xl
//   meta of slice s at byte s*16: {XS_2c, XS_2c+1, u, 0}, XS_j = sum of 254*xh+xl.
// Consecutive lanes read consecutive 16-byte groups: no bank conflicts.
// PERM (the whole-row kernel, whose lane 2j+h reads slices 4j+2h and
// 4j+2h+1): slice s is stored at position (s & 1)*S/2 + s/2 instead, so that
// each of the lane's two reads is again consecutive across lanes.
template <bool PERM = false>
__device__ __forceinline__ void prep_x_vals(const float (&v)[8], uint8_t *img, uint8_t *meta,
                                            int q, int S, int lane) {
    // block maximum of |x|: the bit patterns of non-negative floats order like
    // their values, so one integer warp reduction gives it
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mb = max(mb, __float_as_uint(v[i]) & 0x7fffffffu);
    mb = __reduce_max_sync(0xffffffffu, mb);
    const float amax = __uint_as_float(mb);
    const float s = amax * (1.0f / 127.0f);
    // one reciprocal for both scales (a block whose values are all below 1e-30
    // contributes nothing measurable and gets zero limbs)
    const float rcp = amax > 1e-30f ? __frcp_rn(amax) : 0.f;
    const float inv = 127.0f * rcp, inv2 = (254.0f * 127.0f) * rcp;
    // Round to nearest even by adding 1.5 * 2^23: for |t| < 2^22 the sum is
    // exact and its bit pattern is 0x4B400000 + t, so the low byte of the bits
    // is t as a two's-complement byte, ready to pack.  |x*inv| <= 127 by
    // construction; the remainder r obeys |r| <= s/2 up to a relative 3e-5, so
    // |r*inv2| <= 127.01 also rounds into [-127, 127].
    constexpr float kMagic = 12582912.0f;
    uint32_t th[8], tl[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float t = fmaf(v[i], inv, kMagic);
        const float r = fmaf(-s, t - kMagic, v[i]);
        th[i] = __float_as_uint(t);
        tl[i] = __float_as_uint(fmaf(r, inv2, kMagic));
    }
    // low bytes of four words -> one word, value i in byte i
    auto pack4 = [](uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
        return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
    };
    const uint32_t h0 = pack4(th[0], th[1], th[2], th[3]), h1 = pack4(th[4], th[5], th[6], th[7]);
    const uint32_t l0 = pack4(tl[0], tl[1], tl[2], tl[3]), l1 = pack4(tl[4], tl[5], tl[6], tl[7]);
    // sum of 254*xh + xl over the lane's eight values (signed bytes times one)
    int xs = 254 * dp4a_ss(h0, 0x01010101u, dp4a_ss(h1, 0x01010101u, 0)) +
             dp4a_ss(l0, 0x01010101u, dp4a_ss(l1, 0x01010101u, 0));
    xs += __shfl_xor_sync(0xffffffffu, xs, 1);
    xs += __shfl_xor_sync(0xffffffffu, xs, 2);
    const int j = lane >> 2, c = j >> 1, half = j & 1;
    const int slice = PERM ? (c & 1) * (S >> 1) + 2 * q + (c >> 1) : 4 * q + c;
    const int g = 2 * half + ((lane & 3) >> 1);
    const int off8 = 8 * (lane & 1);
    *reinterpret_cast<uint2 *>(img + (g * S + slice) * 16 + off8) = make_uint2(h0, h1);
    *reinterpret_cast<uint2 *>(img + ((g + 4) * S + slice) * 16 + off8) = make_uint2(l0, l1);
    if ((lane & 3) == 0) *reinterpret_cast<int *>(meta + slice * 16 + 4 * half) = xs;
    if ((lane & 7) == 0) *reinterpret_cast<float *>(meta + slice * 16 + 8) = s * (1.0f / 254.0f);
}

__device__ __forceinline__ void prep_x_block(const float *xb, uint8_t *img, uint8_t *meta, int q,
                                             int S, int lane) {
    const float4 a = ldg_f4(xb + q * 256 + 8 * lane);
    const float4 b = ldg_f4(xb + q * 256 + 8 * lane + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    prep_x_vals(v, img, meta, q, S, lane);
}

// The x image of one column, blocks q = first, first+step, ...: the loads of
// up to eight blocks are in flight before any of them is converted.  x is
// read from global memory, or (FROM_SMEM) from a shared-memory copy; a null
// xb stands for a column of zeros.
template <bool FROM_SMEM = false, bool PERM = false>
__device__ __forceinline__ void prep_x_all(const float *xb, uint8_t *img, uint8_t *meta, int nb,
                                           int S, int first, int step, int lane) {
    for (int q0 = first; q0 < nb; q0 += 8 * step) {
        float v[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int q = q0 + r * step;
            if (q < nb) {
                const float *xq = xb + q * 256 + 8 * lane;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;   // a null xb is a zero column
                if (xb) {
                    a = FROM_SMEM ? *reinterpret_cast<const float4 *>(xq) : ldg_f4(xq);
                    b = FROM_SMEM ? *reinterpret_cast<const float4 *>(xq + 4) : ldg_f4(xq + 4);
                }
                v[r][0] = a.x; v[r][1] = a.y; v[r][2] = a.z; v[r][3] = a.w;
                v[r][4] = b.x; v[r][5] = b.y; v[r][6] = b.z; v[r][7] = b.w;
            }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int q = q0 + r * step;
            if (q < nb) prep_x_vals<PERM>(v[r], img, meta, q, S, lane);
        }
    }
}

template <int NB>
__global__ void __launch_bounds__(THREADS, 1) gemv_stream_q4_k(Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int nchunks = (nb + KB - 1) / KB;
    const int S = p.k / 64;
    const int64_t rowbytes = (int64_t)nb * 144;
    const int64_t r0 = (int64_t)p.n_out * blockIdx.x / gridDim.x;
    const int64_t r1 = (int64_t)p.n_out * (blockIdx.x + 1) / gridDim.x;
    const int ntiles = (int)((r1 - r0 + TR - 1) / TR);
    const int units = ntiles * nchunks;
    const int NS = p.nstages;
    uint8_t *ring = smem;
    uint8_t *ximg = smem + NS * STAGE;
    uint8_t *xmeta = ximg + NB * 2 * p.k;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ---------------- producer ----------------
        const uint64_t pol = make_evict_first_policy();
        int slot = 0, tile = 0, ch = 0;
        uint32_t ph = 0;
        for (int u = 0; u < units; ++u) {
            const int64_t row0 = r0 + (int64_t)tile * TR;
            const int rows = (int)(r1 - row0 < TR ? r1 - row0 : TR);
            const int kbc = nb - ch * KB < KB ? nb - ch * KB : KB;
            const uint32_t bytes = (uint32_t)kbc * 144u;
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(&empty_bar[slot], ph ^ 1u);
                if (ok) mbar_arrive_expect_tx(&full_bar[slot], bytes * (uint32_t)rows);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane < rows) {
                const uint8_t *src = p.w + (row0 + lane) * rowbytes + (int64_t)ch * SEG;
                bulk_g2s_hint(ring + slot * STAGE + lane * SEG, src, bytes, &full_bar[slot], pol);
            }
            if (++slot == NS) { slot = 0; ph ^= 1u; }
            if (++ch == nchunks) { ch = 0; ++tile; }
        }
        return;
    }

    // ---------------- consumers: x image ----------------
    for (int b = 0; b < NB; ++b) {
        const float *xb = p.x + (int64_t)b * p.k;
        for (int q = warp; q < nb; q += CW)
            prep_x_block(xb, ximg + b * 2 * p.k, xmeta + b * S * 16, q, S, lane);
    }
    named_sync(1, CW * 32);

    // ---------------- consumers: main loop ----------------
    const int bl = lane >> 2, c = lane & 3;
    // byte selectors: bytes 2c', 2c'+1 (c' = c & 1) of scale words 0 and 1, and of word 2
    const uint32_t c2 = 2u * (uint32_t)(c & 1);
    const uint32_t selP = c2 | ((c2 + 1) << 4) | ((c2 + 4) << 8) | ((c2 + 5) << 12);
    const uint32_t selQ = c2 | ((c2 + 1) << 4) | (c2 << 8) | ((c2 + 1) << 12);
    float acc[RPW][NB];
#pragma unroll
    for (int t = 0; t < RPW; ++t)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[t][b] = 0.f;

    int slot = 0, tile = 0, ch = 0;
    uint32_t ph = 0;
    for (int u = 0; u < units; ++u) {
        const int64_t row0 = r0 + (int64_t)tile * TR;
        const int rows = (int)(r1 - row0 < TR ? r1 - row0 : TR);
        const int kbc = nb - ch * KB < KB ? nb - ch * KB : KB;
        if (!mbar_wait(&full_bar[slot], ph)) break;
        const bool active = bl < kbc;
        const uint8_t *stage = ring + slot * STAGE;

        uint32_t lo[RPW][8], hi[RPW][8];
        int sc0x16[RPW], sc1[RPW], m0[RPW], m1[RPW];
        float d16[RPW], dmin[RPW];
        bool live[RPW];
#pragma unroll
        for (int t = 0; t < RPW; ++t) {
            const int trow = warp * RPW + t;
            live[t] = active && trow < rows;
            uint4 hd = make_uint4(0, 0, 0, 0), qa = hd, qb = hd;
            if (live[t]) {
                const uint8_t *blk = stage + trow * SEG + bl * 144;
                hd = *reinterpret_cast<const uint4 *>(blk);
                qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
                qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
            }
            const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lo[t][i] = qw[i] & 0x0F0F0F0Fu;
                hi[t][i] = qw[i] & 0xF0F0F0F0u;   // 16*q: rescaled by d/16 below
            }
            // (sc, m) of sub-blocks 2c and 2c+1 as bytes {sc0, sc1, m0, m1}
            const uint32_t P = __byte_perm(hd.y, hd.z, selP);
            uint32_t r4;
            if (c < 2) {
                r4 = P & 0x3F3F3F3Fu;
            } else {
                const uint32_t Q = __byte_perm(hd.w, 0u, selQ);
                r4 = ((P >> 2) & 0x30303030u) | (Q & 0x00000F0Fu) | ((Q >> 4) & 0x0F0F0000u);
            }
            sc0x16[t] = (int)((r4 << 4) & 0xFF0u);
            sc1[t] = (int)((r4 >> 8) & 0xFFu);
            m0[t] = (int)((r4 >> 16) & 0xFFu);
            m1[t] = (int)(r4 >> 24);
            d16[t] = h2f(hd.x) * 0.0625f;
            dmin[t] = h2f(hd.x >> 16);
        }

        if (active) {
            const int slice = ch * (4 * KB) + lane;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint8_t *img = ximg + b * 2 * p.k;
                uint4 g[8];
#pragma unroll
                for (int gi = 0; gi < 8; ++gi)
                    g[gi] = *reinterpret_cast<const uint4 *>(img + (gi * S + slice) * 16);
                const int4 mt = *reinterpret_cast<const int4 *>(xmeta + b * S * 16 + slice * 16);
                const float ub = __int_as_float(mt.z);
                const uint32_t xh0[8] = {g[0].x, g[0].y, g[0].z, g[0].w, g[1].x, g[1].y, g[1].z, g[1].w};
                const uint32_t xh1[8] = {g[2].x, g[2].y, g[2].z, g[2].w, g[3].x, g[3].y, g[3].z, g[3].w};
                const uint32_t xl0[8] = {g[4].x, g[4].y, g[4].z, g[4].w, g[5].x, g[5].y, g[5].z, g[5].w};
                const uint32_t xl1[8] = {g[6].x, g[6].y, g[6].z, g[6].w, g[7].x, g[7].y, g[7].z, g[7].w};
#pragma unroll
                for (int t = 0; t < RPW; ++t) {
                    if (!live[t]) continue;
                    int dh0 = 0, dh1 = 0, dl0 = 0, dl1 = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        dh0 = dp4a_ss(lo[t][i], xh0[i], dh0);
                        dl0 = dp4a_ss(lo[t][i], xl0[i], dl0);
                        dh1 = dp4a_us(hi[t][i], xh1[i], dh1);
                        dl1 = dp4a_us(hi[t][i], xl1[i], dl1);
                    }
                    const int H = sc0x16[t] * dh0 + sc1[t] * dh1;
                    const int L = sc0x16[t] * dl0 + sc1[t] * dl1;
                    const int M = m0[t] * mt.x + m1[t] * mt.y;
                    const float val = d16[t] * fmaf(254.0f, (float)H, (float)L) - dmin[t] * (float)M;
                    acc[t][b] = fmaf(ub, val, acc[t][b]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);

        if (ch == nchunks - 1) {
#pragma unroll
            for (int t = 0; t < RPW; ++t) {
                const int trow = warp * RPW + t;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float v = warp_sum(acc[t][b]);
                    if (lane == 0 && trow < rows) p.y[b * p.ldy + row0 + trow] = v;
                    acc[t][b] = 0.f;
                }
            }
        }
        if (++slot == NS) { slot = 0; ph ^= 1u; }
        if (++ch == nchunks) { ch = 0; ++tile; }
    }
}

template <int NB>
cudaError_t launch_nb(const Params &p0, int grid, cudaStream_t s) {
    Params p = p0;
    p.nstages = plan_stages(p.k, NB);
    const int smem = p.nstages * STAGE + x_image_bytes(p.k, NB);
    static PerDeviceOnce configured;
    const cudaError_t ce = configured.run([] {
        return cudaFuncSetAttribute(gemv_stream_q4_k<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBudget - kStaticSmem);
    });
    if (ce != cudaSuccess) return ce;
    gemv_stream_q4_k<NB><<<grid, THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Batch-1 kernel with whole-row stages.
//
// A row of nb super-blocks is split into G = ceil(nb/16) segments of 16
// super-blocks (4096 weights); a "row group" of G warps handles a row, warp
// seg of the group owning segment seg for every row of the kernel.  Lane l of
// a warp owns super-block seg*16 + l/2 and its half l%2 (chunks 2h, 2h+1 =
// sub-blocks 4h..4h+3, 128 weights): its x limbs (64 registers) and sub-block
// sums are loaded once.  NG = CW/G row groups share a stage of RS = 2*NG
// consecutive rows, fetched with a single bulk copy; group gi takes rows gi
// and gi+NG of a stage, two stages per loop iteration, and reduces those four
// rows with one transposed shuffle tree.  With G > 1 the per-warp partials
// of a row are kept in shared memory and summed in segment order at the end.
//
// Launched with programmatic dependent launch: the CTA lets the next kernel
// on the stream start as soon as it is resident, and waits for the previous
// kernel (griddepcontrol.wait) before reading x -- and before reading the
// weights too, unless the caller has declared weights static
// (pq_set_weight_prefetch), in which case the producer starts streaming them
// while the previous kernel finishes.
//
// x is read with ordinary loads by the consumer warps as soon as that wait
// returns.  Data requested by an SM returns roughly in request order, so a
// load of x issued behind the whole ring's worth of weight copies would wait
// for all of them (several microseconds at this SM's share of the HBM
// bandwidth).  Until the consumers have converted x, the producer therefore
// keeps at most a window of stages in flight (issued, not landed); after that
// only the ring depth limits it.  Measured per-CTA timelines (%globaltimer)
// of 14336x4096 launched back to back: x ready 2.8 us after the wait returned
// with the whole ring in flight ahead of it, about 1.2 us with a window of
// two stages; per launch 8.15 -> 7.12 us (7.4 us with 3, 7.9 us with 4).  The
// producer polls the consumers' signal with mbarrier.test_wait: try_wait may
// suspend the thread, which delayed the first weight copies.
//
// The ring (three to five stages) cannot hold a CTA's rows, and between the
// release and the first dot product (release latency, x conversion, the x
// limbs loaded into registers: about 2.4 us) HBM would idle once the window
// has landed.  So, for rows of one warp segment (k <= 4096), the producer
// also asks L2 to prefetch 40 % of the CTA's remaining rows, at most
// kL2PrefetchBytes (cp.async.bulk.prefetch.L2), right after issuing the
// window: HBM keeps streaming into L2 through that time, no shared memory is
// held, and no data comes back to the SM ahead of x; the next stage copies
// then hit L2.  Prefetching all the remaining rows front-loads HBM at the
// moment the x loads and the last-started CTAs' first copies need it
// (14336x4096: 6.65 us with all of them, 6.67 with 30 %, 6.40 with 40 %,
// 6.47 with 50 %; 28672x4096 and the Q6_K head meet the byte cap either way).  With
// the prefetch a window of one stage is best unless the CTA has many stages
// (kWideWindowUnits).  Q4_K, launched back to back: 14336x4096 7.01 -> 6.73
// us, 28672x4096 11.14 -> 10.07 us, decode-layer set 29.0 -> 28.1 us.
// Prefetching for longer rows as well made the set slower (28.7 us).  SwiGLU
// stages read gate and up rows from two regions; the budget is split
// between them (fused gate+up 12.2 -> 10.7 us against 128 KB each).
//
// Consumer warps per CTA are a property of the format (kWarps): 12 where a
// 24-row stage still leaves at least three ring slots and the decode is
// heavy enough for the extra warps to pay (Q4_K, Q3_K, Q2_K: decode-layer
// set 29.8 -> 29.0 us, 4096x14336 8.4 -> 8.2 us), 8 where 24-row stages
// would leave two slots (Q6_K 14336x4096: 9.7 us with 8 warps, 11.2 with 12).
#ifndef PQ_ROWS_MINB
#define PQ_ROWS_MINB 1
#endif
namespace rowk {
constexpr int MINB = PQ_ROWS_MINB;           // CTAs per SM the kernel is sized for
constexpr int kRowsSmem = MINB == 1 ? kSmemBudget : (228 * 1024) / MINB - 1024;
constexpr int KW = 16;                       // super-blocks per warp segment
constexpr int RPG = 2;                       // rows per row group per stage
constexpr int MAX_STAGES = 8;
// consumer warps + the producer warp
template <int CW> constexpr int threads_for() { return (CW + 1) * 32; }
constexpr int kStatic = 512;                 // reserve for the kernel's static shared memory (barriers)
constexpr int kXWindow = 2;                  // stages in flight at most until x is converted
constexpr int kWideWindowUnits = 8;          // ... for CTAs with at least this many stages; one stage below
constexpr uint32_t kL2PrefetchBytes = 128 * 1024;   // rows prefetched into L2 after the window (one segment)
constexpr uint32_t kL2PrefetchBytesLong = 64 * 1024; // ... rows of several segments (k > 4096)
constexpr uint64_t kL2PrefetchPercent = 40;         // ... as a share of the CTA's remaining rows

struct Params {
    const uint8_t *w;
    const float *x;
    float *y;
    int n_out;
    int k;
    int G;          // warps per row
    int NG;         // row groups
    int RS;         // rows per stage
    int nstages;
    int rows_cap;   // max rows of one CTA (partials buffer, G > 1)
    int early_w;    // stream weights before waiting on the previous kernel
    int n_ff;       // SwiGLU: pairs (the matrix has 2 * n_ff rows, gate rows first)
    const float *bias;   // bias epilogue: bias[n_out]
    const float *rscale; // per-row formats: the f32 row scales, rscale[n_out]
    int epi;        // kEpiNone, kEpiBias or kEpiSwiGLU
};

inline int segments(int64_t k) { return (int)((k / 256 + KW - 1) / KW); }

__host__ __device__ inline int red_bytes(const Params &p) { return p.G > 1 ? (p.rows_cap * p.G * 4 + 15) / 16 * 16 : 0; }
// Row scales of a per-row format, copied to shared memory once per CTA (for
// SwiGLU the gate and the up rows' scales of every pair), then the CTA's
// slice of the bias for the bias epilogue.
__host__ __device__ inline int rsc_bytes(const Params &p, bool row_scaled, bool swiglu) {
    return row_scaled ? ((swiglu ? 2 : 1) * p.rows_cap * 4 + 15) / 16 * 16 : 0;
}
inline int bias_bytes(const Params &p, bool bias) { return bias ? (p.rows_cap * 4 + 15) / 16 * 16 : 0; }

// Stage plan for (k, n_out, grid) with super-blocks of `block_bytes`; false
// when this kernel cannot take the shape (rows must be whole multiples of
// 16 bytes for the bulk copy).
// With `swiglu` the CTA's items are (gate, up) row pairs: a stage holds NG
// gate rows, then the NG up rows of the same pairs, and n_out is 2 * pairs.
inline bool plan(int64_t k, int64_t n_out, int grid, int block_bytes, int CW, Params &p, bool swiglu = false,
                 bool row_scaled = false, bool bias = false) {
    if (k % 256 || grid < 1 || ((k / 256) * block_bytes) % 16) return false;
    const int G = segments(k);
    if (G < 1 || G > CW) return false;
    p.G = G;
    p.NG = CW / G;
    p.RS = RPG * p.NG;
    if (swiglu) {
        const int64_t pairs_cap = (n_out / 2 + grid - 1) / grid;
        p.rows_cap = (int)((pairs_cap + p.NG - 1) / p.NG * p.RS);   // stage-relative rows
    } else {
        p.rows_cap = (int)((n_out + grid - 1) / grid);
    }
    const int64_t stage = (int64_t)p.RS * (k / 256) * block_bytes;
    const int64_t avail = kRowsSmem - kStatic - x_image_bytes(k, 1) - red_bytes(p) - rsc_bytes(p, row_scaled, swiglu) -
                          bias_bytes(p, bias);
    int64_t ns = avail / stage;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    p.nstages = (int)ns;
    return ns >= 2;
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ uint4 lds(uint32_t a) { return lds128(a); }
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ int byte_of(uint32_t v, int i) {
    return (int)__byte_perm(v, 0u, 0x4440u | (uint32_t)i);
}
// byte i of v as a signed value
__device__ __forceinline__ int sbyte_of(uint32_t v, int i) { return (int)(int8_t)(v >> (8 * i)); }

// The lane's 64 x limb words from the x image (PERM layout): chunks 2h, 2h+1
// of super-block kbc (slices 4kbc+2h, 4kbc+2h+1).  part[0..3] = the four runs
// of 32 positions, in order; meta gives the 32-position sums and the scale u.
__device__ __forceinline__ void load_x_parts(uint32_t (&xh)[4][8], uint32_t (&xl)[4][8], int (&xs32)[4],
                                             float &u, const uint8_t *ximg, const uint8_t *xmeta,
                                             int S, int kbc, int hf) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int slice = cc * (S >> 1) + 2 * kbc + hf;   // slice 4kbc + 2hf + cc, permuted
        uint4 g[8];
#pragma unroll
        for (int gi2 = 0; gi2 < 8; ++gi2)
            g[gi2] = *reinterpret_cast<const uint4 *>(ximg + (gi2 * S + slice) * 16);
        const uint32_t *gw = reinterpret_cast<const uint32_t *>(g);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xh[2 * cc][i] = gw[i];
            xh[2 * cc + 1][i] = gw[8 + i];
            xl[2 * cc][i] = gw[16 + i];
            xl[2 * cc + 1][i] = gw[24 + i];
        }
        const int4 mt = *reinterpret_cast<const int4 *>(xmeta + slice * 16);
        xs32[2 * cc] = mt.x;
        xs32[2 * cc + 1] = mt.y;
        u = __int_as_float(mt.z);
    }
}

// ---------------------------------------------------------------------------
// Q4_K: lane owns sub-blocks 4h..4h+3 (chunks 2h, 2h+1) of its super-block.
struct Q4K {
    static int64_t scale_offset(int64_t, int64_t) { return 0; }
    static constexpr int kBlockBytes = 144;
    static constexpr bool kRowScaled = false;
    static constexpr int kWarps = 12;
    struct X {
        uint32_t xh[4][8], xl[4][8];   // limbs of the 4 sub-blocks (32 positions each)
        int xs[4];                     // sum of X = 254*xh + xl per sub-block
        float u;                       // x ~= u * X
        uint32_t mA, mB, qoff;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t) {
        load_x_parts(R.xh, R.xl, R.xs, R.u, ximg, xmeta, S, kbc, hf);
        if (!valid) R.u = 0.f;
        R.mA = hf ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
        R.mB = hf ? 0x30303030u : 0u;
        R.qoff = 16u + 64u * (uint32_t)hf;
    }
    // Partial dot product of this lane's 128 weights of the row whose
    // super-block starts at shared address blk.
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint4 hd = lds(blk);
        const uint4 qa = lds(blk + R.qoff), qb = lds(blk + R.qoff + 16);
        const uint4 qc = lds(blk + R.qoff + 32), qd = lds(blk + R.qoff + 48);
        const uint32_t w0[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const uint32_t w1[8] = {qc.x, qc.y, qc.z, qc.w, qd.x, qd.y, qd.z, qd.w};
        // packed 6-bit scales / mins of sub-blocks 4h..4h+3, one per byte
        const uint32_t sc4 = ((hf ? hd.w : hd.y) & R.mA) | ((hd.y >> 2) & R.mB);
        const uint32_t m4 = ((hf ? (hd.w >> 4) : hd.z) & R.mA) | ((hd.z >> 2) & R.mB);
        int dh0 = 0, dl0 = 0, dh1 = 0, dl1 = 0, dh2 = 0, dl2 = 0, dh3 = 0, dl3 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo0 = w0[i] & 0x0F0F0F0Fu, hi0 = w0[i] & 0xF0F0F0F0u;
            const uint32_t lo1 = w1[i] & 0x0F0F0F0Fu, hi1 = w1[i] & 0xF0F0F0F0u;
            dh0 = dp4a_ss(lo0, R.xh[0][i], dh0);
            dl0 = dp4a_ss(lo0, R.xl[0][i], dl0);
            dh1 = dp4a_us(hi0, R.xh[1][i], dh1);
            dl1 = dp4a_us(hi0, R.xl[1][i], dl1);
            dh2 = dp4a_ss(lo1, R.xh[2][i], dh2);
            dl2 = dp4a_ss(lo1, R.xl[2][i], dl2);
            dh3 = dp4a_us(hi1, R.xh[3][i], dh3);
            dl3 = dp4a_us(hi1, R.xl[3][i], dl3);
        }
        // even sub-blocks pair with low nibbles (x1), odd ones with high nibbles (x16)
        const int s0 = byte_of(sc4, 0) << 4, s1 = byte_of(sc4, 1);
        const int s2 = byte_of(sc4, 2) << 4, s3 = byte_of(sc4, 3);
        const int H = s0 * dh0 + s1 * dh1 + s2 * dh2 + s3 * dh3;        // |H| < 2^28
        const int L = s0 * dl0 + s1 * dl1 + s2 * dl2 + s3 * dl3;
        const int M = byte_of(m4, 0) * R.xs[0] + byte_of(m4, 1) * R.xs[1] +
                      byte_of(m4, 2) * R.xs[2] + byte_of(m4, 3) * R.xs[3];    // |M| < 2^28
        const float d = h2f(hd.x) * 0.0625f, dmin = h2f(hd.x >> 16);
        return R.u * (d * fmaf(254.0f, (float)H, (float)L) - dmin * (float)M);
    }
};

// ---------------------------------------------------------------------------
// Q6_K: lane owns half h of its super-block (weights 128h..128h+127): ql bytes
// 64h..64h+63, qh bytes 32h..32h+31, scales 8h..8h+7.  Blocks are 210 bytes,
// so a block may start 2 bytes past a 4-byte boundary: the lane loads aligned
// words and realigns them with one byte permute each (selector fixed per lane,
// since row and stage sizes are multiples of 16 bytes).
struct Q6K {
    static int64_t scale_offset(int64_t, int64_t) { return 0; }
    static constexpr int kBlockBytes = 210;
    static constexpr bool kRowScaled = false;
    static constexpr int kWarps = 8;
    struct X {
        uint32_t xh[4][8], xl[4][8];   // limbs of the four 32-position parts t = 0..3
        int xs[8];                     // sum of X over the 8 sub-blocks of 16
        float u;
        uint32_t delta, sel, dsh;      // misalignment (0/2), realign selector, d shift
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t lane_base) {
        int xs32[4];
        load_x_parts(R.xh, R.xl, xs32, R.u, ximg, xmeta, S, kbc, hf);
#pragma unroll
        for (int sb = 0; sb < 8; ++sb) {
            int sh = 0, sl = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sh = dp4a_ss(R.xh[sb >> 1][4 * (sb & 1) + i], 0x01010101u, sh);
                sl = dp4a_ss(R.xl[sb >> 1][4 * (sb & 1) + i], 0x01010101u, sl);
            }
            R.xs[sb] = 254 * sh + sl;
        }
        if (!valid) R.u = 0.f;
        R.delta = lane_base & 2u;
        R.sel = R.delta ? 0x5432u : 0x3210u;
        R.dsh = R.delta ? 16u : 0u;
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint32_t a = blk - R.delta;
        uint32_t ql[16], qh[8], scw[2];
        {
            uint32_t w[17];
#pragma unroll
            for (int j = 0; j < 17; ++j) w[j] = lds32(a + 64u * (uint32_t)hf + 4u * (uint32_t)j);
#pragma unroll
            for (int j = 0; j < 16; ++j) ql[j] = __byte_perm(w[j], w[j + 1], R.sel);
        }
        {
            uint32_t w[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) w[j] = lds32(a + 128u + 32u * (uint32_t)hf + 4u * (uint32_t)j);
#pragma unroll
            for (int j = 0; j < 8; ++j) qh[j] = __byte_perm(w[j], w[j + 1], R.sel);
        }
        {
            uint32_t w[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) w[j] = lds32(a + 192u + 8u * (uint32_t)hf + 4u * (uint32_t)j);
            scw[0] = __byte_perm(w[0], w[1], R.sel);
            scw[1] = __byte_perm(w[1], w[2], R.sel);
        }
        const uint32_t dw = lds32(a + 208u) >> R.dsh;
        // 6-bit codes (0..63) of the four parts, four positions per word;
        // sub-block of part t, word i: 2t + i/4
        int dh[8], dl[8];
#pragma unroll
        for (int sb = 0; sb < 8; ++sb) dh[sb] = dl[sb] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t la = ql[i], lb = ql[8 + i], h = qh[i];
            const uint32_t q0 = (la & 0x0F0F0F0Fu) | ((h << 4) & 0x30303030u);
            const uint32_t q1 = (lb & 0x0F0F0F0Fu) | ((h << 2) & 0x30303030u);
            const uint32_t q2 = ((la >> 4) & 0x0F0F0F0Fu) | (h & 0x30303030u);
            const uint32_t q3 = ((lb >> 4) & 0x0F0F0F0Fu) | ((h >> 2) & 0x30303030u);
            const int s = i >> 2;
            dh[0 + s] = dp4a_us(q0, R.xh[0][i], dh[0 + s]);
            dl[0 + s] = dp4a_us(q0, R.xl[0][i], dl[0 + s]);
            dh[2 + s] = dp4a_us(q1, R.xh[1][i], dh[2 + s]);
            dl[2 + s] = dp4a_us(q1, R.xl[1][i], dl[2 + s]);
            dh[4 + s] = dp4a_us(q2, R.xh[2][i], dh[4 + s]);
            dl[4 + s] = dp4a_us(q2, R.xl[2][i], dl[4 + s]);
            dh[6 + s] = dp4a_us(q3, R.xh[3][i], dh[6 + s]);
            dl[6 + s] = dp4a_us(q3, R.xl[3][i], dl[6 + s]);
        }
        // signed sub-block scales; |H|, |L| < 2^28, |M| < 2^30
        int H = 0, L = 0, M = 0;
#pragma unroll
        for (int sb = 0; sb < 8; ++sb) {
            const int sc = sbyte_of(scw[sb >> 2], sb & 3);
            H += sc * dh[sb];
            L += sc * dl[sb];
            M += sc * R.xs[sb];
        }
        const float d = h2f(dw);
        return R.u * d * (fmaf(254.0f, (float)H, (float)L) - 32.0f * (float)M);
    }
};

// ---------------------------------------------------------------------------
// Q8_0: eight 34-byte blocks (d, 32 int8 codes) make one 272-byte group of 256
// weights; the lane owns blocks 4h..4h+3 of its group (136 bytes at an 8-byte
// boundary).  Blocks 4h and 4h+2 start 2 bytes past a word boundary, so their
// codes are realigned with one byte permute per word.
struct Q80 {
    static int64_t scale_offset(int64_t, int64_t) { return 0; }
    static constexpr int kBlockBytes = 272;
    static constexpr bool kRowScaled = false;
    static constexpr int kWarps = 8;
    struct X {
        uint32_t xh[4][8], xl[4][8];   // limbs of the four 32-weight blocks
        float u;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t) {
        int xs32[4];
        load_x_parts(R.xh, R.xl, xs32, R.u, ximg, xmeta, S, kbc, hf);
        if (!valid) R.u = 0.f;
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint32_t a = blk + 136u * (uint32_t)hf;
        uint32_t w[34];
#pragma unroll
        for (int j = 0; j < 17; ++j) {
            uint2 v;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a + 8u * (uint32_t)j));
            w[2 * j] = v.x;
            w[2 * j + 1] = v.y;
        }
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            // block t at byte 34t of the lane's range: d, then 32 codes
            const int wd = (34 * t) / 4;              // word holding d
            const bool odd = (t & 1) != 0;            // d in the high half, codes word-aligned
            const uint32_t dbits = odd ? (w[wd] >> 16) : w[wd];
            int dh = 0, dl = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t q = odd ? w[wd + 1 + i] : __byte_perm(w[wd + i], w[wd + i + 1], 0x5432u);
                dh = dp4a_ss(q, R.xh[t][i], dh);
                dl = dp4a_ss(q, R.xl[t][i], dl);
            }
            // |254 dh + dl| < 2^28: exact in 32-bit integers
            acc = fmaf(h2f(dbits), (float)(254 * dh + dl), acc);
        }
        return R.u * acc;
    }
};

// ---------------------------------------------------------------------------
// Per-row int8: a row is k int8 codes; the lane owns 128 codes (16-byte
// aligned) of its 256-weight group.  Lanes' ranges are 128 bytes apart, so
// all of them would read the same shared-memory banks at each step: lane l
// reads its eight 16-byte chunks in the rotated order c' = (c + l) mod 8, with
// its x limbs loaded in the same order.  The row's f32 scale multiplies the
// reduced sum.
struct I8R {
    static constexpr int kBlockBytes = 256;
    static constexpr bool kRowScaled = true;
    static constexpr int kWarps = 8;
    static int64_t scale_offset(int64_t n_out, int64_t k) { return i8row_scale_offset(n_out, k); }
    struct X {
        uint32_t xh[8][4], xl[8][4];   // limbs of chunk (c + lane) mod 8, 16 positions each
        float u;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t) {
        uint32_t xh[4][8], xl[4][8];
        int xs32[4];
        load_x_parts(xh, xl, xs32, R.u, ximg, xmeta, S, kbc, hf);
        if (!valid) R.u = 0.f;
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int m = (c + lane) & 7;          // chunk m: part m/2, words 4(m%2)..4(m%2)+3
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // select without dynamic register indexing
                uint32_t h = 0, l = 0;
#pragma unroll
                for (int mm = 0; mm < 8; ++mm)
                    if (mm == m) { h = xh[mm >> 1][4 * (mm & 1) + i]; l = xl[mm >> 1][4 * (mm & 1) + i]; }
                R.xh[c][i] = h;
                R.xl[c][i] = l;
            }
        }
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint32_t a = blk + 128u * (uint32_t)hf;
        const uint32_t lane = threadIdx.x & 31u;
        int dh = 0, dl = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 q = lds(a + 16u * ((c + lane) & 7u));
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dh = dp4a_ss(qw[i], R.xh[c][i], dh);
                dl = dp4a_ss(qw[i], R.xl[c][i], dl);
            }
        }
        // |dh|, |dl| <= 128 * 128 * 127 < 2^21: 254 dh + dl is exact in 32 bits
        return R.u * (float)(254 * dh + dl);
    }
};

// ---------------------------------------------------------------------------
// Q5_K: Q4_K's layout plus 32 bytes of fifth bits (qh at byte 16, qs at 48):
// weight 64c + 32h + l takes bit 2c + h of qh[l] as 16.  The lane owns
// sub-blocks 4hf..4hf+3 as in Q4_K; each code byte gets its fifth bit OR'ed
// into bit 4, and the integer dot products run on 5-bit codes.
struct Q5K {
    static int64_t scale_offset(int64_t, int64_t) { return 0; }
    static constexpr int kBlockBytes = 176;
    static constexpr bool kRowScaled = false;
    static constexpr int kWarps = 8;
    struct X {
        uint32_t xh[4][8], xl[4][8];
        int xs[4];
        float u;
        uint32_t mA, mB, qoff, hsh;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t) {
        load_x_parts(R.xh, R.xl, R.xs, R.u, ximg, xmeta, S, kbc, hf);
        if (!valid) R.u = 0.f;
        R.mA = hf ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
        R.mB = hf ? 0x30303030u : 0u;
        R.qoff = 48u + 64u * (uint32_t)hf;
        R.hsh = 4u * (uint32_t)hf;
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint4 hd = lds(blk);
        const uint4 ha = lds(blk + 16u), hb = lds(blk + 32u);
        const uint4 qa = lds(blk + R.qoff), qb = lds(blk + R.qoff + 16);
        const uint4 qc = lds(blk + R.qoff + 32), qd = lds(blk + R.qoff + 48);
        const uint32_t w0[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const uint32_t w1[8] = {qc.x, qc.y, qc.z, qc.w, qd.x, qd.y, qd.z, qd.w};
        const uint32_t qh[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
        const uint32_t sc4 = ((hf ? hd.w : hd.y) & R.mA) | ((hd.y >> 2) & R.mB);
        const uint32_t m4 = ((hf ? (hd.w >> 4) : hd.z) & R.mA) | ((hd.z >> 2) & R.mB);
        int dh0 = 0, dl0 = 0, dh1 = 0, dl1 = 0, dh2 = 0, dl2 = 0, dh3 = 0, dl3 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // bits 4hf..4hf+3 of each qh byte are the fifth bits of the lane's four sub-blocks
            const uint32_t hb4 = qh[i] >> R.hsh;
            const uint32_t c0 = (w0[i] & 0x0F0F0F0Fu) | ((hb4 << 4) & 0x10101010u);
            const uint32_t c1 = ((w0[i] >> 4) & 0x0F0F0F0Fu) | ((hb4 << 3) & 0x10101010u);
            const uint32_t c2 = (w1[i] & 0x0F0F0F0Fu) | ((hb4 << 2) & 0x10101010u);
            const uint32_t c3 = ((w1[i] >> 4) & 0x0F0F0F0Fu) | ((hb4 << 1) & 0x10101010u);
            dh0 = dp4a_us(c0, R.xh[0][i], dh0);
            dl0 = dp4a_us(c0, R.xl[0][i], dl0);
            dh1 = dp4a_us(c1, R.xh[1][i], dh1);
            dl1 = dp4a_us(c1, R.xl[1][i], dl1);
            dh2 = dp4a_us(c2, R.xh[2][i], dh2);
            dl2 = dp4a_us(c2, R.xl[2][i], dl2);
            dh3 = dp4a_us(c3, R.xh[3][i], dh3);
            dl3 = dp4a_us(c3, R.xl[3][i], dl3);
        }
        const int s0 = byte_of(sc4, 0), s1 = byte_of(sc4, 1), s2 = byte_of(sc4, 2), s3 = byte_of(sc4, 3);
        const int H = s0 * dh0 + s1 * dh1 + s2 * dh2 + s3 * dh3;        // |H| < 2^25
        const int L = s0 * dl0 + s1 * dl1 + s2 * dl2 + s3 * dl3;
        const int M = byte_of(m4, 0) * R.xs[0] + byte_of(m4, 1) * R.xs[1] +
                      byte_of(m4, 2) * R.xs[2] + byte_of(m4, 3) * R.xs[3];
        const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
        return R.u * (d * fmaf(254.0f, (float)H, (float)L) - dmin * (float)M);
    }
};

// ---------------------------------------------------------------------------
// Per-row int4: a row is k/2 bytes, weight 2i in the low nibble of byte i;
// the lane owns 128 weights (64 bytes).  XOR with 0x88 turns each two's-
// complement code q into q + 8 (0..15), so the integer dot products run on
// unsigned codes and 8 * (sum of x) is subtracted; low nibbles meet the even
// positions' x limbs and high nibbles (kept in place, 16 (q + 8)) the odd
// ones, split apart once at load.  As for per-row int8 the lanes' ranges
// would share banks, so lane l reads its four 16-byte chunks in the order
// (c + l/2) mod 4.  The row's f32 scale multiplies the reduced sum.
struct I4R {
    static constexpr int kBlockBytes = 128;
    static constexpr bool kRowScaled = true;
    static constexpr int kWarps = 8;
    static int64_t scale_offset(int64_t n_out, int64_t k) { return i4row_scale_offset(n_out, k); }
    struct X {
        uint32_t eh[4][4], el[4][4], oh[4][4], ol[4][4];   // chunk (c + lane/2) mod 4: even / odd limbs
        int xs;                                          // sum of 254 xh + xl over the lane's 128 positions
        float u;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t) {
        uint32_t xh[4][8], xl[4][8];
        int xs32[4];
        load_x_parts(xh, xl, xs32, R.u, ximg, xmeta, S, kbc, hf);
        if (!valid) R.u = 0.f;
        R.xs = xs32[0] + xs32[1] + xs32[2] + xs32[3];
        const int rot = (threadIdx.x & 31) >> 1;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int m = (c + rot) & 3;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t ah = 0, bh = 0, al = 0, bl = 0;
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    if (mm == m) { ah = xh[mm][2 * i]; bh = xh[mm][2 * i + 1]; al = xl[mm][2 * i]; bl = xl[mm][2 * i + 1]; }
                R.eh[c][i] = __byte_perm(ah, bh, 0x6420u);
                R.oh[c][i] = __byte_perm(ah, bh, 0x7531u);
                R.el[c][i] = __byte_perm(al, bl, 0x6420u);
                R.ol[c][i] = __byte_perm(al, bl, 0x7531u);
            }
        }
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint32_t a = blk + 64u * (uint32_t)hf;
        const uint32_t rot = (threadIdx.x & 31u) >> 1;
        int eh = 0, el = 0, oh = 0, ol = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 q = lds(a + 16u * ((c + rot) & 3u));
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = (qw[i] ^ 0x88888888u) & 0x0F0F0F0Fu;     // q + 8 of even weights
                const uint32_t hi = (qw[i] ^ 0x88888888u) & 0xF0F0F0F0u;     // 16 (q + 8) of odd weights
                eh = dp4a_us(lo, R.eh[c][i], eh);
                el = dp4a_us(lo, R.el[c][i], el);
                oh = dp4a_us(hi, R.oh[c][i], oh);
                ol = dp4a_us(hi, R.ol[c][i], ol);
            }
        }
        // 16 * sum (q + 8) X, exact in 32 bits (|.| < 2^22), then minus 16 * 8 * sum X
        const float h16 = (float)(16 * eh + oh), l16 = (float)(16 * el + ol);
        return R.u * 0.0625f * (fmaf(254.0f, h16, l16) - 128.0f * (float)R.xs);
    }
};

// ---------------------------------------------------------------------------
// Q2_K (84 bytes: 16 scale/min bytes, 64 bytes of 2-bit codes, f16 d, dmin):
// weight 128n + 32j + l takes bits 2j, 2j+1 of qs[32n + l]; its group of 16
// (i / 16) has scale = low nibble, min = high nibble of scales[i / 16].  The
// lane owns half n = hf: codes qs[32hf..32hf+31], groups 8hf..8hf+7.  Blocks
// are 4-byte aligned, so every read is a 32-bit word.
struct Q2K {
    static constexpr int kBlockBytes = 84;
    static constexpr bool kRowScaled = false;
    static constexpr int kWarps = 12;
    static int64_t scale_offset(int64_t, int64_t) { return 0; }
    struct X {
        uint32_t xh[4][8], xl[4][8];
        int xs[8];          // sum of 254 xh + xl over each group of 16
        float u;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t) {
        int xs32[4];
        load_x_parts(R.xh, R.xl, xs32, R.u, ximg, xmeta, S, kbc, hf);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            int sh = 0, sl = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sh = dp4a_ss(R.xh[g >> 1][4 * (g & 1) + i], 0x01010101u, sh);
                sl = dp4a_ss(R.xl[g >> 1][4 * (g & 1) + i], 0x01010101u, sl);
            }
            R.xs[g] = 254 * sh + sl;
        }
        if (!valid) R.u = 0.f;
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = lds32(blk + 16u + 32u * (uint32_t)hf + 4u * (uint32_t)i);
        const uint32_t s0 = lds32(blk + 8u * (uint32_t)hf), s1 = lds32(blk + 8u * (uint32_t)hf + 4u);
        const uint32_t dd = lds32(blk + 80u);
        int H = 0, L = 0, M = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            // groups 2t (words 0-3) and 2t+1 (words 4-7) of part t
            int dh0 = 0, dl0 = 0, dh1 = 0, dl1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // the codes of part t in place, i.e. 4^t times their value
                const uint32_t c0 = q[i] & (0x03030303u << (2 * t));
                const uint32_t c1 = q[4 + i] & (0x03030303u << (2 * t));
                dh0 = dp4a_us(c0, R.xh[t][i], dh0);
                dl0 = dp4a_us(c0, R.xl[t][i], dl0);
                dh1 = dp4a_us(c1, R.xh[t][4 + i], dh1);
                dl1 = dp4a_us(c1, R.xl[t][4 + i], dl1);
            }
            const uint32_t sw = t < 2 ? s0 : s1;
            const int g0 = byte_of(sw, 2 * (t & 1)), g1 = byte_of(sw, 2 * (t & 1) + 1);
            // times 4^(3-t): every part of H and L then carries 64 (|H|, |L| < 2^26)
            H += ((g0 & 15) * dh0 + (g1 & 15) * dh1) << (6 - 2 * t);
            L += ((g0 & 15) * dl0 + (g1 & 15) * dl1) << (6 - 2 * t);
            M += (g0 >> 4) * R.xs[2 * t] + (g1 >> 4) * R.xs[2 * t + 1];
        }
        const float d = h2f(dd), dmin = h2f(dd >> 16);
        return R.u * (d * (1.0f / 64.0f) * fmaf(254.0f, (float)H, (float)L) - dmin * (float)M);
    }
};

// ---------------------------------------------------------------------------
// Q3_K (110 bytes: hmask[32], 64 bytes of 2-bit codes, 12 bytes of sixteen
// signed 6-bit scales, f16 d): weight 128n + 32j + l takes bits 2j, 2j+1 of
// qs[32n + l] as a code and bit 4n + j of hmask[l] as its high bit, value =
// code - 4 when that bit is clear, code when set; group i / 16 has scale
// (low nibble of byte s (s < 8) or high nibble of byte s - 8, with bits
// 2(s/4), 2(s/4)+1 of byte 8 + s % 4 on top) - 32.  The lane owns half n =
// hf; code | high << 2 = value + 4 (0..7) feeds the dot products and 4 * (sum
// of x) per group is subtracted.  Blocks may start 2 bytes past a word
// boundary: the lane reads aligned words and realigns each with one permute.
struct Q3K {
    static constexpr int kBlockBytes = 110;
    static constexpr bool kRowScaled = false;
    static constexpr int kWarps = 12;
    static int64_t scale_offset(int64_t, int64_t) { return 0; }
    struct X {
        uint32_t xh[4][8], xl[4][8];
        int xs[8];          // sum of 254 xh + xl over each group of 16
        float u;
        uint32_t delta, sel, dsh;
    };
    static __device__ __forceinline__ void load(X &R, const uint8_t *ximg, const uint8_t *xmeta, int S,
                                                int kbc, int hf, bool valid, uint32_t lane_base) {
        int xs32[4];
        load_x_parts(R.xh, R.xl, xs32, R.u, ximg, xmeta, S, kbc, hf);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            int sh = 0, sl = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sh = dp4a_ss(R.xh[g >> 1][4 * (g & 1) + i], 0x01010101u, sh);
                sl = dp4a_ss(R.xl[g >> 1][4 * (g & 1) + i], 0x01010101u, sl);
            }
            R.xs[g] = 254 * sh + sl;
        }
        if (!valid) R.u = 0.f;
        R.delta = lane_base & 2u;
        R.sel = R.delta ? 0x5432u : 0x3210u;
        R.dsh = R.delta ? 16u : 0u;
    }
    static __device__ __forceinline__ float dot(uint32_t blk, const X &R, int hf) {
        const uint32_t a = blk - R.delta;
        uint32_t hm[8], q[8], sc[3];
        {
            uint32_t w[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) w[j] = lds32(a + 4u * (uint32_t)j);
#pragma unroll
            for (int j = 0; j < 8; ++j) hm[j] = __byte_perm(w[j], w[j + 1], R.sel) >> (4u * (uint32_t)hf);
        }
        {
            uint32_t w[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) w[j] = lds32(a + 32u + 32u * (uint32_t)hf + 4u * (uint32_t)j);
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = __byte_perm(w[j], w[j + 1], R.sel);
        }
        uint32_t dw;
        {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = lds32(a + 96u + 4u * (uint32_t)j);
#pragma unroll
            for (int j = 0; j < 3; ++j) sc[j] = __byte_perm(w[j], w[j + 1], R.sel);
            dw = lds32(a + 108u) >> R.dsh;
        }
        // signed scales of the lane's groups g = 0..7 (absolute 8hf + g)
        const uint32_t lo = hf ? ((sc[0] >> 4) & 0x0F0F0F0Fu) : (sc[0] & 0x0F0F0F0Fu);
        const uint32_t lo2 = hf ? ((sc[1] >> 4) & 0x0F0F0F0Fu) : (sc[1] & 0x0F0F0F0Fu);
        const uint32_t hi = sc[2] >> (4u * (uint32_t)hf);       // bits 2(g/4) + 4hf of byte g % 4
        int H = 0, L = 0, M = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            int dh0 = 0, dl0 = 0, dh1 = 0, dl1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // parts 0-2: the 3-bit codes assembled in place (4^t times their
                // value, at most 112); part 3 shifted down (7 * 64 is no byte)
                const uint32_t c0 = t < 3 ? (q[i] & (0x03030303u << (2 * t))) | ((hm[i] << (t + 2)) & (0x04040404u << (2 * t)))
                                          : ((q[i] >> 6) & 0x03030303u) | (((hm[i] >> 3) & 0x01010101u) << 2);
                const uint32_t c1 = t < 3 ? (q[4 + i] & (0x03030303u << (2 * t))) | ((hm[4 + i] << (t + 2)) & (0x04040404u << (2 * t)))
                                          : ((q[4 + i] >> 6) & 0x03030303u) | (((hm[4 + i] >> 3) & 0x01010101u) << 2);
                dh0 = dp4a_us(c0, R.xh[t][i], dh0);
                dl0 = dp4a_us(c0, R.xl[t][i], dl0);
                dh1 = dp4a_us(c1, R.xh[t][4 + i], dh1);
                dl1 = dp4a_us(c1, R.xl[t][4 + i], dl1);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int g = 2 * t + e;
                const int lo4 = byte_of(g < 4 ? lo : lo2, g & 3);
                const int hi2 = (byte_of(hi, g & 3) >> (2 * (g >> 2))) & 3;
                const int scg = (lo4 | (hi2 << 4)) - 32;
                // every part of H and L carries 64 (|H|, |L| < 2^28)
                const int sh = t < 3 ? 6 - 2 * t : 6;
                H += (scg * (e ? dh1 : dh0)) << sh;
                L += (scg * (e ? dl1 : dl0)) << sh;
                M += scg * R.xs[g];
            }
        }
        // sum of value * X = sum of (value + 4) * X - 4 * sum of X, per group
        return R.u * h2f(dw) * (fmaf(254.0f, (float)H, (float)L) * (1.0f / 64.0f) - 4.0f * (float)M);
    }
};

// Rows gi and gi+NG of one stage (lane base address s); CHECK handles a
// partial last stage (v0, v1: whether each row is present).
template <class F, bool CHECK>
__device__ __forceinline__ void two_rows(float &p0, float &p1, uint32_t s, uint32_t rA0, uint32_t rA1,
                                         bool v0, bool v1, const typename F::X &X, int hf) {
    if (!CHECK) {
        p0 = F::dot(s + rA0, X, hf);
        p1 = F::dot(s + rA1, X, hf);
    } else {
        p0 = v0 ? F::dot(s + rA0, X, hf) : 0.f;
        p1 = v1 ? F::dot(s + rA1, X, hf) : 0.f;
    }
}

// Epilogues fused into the store (PESTI README, "Conformance": the QKV
// projections carry a bias, the MLP multiplies silu of the gate projection by
// the up projection).
// silu(z) = z * sigmoid(z) = z / (1 + e^-z), with CUDA's expf; for z below
// about -88 e^-z is inf and the quotient is -0, the limit.
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Two instances per format: RT = false has no epilogue at compile time (the
// plain mat-vec), RT = true takes the epilogue as a run-time parameter and
// serves both the bias and SwiGLU, so a decode step that mixes them runs two
// codes, not three.  Three template instances of this large kernel cycling
// in one step measured 3 us per step slower (instruction fetch); one
// run-time instance for everything 0.4 us slower on the plain step.
template <class F, bool RT>
__global__ void __launch_bounds__(threads_for<F::kWarps>(), MINB) gemv_rows(Params p) {
    constexpr int CW = F::kWarps;
    constexpr int kThreads = threads_for<CW>();
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t x_bar;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int S = p.k / 64;
    const uint32_t rowbytes = (uint32_t)nb * (uint32_t)F::kBlockBytes;
    const int G = p.G, NG = p.NG, RS = p.RS, CA = G * NG;
    const bool SW = RT && p.epi == kEpiSwiGLU, BIAS = RT && p.epi == kEpiBias;
    // items: rows, or (SwiGLU) row pairs; IPS items per stage
    const int64_t n_items = SW ? (int64_t)p.n_ff : (int64_t)p.n_out;
    const int64_t r0 = n_items * blockIdx.x / gridDim.x;
    const int nrows = (int)(n_items * (blockIdx.x + 1) / gridDim.x - r0);
    const int IPS = SW ? NG : RS;
    const int units = (nrows + IPS - 1) / IPS;
    const int NS = p.nstages;
    const uint32_t stage_bytes = (uint32_t)RS * rowbytes;
    uint8_t *ximg = smem + (size_t)NS * stage_bytes;
    uint8_t *xmeta = ximg + 2 * p.k;
    float *red = reinterpret_cast<float *>(xmeta + S * 16);
    float *rsc = red + red_bytes(p) / 4;      // row scales (per-row formats): rows, then (SwiGLU) up rows
    float *bsm = rsc + rsc_bytes(p, F::kRowScaled, SW) / 4;   // bias slice (bias epilogue)
    const uint32_t ring_s = smem_u32(smem);

    // The producer lane initialises the barriers and releases the consumers
    // with a non-blocking arrive on named barrier 3 (its earlier writes are
    // then visible to them), so its first copy does not wait for the whole
    // CTA to reach a barrier (decode-layer set 28.0 -> 27.6 us).
    grid_dep_launch();   // the next kernel on the stream may start when resident
    if (warp == CW) {
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_init(&full_bar[s], 1);
                mbar_init(&empty_bar[s], CA);
            }
            mbar_init(&x_bar, 1);
            fence_mbar_init();
        }
        __syncwarp();
        named_arrive(3, kThreads);
    } else {
        named_sync(3, kThreads);
    }

    if (warp == CW) {
        // ---------------- producer: one contiguous copy per stage ----------------
        if (lane == 0) {
            if (!p.early_w) grid_dep_wait();   // the weights may be the previous kernel's output
            const uint64_t pol = make_evict_first_policy();
            const uint8_t *src = p.w + r0 * (int64_t)rowbytes;
            const int wsel = units >= kWideWindowUnits ? kXWindow : 1;
            const int window = wsel < NS ? wsel : NS;
            bool x_in = false;         // the consumers have converted x
            int landed = 0, lslot = 0; // stages known to have landed; slot of the next one
            uint32_t lph = 0;
            int slot = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int u = 0; u < units && ok; ++u) {
                const int rows = nrows - u * IPS < IPS ? nrows - u * IPS : IPS;
                const uint32_t bytes = (uint32_t)rows * rowbytes;
                if (!mbar_wait(&empty_bar[slot], ph ^ 1u)) break;
                if (!x_in) x_in = mbar_test_wait(&x_bar, 0);   // poll, never suspend
                // until x is in, stage u - window must have landed before stage u
                // is issued (window <= NS: that stage's slot is not re-armed yet)
                while (!x_in && landed <= u - window) {
                    if (!mbar_wait(&full_bar[lslot], lph)) { ok = false; break; }
                    if (++lslot == NS) { lslot = 0; lph ^= 1u; }
                    ++landed;
                }
                if (!ok) break;
                uint8_t *dst = smem + (size_t)slot * stage_bytes;
                if (SW) {
                    // gate rows to the stage's first half, the same pairs' up rows to the second
                    mbar_arrive_expect_tx(&full_bar[slot], 2 * bytes);
                    bulk_g2s_hint(dst, src, bytes, &full_bar[slot], pol);
                    bulk_g2s_hint(dst + (size_t)NG * rowbytes, src + (size_t)p.n_ff * rowbytes, bytes, &full_bar[slot], pol);
                } else {
                    mbar_arrive_expect_tx(&full_bar[slot], bytes);
                    bulk_g2s_hint(dst, src, bytes, &full_bar[slot], pol);
                }
                src += (size_t)IPS * rowbytes;
                if (u + 1 == window && u + 1 < units) {
                    // kL2PrefetchPercent of the rows after the window, rounded up to
                    // 16 bytes, at most kL2PrefetchBytes (kL2PrefetchBytesLong for
                    // rows of several segments: 4096x14336 7.81 -> 7.54 us, where
                    // 128 KB or 60 % slowed the decode-layer set); SwiGLU splits the
                    // budget between its gate and up rows
                    uint64_t pfb = (uint64_t)(nrows - (u + 1) * IPS) * rowbytes;
                    pfb = (pfb * kL2PrefetchPercent / 100 + 15) / 16 * 16;
                    const uint64_t budget = G == 1 ? kL2PrefetchBytes : kL2PrefetchBytesLong;
                    const uint64_t cap = SW ? budget / 2 : budget;
                    if (pfb > cap) pfb = cap;
                    bulk_prefetch_l2(src, (uint32_t)pfb);
                    if (SW) bulk_prefetch_l2(src + (size_t)p.n_ff * rowbytes, (uint32_t)pfb);
                }
                if (++slot == NS) { slot = 0; ph ^= 1u; }
            }
        }
        return;
    }

    // ---------------- x image (all consumer warps) ----------------
    bool dead = false;   // a wait ran out: stop waiting, keep going so every warp finishes
    grid_dep_wait();     // x may be the previous kernel's output
    // the CTA's row scales and bias slice: the first values' loads are issued
    // with x's and stored to shared memory after the x conversion
    const bool kVec = F::kRowScaled || BIAS;
    float v0 = 0.f, v1 = 0.f;
    const int i0v = threadIdx.x;
    if (kVec) {
        if (i0v < nrows) {
            v0 = F::kRowScaled ? __ldg(p.rscale + r0 + i0v) : __ldg(p.bias + r0 + i0v);
            if (F::kRowScaled && SW) v1 = __ldg(p.rscale + p.n_ff + r0 + i0v);
        }
    }
    prep_x_all<false, true>(p.x, ximg, xmeta, nb, S, warp, CW, lane);
    if (kVec) {
        float *dst = F::kRowScaled ? rsc : bsm;
        if (i0v < nrows) {
            dst[i0v] = v0;
            if (F::kRowScaled && SW) rsc[p.rows_cap + i0v] = v1;
        }
        for (int i = i0v + CW * 32; i < nrows; i += CW * 32) {
            if constexpr (F::kRowScaled) {
                rsc[i] = __ldg(p.rscale + r0 + i);
                if (SW) rsc[p.rows_cap + i] = __ldg(p.rscale + p.n_ff + r0 + i);
            } else {
                bsm[i] = __ldg(p.bias + r0 + i);
            }
        }
        if (F::kRowScaled && BIAS)
            for (int i = i0v; i < nrows; i += CW * 32) bsm[i] = __ldg(p.bias + r0 + i);
    }
    named_sync(1, CW * 32);
    if (threadIdx.x == 0) mbar_arrive(&x_bar);   // lifts the producer's in-flight limit
    if (warp >= CA) return;

    const int gi = warp / G, seg = warp - gi * G;
    const int hf = lane & 1;
    const int kb = seg * KW + (lane >> 1);
    const bool valid = kb < nb;
    const int kbc = valid ? kb : nb - 1;       // idle lanes read a real block, weight 0
    const uint32_t lane_base = ring_s + (uint32_t)kbc * (uint32_t)F::kBlockBytes;

    typename F::X X;
    F::load(X, ximg, xmeta, S, kbc, hf, valid, lane_base);
    const uint32_t rA0 = (uint32_t)gi * rowbytes, rA1 = (uint32_t)(gi + NG) * rowbytes;
    const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
    // the row this lane's reduced value belongs to: 0,1 of stage A, 2,3 of stage B
    // (SwiGLU: rows gi and gi+NG of a stage are the gate and up rows of pair gi)
    const int my_t = gi + (b3 ? NG : 0);

    int slot = 0;
    uint32_t ph = 0;
    for (int u = 0; u < units; u += 2) {
        const bool hasB = u + 1 < units;
        const int slotA = slot;
        const uint32_t phA = ph;
        if (++slot == NS) { slot = 0; ph ^= 1u; }
        const int slotB = slot;
        const uint32_t phB = ph;
        if (hasB) {
            if (++slot == NS) { slot = 0; ph ^= 1u; }
        }
        const uint32_t sA = lane_base + (uint32_t)slotA * stage_bytes;
        const uint32_t sB = lane_base + (uint32_t)slotB * stage_bytes;
        // items (rows, or pairs) in stages A and B
        const int nA = nrows - u * IPS < IPS ? nrows - u * IPS : IPS;
        const int nB = hasB ? (nrows - (u + 1) * IPS < IPS ? nrows - (u + 1) * IPS : IPS) : 0;
        float pr[4];
        // stage A: wait, compute its two rows, hand the slot back; then stage B
        if (!dead && !mbar_wait(&full_bar[slotA], phA)) dead = true;
        if (nA == IPS)
            two_rows<F, false>(pr[0], pr[1], sA, rA0, rA1, true, true, X, hf);
        else
            two_rows<F, true>(pr[0], pr[1], sA, rA0, rA1, gi < nA, SW ? gi < nA : gi + NG < nA, X, hf);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slotA]);
        if (hasB && !dead && !mbar_wait(&full_bar[slotB], phB)) dead = true;
        if (nB == IPS)
            two_rows<F, false>(pr[2], pr[3], sB, rA0, rA1, true, true, X, hf);
        else
            two_rows<F, true>(pr[2], pr[3], sB, rA0, rA1, gi < nB, SW ? gi < nB : gi + NG < nB, X, hf);
        __syncwarp();
        if (lane == 0 && hasB) mbar_arrive(&empty_bar[slotB]);
        // transposed reduction of the four rows: lanes 0-7 end with row 0,
        // 8-15 row 1, 16-23 row 2, 24-31 row 3
        float a0 = b4 ? pr[2] : pr[0], a1 = b4 ? pr[3] : pr[1];
        a0 += __shfl_xor_sync(0xffffffffu, b4 ? pr[0] : pr[2], 16);
        a1 += __shfl_xor_sync(0xffffffffu, b4 ? pr[1] : pr[3], 16);
        float v = (b3 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, b3 ? a0 : a1, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        const int n_here = b4 ? nB : nA;
        if (SW) {
            const float up = __shfl_down_sync(0xffffffffu, v, 8);   // lanes 0 and 16: the pair's up row
            if ((lane & 15) == 0 && gi < n_here) {
                if (G == 1) {
                    const int pair = (u + (b4 ? 1 : 0)) * NG + gi;    // relative to r0
                    if constexpr (F::kRowScaled)
                        p.y[r0 + pair] = silu(v * rsc[pair]) * (up * rsc[p.rows_cap + pair]);
                    else
                        p.y[r0 + pair] = silu(v) * up;
                } else {
                    const int row = (u + (b4 ? 1 : 0)) * RS + gi;    // stage-relative gate row
                    red[row * G + seg] = v;
                    red[(row + NG) * G + seg] = up;
                }
            }
        } else if ((lane & 7) == 0 && my_t < n_here) {
            const int row = (u + (b4 ? 1 : 0)) * RS + my_t;     // relative to r0
            if (G == 1) {
                const float yv = F::kRowScaled ? v * rsc[row] : v;
                p.y[r0 + row] = BIAS ? yv + bsm[row] : yv;
            } else {
                red[row * G + seg] = v;
            }
        }
    }
    if (G > 1) {
        // partial sums of the G segments of each row, added in segment order
        named_sync(2, CA * 32);
        for (int i = warp * 32 + lane; i < nrows; i += CA * 32) {
            if (SW) {
                const int row = (i / NG) * RS + i % NG;       // gate row of pair i; its up row is row + NG
                float g = red[row * G], up = red[(row + NG) * G];
                for (int g2 = 1; g2 < G; ++g2) {
                    g += red[row * G + g2];
                    up += red[(row + NG) * G + g2];
                }
                if constexpr (F::kRowScaled) {
                    g *= rsc[i];
                    up *= rsc[p.rows_cap + i];
                }
                p.y[r0 + i] = silu(g) * up;
            } else {
                float sum = red[i * G];
                for (int g2 = 1; g2 < G; ++g2) sum += red[i * G + g2];
                if constexpr (F::kRowScaled) sum *= rsc[i];
                p.y[r0 + i] = BIAS ? sum + bsm[i] : sum;
            }
        }
    }
}

// One launch over n_out rows (no epilogue or bias), or over the 2 * n_ff rows
// of a fused gate+up matrix writing n_ff SwiGLU outputs (n_out =
// 2 * n_ff); grid <= the number of items.
template <class F>
cudaError_t launch(const uint8_t *w, int64_t n_out, int64_t k, const float *x, float *y, int grid,
                   cudaStream_t s, int early_w, const float *bias, int epi_kind) {
    const float *rscale = F::kRowScaled ? reinterpret_cast<const float *>(w + F::scale_offset(n_out, k)) : nullptr;
    Params p{w, x, y, (int)n_out, (int)k, 0, 0, 0, 0, 0, early_w, (int)(n_out / 2), bias, rscale, epi_kind};
    if (!plan(k, n_out, grid, F::kBlockBytes, F::kWarps, p, epi_kind == kEpiSwiGLU, F::kRowScaled, epi_kind == kEpiBias))
        return cudaErrorInvalidValue;
    const int smem = p.nstages * p.RS * (int)(k / 256) * F::kBlockBytes + x_image_bytes(k, 1) + red_bytes(p) +
                     rsc_bytes(p, F::kRowScaled, epi_kind == kEpiSwiGLU) + bias_bytes(p, epi_kind == kEpiBias);
    auto kern = epi_kind == kEpiNone ? gemv_rows<F, false> : gemv_rows<F, true>;
    static PerDeviceOnce configured[2];
    const cudaError_t ce = configured[epi_kind == kEpiNone ? 0 : 1].run([kern] {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.sharedSizeBytes > (size_t)kStatic) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsSmem - kStatic);
    });
    if (ce != cudaSuccess) return ce;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads_for<F::kWarps>());
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <class F>
cudaError_t launch_epi(const uint8_t *w, int64_t n_out, int64_t k, const float *x, float *y, int grid,
                       cudaStream_t s, int early_w, const Epilogue &epi) {
    return launch<F>(w, n_out, k, x, y, grid, s, early_w, epi.kind == kEpiBias ? epi.bias : nullptr, epi.kind);
}

// Whether the whole-row kernel takes (fmt, k, n_out) at batch 1 (n_out = 2 *
// pairs for the SwiGLU epilogue).
inline bool takes(int fmt, int64_t k, int64_t n_out, bool swiglu = false) {
    Params p{};
    const int grid_est = 132;      // fewer SMs than any sm_103 part: a conservative row count
    const int64_t items = swiglu ? n_out / 2 : n_out;
    const int grid = (int)(items < grid_est ? items : grid_est);
    if (swiglu && (n_out % 2 || items < 1)) return false;
    if (fmt == PQ_Q4_K) return plan(k, n_out, grid, Q4K::kBlockBytes, Q4K::kWarps, p, swiglu);
    if (fmt == PQ_Q6_K) return plan(k, n_out, grid, Q6K::kBlockBytes, Q6K::kWarps, p, swiglu);
    if (fmt == PQ_Q8_0) return k % 256 == 0 && plan(k, n_out, grid, Q80::kBlockBytes, Q80::kWarps, p, swiglu);
    if (fmt == PQ_I8_ROW) return k % 256 == 0 && plan(k, n_out, grid, I8R::kBlockBytes, I8R::kWarps, p, swiglu, true);
    if (fmt == PQ_Q5_K) return plan(k, n_out, grid, Q5K::kBlockBytes, Q5K::kWarps, p, swiglu);
    if (fmt == PQ_I4_ROW) return k % 256 == 0 && plan(k, n_out, grid, I4R::kBlockBytes, I4R::kWarps, p, swiglu, true);
    if (fmt == PQ_Q2_K) return plan(k, n_out, grid, Q2K::kBlockBytes, Q2K::kWarps, p, swiglu);
    if (fmt == PQ_Q3_K) return plan(k, n_out, grid, Q3K::kBlockBytes, Q3K::kWarps, p, swiglu);
    return false;
}
}  // namespace rowk

// ---------------------------------------------------------------------------
// Batch 2 (NB = 2; NB = 4 also works, batch 3 as 4 with a zero column, but is
// not the fastest choice there), Q4_K: the whole-row kernel for NB columns.  A lane owns 256/(2*NB) weights of one super-block (chunk c
// = 64 weights for NB = 2; half a chunk, 16 bytes of qs = 32 weights over two
// sub-blocks, for NB = 4), so the x limbs of all NB columns for its k range
// still fit in 64 registers; a warp covers 32/(2*NB) super-blocks and G warps
// a row.  Stages are runs of whole rows (one bulk copy each) as at batch 1;
// each lane's partial products of four rows x NB columns are reduced with one
// transposed shuffle tree, split rows (G > 1) in shared memory in fixed order.
//
// x is converted once per call by prep_x_nb into the limb image (2.25 bytes
// per element per column) in scratch memory; each CTA fetches that image with
// one bulk copy.  Both kernels use programmatic dependent launch: prep_x_nb
// waits for the previous kernel before it lets this one launch, so the
// weights this kernel streams at once are complete, and this kernel waits for
// prep_x_nb only before its x copy.
namespace rowsnb {
constexpr int CW = 15;                       // consumer warps (with the producer: 512 threads, 128 registers)
// Rows up to kNbConvertMaxK long: the consumer warps convert x themselves
// after the dependency wait (the producer keeps kNbXWindow stages in flight
// until they have), so a call is one launch with no scratch; longer rows
// take the x image from prep_x_nb, which converts it once for all CTAs.
// Batch 2, Q4_K, launched back to back: 4096x14336 13.9 -> 13.0 us,
// 4096x8192 10.4 -> 8.7 us; at 8192x28672 (224 blocks of x per CTA) the
// prep kernel is faster, 30.3 against 32.0 us.
constexpr int64_t kNbConvertMaxK = 16384;
constexpr int kNbXWindow = 2;
constexpr int THREADS = (CW + 1) * 32;
constexpr int MAX_STAGES = 8;
constexpr int kStatic = 512;

template <int NB> struct Geo {
    static constexpr int LPB = 2 * NB;       // lanes per super-block
    static constexpr int KW = 32 / LPB;      // super-blocks per warp
    static constexpr int V = 4 * NB;         // values per lane per iteration (4 rows x NB columns)
    static constexpr int LOGV = NB == 2 ? 3 : 4;
};

// Bytes of one column of the limb image: 2k of limb groups, then k/64 x 16
// bytes of metadata (the layout prep_x_vals writes).
inline __host__ __device__ int col_bytes(int64_t k) { return (int)(2 * k + (k / 64) * 16); }

struct Params {
    const uint8_t *w;
    const uint8_t *x_img;   // NB columns of col_bytes(k), from prep_x_nb; null: x is converted in the kernel
    const float *x;         // with a null x_img: NB columns of k values (nb_cols real)
    float *y;
    long long ldy;
    int n_out;
    int k;
    int nb_cols;    // real columns (<= NB); the others are zero
    int G;          // warps per row
    int NG;         // row groups
    int RS;         // rows per stage
    int nstages;
    int rows_cap;
    int early_w;
};

template <int NB> inline int segments(int64_t k) { return (int)((k / 256 + Geo<NB>::KW - 1) / Geo<NB>::KW); }
template <int NB> inline int red_bytes(const Params &p) {
    return p.G > 1 ? (p.rows_cap * p.G * NB * 4 + 15) / 16 * 16 : 0;
}

template <int NB> inline bool plan(int64_t k, int64_t n_out, int grid, Params &p) {
    if (k % 256 || grid < 1) return false;
    const int G = segments<NB>(k);
    if (G < 1 || G > CW) return false;
    p.G = G;
    p.NG = CW / G;
    p.RS = 2 * p.NG;
    p.rows_cap = (int)((n_out + grid - 1) / grid);
    const int64_t stage = (int64_t)p.RS * (k / 256) * 144;
    const int64_t avail = kSmemBudget - kStatic - (int64_t)NB * col_bytes(k) - red_bytes<NB>(p);
    int64_t ns = avail / stage;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    p.nstages = (int)ns;
    return ns >= 2;
}

// Sum over the warp's 32 lanes of each of V values; afterwards lane l holds the
// total of value l >> (5 - LOGV) (a transposed tree: each step halves the
// values a lane carries).
template <int V, int LOGV>
__device__ __forceinline__ float transposed_sum(float (&v)[V], int lane) {
#pragma unroll
    for (int st = 0; st < LOGV; ++st) {
        const int o = 16 >> st, n = V >> st;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float send = up ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 >> LOGV; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Limb image of NB columns: warp w of block (i, b) converts 256-value block
// 8i + w of column b (zeros for b >= nb_cols).
template <int NB>
__global__ void __launch_bounds__(256) prep_x_nb(const float *__restrict__ x, int k, int nb_cols,
                                                 uint8_t *__restrict__ img) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = blockIdx.x * 8 + warp, b = blockIdx.y;
    const int nb = k / 256;
    if (q >= nb) return;
    uint8_t *col = img + (size_t)b * col_bytes(k);
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (b < nb_cols) {
        const float *xq = x + (size_t)b * k + q * 256 + 8 * lane;
        const float4 a = ldg_f4(xq), c = ldg_f4(xq + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    }
    prep_x_vals(v, col, col + 2 * k, q, k / 64, lane);
}

template <int NB>
__global__ void __launch_bounds__(THREADS, 1) gemv_rows_nb(Params p) {
    using Gm = Geo<NB>;
    constexpr int W4 = 8 / (NB / 2);         // qs words per lane: 8 (NB = 2) or 4 (NB = 4)
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t x_bar;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int S = p.k / 64;
    const int CB = col_bytes(p.k);
    const uint32_t rowbytes = (uint32_t)nb * 144u;
    const int G = p.G, NG = p.NG, RS = p.RS, CA = G * NG;
    const int64_t r0 = (int64_t)p.n_out * blockIdx.x / gridDim.x;
    const int nrows = (int)((int64_t)p.n_out * (blockIdx.x + 1) / gridDim.x - r0);
    const int units = (nrows + RS - 1) / RS;
    const int NS = p.nstages;
    const uint32_t stage_bytes = (uint32_t)RS * rowbytes;
    uint8_t *ximg = smem + (size_t)NS * stage_bytes;            // NB columns of CB bytes
    float *red = reinterpret_cast<float *>(ximg + (size_t)NB * CB);
    const uint32_t ring_s = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CA);
        }
        mbar_init(&x_bar, 1);
        fence_mbar_init();
    }
    rowk::grid_dep_launch();
    __syncthreads();

    if (warp == CW) {
        // ---------------- producer: one contiguous copy per stage ----------------
        if (lane == 0) {
            // with the x image from prep_x_nb: the first ring's worth of weights
            // (the preceding kernel is prep_x_nb, which waited for the caller's
            // kernel), then the image; with x converted here: a window of
            // kNbXWindow stages, then the rest once the consumers have converted x
            const bool img = p.x_img != nullptr;
            if (!img && !p.early_w) rowk::grid_dep_wait();   // the weights may be the previous kernel's output
            const int cap = img ? NS : (kNbXWindow < NS ? kNbXWindow : NS);
            const int early = units < cap ? units : cap;
            const uint64_t pol = make_evict_first_policy();
            const uint8_t *src = p.w + r0 * (int64_t)rowbytes;
            int slot = 0;
            uint32_t ph = 0;
            for (int u = 0; u <= units; ++u) {
                if (u == early) {
                    if (img) {
                        rowk::grid_dep_wait();
                        mbar_arrive_expect_tx(&x_bar, (uint32_t)(NB * CB));
                        bulk_g2s(ximg, p.x_img, (uint32_t)(NB * CB), &x_bar);
                    } else if (u < units && !mbar_wait(&x_bar, 0)) {
                        break;
                    }
                }
                if (u == units) break;
                const int rows = nrows - u * RS < RS ? nrows - u * RS : RS;
                const uint32_t bytes = (uint32_t)rows * rowbytes;
                if (!mbar_wait(&empty_bar[slot], ph ^ 1u)) break;
                mbar_arrive_expect_tx(&full_bar[slot], bytes);
                bulk_g2s_hint(smem + (size_t)slot * stage_bytes, src, bytes, &full_bar[slot], pol);
                src += (size_t)RS * rowbytes;
                if (++slot == NS) { slot = 0; ph ^= 1u; }
            }
        }
        return;
    }

    bool dead = false;   // a wait ran out: stop waiting, keep going so every warp finishes
    if (p.x_img) {
        if (warp >= CA) return;
        if (!mbar_wait(&x_bar, 0)) dead = true;
    } else {
        // x of the NB columns to limbs in shared memory, by every consumer warp
        rowk::grid_dep_wait();                   // x may be the previous kernel's output
#pragma unroll
        for (int b = 0; b < NB; ++b)
            prep_x_all(b < p.nb_cols ? p.x + (size_t)b * p.k : nullptr, ximg + (size_t)b * CB,
                       ximg + (size_t)b * CB + 2 * p.k, nb, S, warp, CW, lane);
        named_sync(1, CW * 32);
        if (threadIdx.x == 0) mbar_arrive(&x_bar);   // the producer may stream past its window
        if (warp >= CA) return;
    }

    const int gi = warp / G, seg = warp - gi * G;
    const int part = lane % Gm::LPB;
    const int kb = seg * Gm::KW + lane / Gm::LPB;
    const bool valid = kb < nb;
    const int kbc = valid ? kb : nb - 1;       // idle lanes read a real block, weight 0
    // chunk c (sub-blocks 2c, 2c+1) and, for NB = 4, the 16-byte half h of its qs
    const int c = NB == 2 ? part : part >> 1;
    const int h = NB == 2 ? 0 : (part & 1);
    const int slice = 4 * kbc + c;

    // x limbs of the lane's positions, per column: [b][0..W4) xh of sub-block 2c,
    // then 2c+1; xl likewise
    uint32_t xh0[NB][W4], xh1[NB][W4], xl0[NB][W4], xl1[NB][W4];
    int xs0[NB], xs1[NB];
    float u[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const uint8_t *img = ximg + (size_t)b * CB;
        const uint8_t *meta = img + 2 * p.k;
        if constexpr (NB == 2) {
            uint4 g[8];
#pragma unroll
            for (int gi2 = 0; gi2 < 8; ++gi2) g[gi2] = *reinterpret_cast<const uint4 *>(img + (gi2 * S + slice) * 16);
            const uint32_t *gw = reinterpret_cast<const uint32_t *>(g);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                xh0[b][i] = gw[i];
                xh1[b][i] = gw[8 + i];
                xl0[b][i] = gw[16 + i];
                xl1[b][i] = gw[24 + i];
            }
        } else {
            const uint4 a0 = *reinterpret_cast<const uint4 *>(img + ((0 + h) * S + slice) * 16);
            const uint4 a1 = *reinterpret_cast<const uint4 *>(img + ((2 + h) * S + slice) * 16);
            const uint4 a2 = *reinterpret_cast<const uint4 *>(img + ((4 + h) * S + slice) * 16);
            const uint4 a3 = *reinterpret_cast<const uint4 *>(img + ((6 + h) * S + slice) * 16);
            const uint32_t w0[4] = {a0.x, a0.y, a0.z, a0.w}, w1[4] = {a1.x, a1.y, a1.z, a1.w};
            const uint32_t w2[4] = {a2.x, a2.y, a2.z, a2.w}, w3[4] = {a3.x, a3.y, a3.z, a3.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xh0[b][i] = w0[i];
                xh1[b][i] = w1[i];
                xl0[b][i] = w2[i];
                xl1[b][i] = w3[i];
            }
        }
        const int4 mt = *reinterpret_cast<const int4 *>(meta + slice * 16);
        // the sub-block sums go with one lane of each sub-block pair (h == 0)
        xs0[b] = h == 0 ? mt.x : 0;
        xs1[b] = h == 0 ? mt.y : 0;
        u[b] = valid ? __int_as_float(mt.z) : 0.f;
    }

    // byte selectors for (sc, m) of sub-blocks 2c and 2c+1 from the packed scales
    const uint32_t c2 = 2u * (uint32_t)(c & 1);
    const uint32_t selP = c2 | ((c2 + 1) << 4) | ((c2 + 4) << 8) | ((c2 + 5) << 12);
    const uint32_t selQ = c2 | ((c2 + 1) << 4) | (c2 << 8) | ((c2 + 1) << 12);
    const uint32_t lane_base = ring_s + (uint32_t)kbc * 144u;
    const uint32_t qoff = 16u + 32u * (uint32_t)c + 16u * (uint32_t)h;

    // products of one row (block at shared address blk) with all NB columns
    auto row_dot = [&](uint32_t blk, float (&out)[NB]) {
        const uint4 hd = lds128(blk);
        uint32_t wq[W4];
        {
            const uint4 qa = lds128(blk + qoff);
            wq[0] = qa.x; wq[1] = qa.y; wq[2] = qa.z; wq[3] = qa.w;
            if constexpr (W4 == 8) {
                const uint4 qb = lds128(blk + qoff + 16);
                wq[4] = qb.x; wq[5] = qb.y; wq[6] = qb.z; wq[7] = qb.w;
            }
        }
        const uint32_t P = __byte_perm(hd.y, hd.z, selP);
        uint32_t r4;
        if (c < 2) {
            r4 = P & 0x3F3F3F3Fu;
        } else {
            const uint32_t Q = __byte_perm(hd.w, 0u, selQ);
            r4 = ((P >> 2) & 0x30303030u) | (Q & 0x00000F0Fu) | ((Q >> 4) & 0x0F0F0000u);
        }
        const int sc0x16 = (int)((r4 << 4) & 0xFF0u), sc1 = (int)((r4 >> 8) & 0xFFu);
        const int m0 = (int)((r4 >> 16) & 0xFFu), m1 = (int)(r4 >> 24);
        const float d16 = h2f(hd.x) * 0.0625f, dmin = h2f(hd.x >> 16);
        uint32_t lo[W4], hi[W4];
#pragma unroll
        for (int i = 0; i < W4; ++i) {
            lo[i] = wq[i] & 0x0F0F0F0Fu;
            hi[i] = wq[i] & 0xF0F0F0F0u;     // 16*q: rescaled by d/16 below
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            int dh0 = 0, dl0 = 0, dh1 = 0, dl1 = 0;
#pragma unroll
            for (int i = 0; i < W4; ++i) {
                dh0 = dp4a_ss(lo[i], xh0[b][i], dh0);
                dl0 = dp4a_ss(lo[i], xl0[b][i], dl0);
                dh1 = dp4a_us(hi[i], xh1[b][i], dh1);
                dl1 = dp4a_us(hi[i], xl1[b][i], dl1);
            }
            const int H = sc0x16 * dh0 + sc1 * dh1;
            const int L = sc0x16 * dl0 + sc1 * dl1;
            const int M = m0 * xs0[b] + m1 * xs1[b];
            out[b] = u[b] * (d16 * fmaf(254.0f, (float)H, (float)L) - dmin * (float)M);
        }
    };

    const uint32_t rA0 = (uint32_t)gi * rowbytes, rA1 = (uint32_t)(gi + NG) * rowbytes;
    constexpr int SHIFT = 5 - Gm::LOGV;                 // lane >> SHIFT = value index after the tree
    const int my_v = lane >> SHIFT;
    const int my_t = my_v / NB, my_b = my_v % NB;       // row slot (0,1 stage A; 2,3 stage B), column
    const int my_rowoff = gi + ((my_t & 1) ? NG : 0);

    int slot = 0;
    uint32_t ph = 0;
    for (int uu = 0; uu < units; uu += 2) {
        const bool hasB = uu + 1 < units;
        const int slotA = slot;
        const uint32_t phA = ph;
        if (++slot == NS) { slot = 0; ph ^= 1u; }
        const int slotB = slot;
        const uint32_t phB = ph;
        if (hasB) {
            if (++slot == NS) { slot = 0; ph ^= 1u; }
        }
        const int nA = nrows - uu * RS < RS ? nrows - uu * RS : RS;
        const int nB = hasB ? (nrows - (uu + 1) * RS < RS ? nrows - (uu + 1) * RS : RS) : 0;
        float v[Gm::V];
        float tmp[NB];
        if (!dead && !mbar_wait(&full_bar[slotA], phA)) dead = true;
        {
            const uint32_t sA = lane_base + (uint32_t)slotA * stage_bytes;
            row_dot(sA + rA0, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[b] = gi < nA ? tmp[b] : 0.f;
            row_dot(sA + rA1, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[NB + b] = gi + NG < nA ? tmp[b] : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slotA]);
        if (hasB && !dead && !mbar_wait(&full_bar[slotB], phB)) dead = true;
        {
            const uint32_t sB = lane_base + (uint32_t)slotB * stage_bytes;
            row_dot(sB + rA0, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[2 * NB + b] = gi < nB ? tmp[b] : 0.f;
            row_dot(sB + rA1, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[3 * NB + b] = gi + NG < nB ? tmp[b] : 0.f;
        }
        __syncwarp();
        if (lane == 0 && hasB) mbar_arrive(&empty_bar[slotB]);
        const float tot = transposed_sum<Gm::V, Gm::LOGV>(v, lane);
        if ((lane & ((1 << SHIFT) - 1)) == 0 && my_b < p.nb_cols) {
            const int n_here = my_t >= 2 ? nB : nA;
            if (my_rowoff < n_here) {
                const int row = (uu + (my_t >= 2 ? 1 : 0)) * RS + my_rowoff;   // relative to r0
                if (G == 1)
                    p.y[(size_t)my_b * p.ldy + r0 + row] = tot;
                else
                    red[((size_t)row * G + seg) * NB + my_b] = tot;
            }
        }
    }
    if (G > 1) {
        named_sync(2, CA * 32);
        for (int i = warp * 32 + lane; i < nrows * NB; i += CA * 32) {
            const int row = i / NB, b = i % NB;
            if (b >= p.nb_cols) continue;
            float sum = red[((size_t)row * G) * NB + b];
            for (int g2 = 1; g2 < G; ++g2) sum += red[((size_t)row * G + g2) * NB + b];
            p.y[(size_t)b * p.ldy + r0 + row] = sum;
        }
    }
}

template <int NB>
cudaError_t launch(const uint8_t *w, int64_t n_out, int64_t k, const float *x, int nb_cols, float *y, int64_t ldy,
                   int grid, cudaStream_t s) {
    Params p{w, nullptr, x, y, (long long)ldy, (int)n_out, (int)k, nb_cols, 0, 0, 0, 0, 0, weight_prefetch()};
    if (!plan<NB>(k, n_out, grid, p)) return cudaErrorInvalidValue;
    const int smem = p.nstages * p.RS * (int)(k / 256) * 144 + NB * col_bytes(k) + red_bytes<NB>(p);
    static PerDeviceOnce configured;
    const cudaError_t ce = configured.run([] {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, gemv_rows_nb<NB>);
        if (e != cudaSuccess) return e;
        if (fa.sharedSizeBytes > (size_t)kStatic) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(gemv_rows_nb<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBudget - kStatic);
    });
    if (ce != cudaSuccess) return ce;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (k <= kNbConvertMaxK) {
        // x converted by the kernel itself: one launch, no scratch
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_rows_nb<NB>, p);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    cudaMemPool_t pool = scratch_pool();
    if (!pool) return cudaErrorMemoryAllocation;
    void *img = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&img, (size_t)NB * col_bytes(k), pool, s);
    if (e != cudaSuccess) return e;
    p.x_img = static_cast<const uint8_t *>(img);
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3((unsigned)((k / 256 + 7) / 8), NB);
    pcfg.blockDim = dim3(256);
    pcfg.stream = s;
    pcfg.attrs = attr;
    pcfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&pcfg, prep_x_nb<NB>, x, (int)k, nb_cols, static_cast<uint8_t *>(img));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gemv_rows_nb<NB>, p);
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    const cudaError_t f = cudaFreeAsync(img, s);
    return e != cudaSuccess ? e : f;
}

// Whether this kernel runs Q4_K (k, n_out) at `batch` columns.  It is used at
// batch 2 for long rows (k >= 8192), where it beats the chunked kernel
// (4096x14336: 14.0 vs 18.6 us), and at k = 4096 for tall matrices
// (kNbTallRows rows or more, 128 per CTA on a full GPU), where its streaming
// beats the register-operand kernel's half-empty 4-column tiles (28672x4096:
// 16.8 against 19.1 us; 14336x4096: 11.4 against 10.8, so shorter matrices
// keep that kernel); at batch 3-4 (NB = 4) other kernels are faster.
constexpr int64_t kNbTallRows = 19456;
inline bool takes(int64_t k, int64_t n_out, int batch) {
    Params p{};
    const int grid_est = 132;      // fewer SMs than any sm_103 part: a conservative row count
    const int grid = (int)(n_out < grid_est ? n_out : grid_est);
    return batch == 2 && (k >= 8192 || (k == 4096 && n_out >= kNbTallRows)) && plan<2>(k, n_out, grid, p);
}
}  // namespace rowsnb

// ---------------------------------------------------------------------------
// Q6_K at batch 2-4: the whole-row kernel for several columns, so that the
// 210-byte super-blocks (GGUF Q6_K; PESTI README, "What This Is") stream once
// per call instead of once per column.
//
// Lane (h, t, j) of a super-block's eight lanes owns 32 weights: the 16
// positions 16j..16j+15 of the runs t and t+2 of half h (run t of half h is
// weights 128h + 32t .. +31).  Both runs take their low four bits from the
// same 16 ql bytes (low and high nibbles) and their high two bits from the
// same 16 qh bytes (bit pairs t and t+2), and each run's 16 positions share
// one signed 8-bit scale, so a lane reads 32 bytes and two scales per row.
// Its x limbs (four 16-byte groups per column of the image prep_x_nb writes)
// stay in registers: 16 words per column.  Per row and column: 16 dp4a on
// the unsigned 6-bit codes, then
//   y += u * d * (sc_a * (254*H_a + L_a - 32*XS_a) + sc_b * (...)_b)
// with XS the run's sum of 254*xh + xl (the code offset of 32), made once
// per call.  A warp covers four super-blocks; G warps a row (partials added
// in shared memory in segment order); four rows per iteration are reduced by
// one transposed shuffle tree.  Rows must be whole multiples of 16 bytes
// (k a multiple of 2048).
namespace rows6 {
// consumer warps: 16 at two columns (544 threads: 96 registers each), 15 at
// four (512 threads: 128 registers, which the four columns' 72 limb words need)
template <int NB> constexpr int cw() { return NB == 2 ? 16 : 15; }
template <int NB> constexpr int threads() { return (cw<NB>() + 1) * 32; }
constexpr int MAX_STAGES = 8;
constexpr int kStatic = 512;
constexpr int LPB = 8;                       // lanes per super-block
constexpr int KW = 32 / LPB;                 // super-blocks per warp
constexpr int BB = 210;                      // bytes per super-block
using rowsnb::Params;
using rowsnb::col_bytes;

inline int segments(int64_t k) { return (int)((k / 256 + KW - 1) / KW); }
template <int NB> inline int red_bytes(const Params &p) {
    return p.G > 1 ? (p.rows_cap * p.G * NB * 4 + 15) / 16 * 16 : 0;
}

template <int NB> inline bool plan(int64_t k, int64_t n_out, int grid, Params &p) {
    if (k % 2048 || grid < 1 || n_out < 1) return false;
    const int G = segments(k);
    if (G < 1 || G > cw<NB>()) return false;
    p.G = G;
    p.NG = cw<NB>() / G;
    p.RS = 2 * p.NG;
    p.rows_cap = (int)((n_out + grid - 1) / grid);
    const int64_t stage = (int64_t)p.RS * (k / 256) * BB;
    const int64_t avail = kSmemBudget - kStatic - (int64_t)NB * col_bytes(k) - rows6::red_bytes<NB>(p);
    int64_t ns = avail / stage;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    p.nstages = (int)ns;
    return ns >= 2;
}

template <int NB>
__global__ void __launch_bounds__(threads<NB>(), 1) gemv_q6_k_nb(Params p) {
    constexpr int CW = cw<NB>();
    constexpr int V = 4 * NB;                // values per lane per iteration (4 rows x NB columns)
    constexpr int LOGV = NB == 2 ? 3 : 4;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t x_bar;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int S = p.k / 64;
    const int CB = col_bytes(p.k);
    const uint32_t rowbytes = (uint32_t)nb * (uint32_t)BB;
    const int G = p.G, NG = p.NG, RS = p.RS, CA = G * NG;
    const int64_t r0 = (int64_t)p.n_out * blockIdx.x / gridDim.x;
    const int nrows = (int)((int64_t)p.n_out * (blockIdx.x + 1) / gridDim.x - r0);
    const int units = (nrows + RS - 1) / RS;
    const int NS = p.nstages;
    const uint32_t stage_bytes = (uint32_t)RS * rowbytes;
    uint8_t *ximg = smem + (size_t)NS * stage_bytes;            // NB columns of CB bytes
    float *red = reinterpret_cast<float *>(ximg + (size_t)NB * CB);
    const uint32_t ring_s = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CA);
        }
        mbar_init(&x_bar, 1);
        fence_mbar_init();
    }
    rowk::grid_dep_launch();
    __syncthreads();

    if (warp == CW) {
        // ---------------- producer: one contiguous copy per stage ----------------
        if (lane == 0) {
            // as in rowsnb::gemv_rows_nb: with the x image from prep_x_nb, the
            // first ring's worth of weights, then the image; with x converted
            // here, a window of stages until the consumers have converted it
            const bool img = p.x_img != nullptr;
            if (!img && !p.early_w) rowk::grid_dep_wait();   // the weights may be the previous kernel's output
            const int cap = img ? NS : (rowsnb::kNbXWindow < NS ? rowsnb::kNbXWindow : NS);
            const int early = units < cap ? units : cap;
            const uint64_t pol = make_evict_first_policy();
            const uint8_t *src = p.w + r0 * (int64_t)rowbytes;
            int slot = 0;
            uint32_t ph = 0;
            for (int u = 0; u <= units; ++u) {
                if (u == early) {
                    if (img) {
                        rowk::grid_dep_wait();
                        mbar_arrive_expect_tx(&x_bar, (uint32_t)(NB * CB));
                        bulk_g2s(ximg, p.x_img, (uint32_t)(NB * CB), &x_bar);
                    } else if (u < units && !mbar_wait(&x_bar, 0)) {
                        break;
                    }
                }
                if (u == units) break;
                const int rows = nrows - u * RS < RS ? nrows - u * RS : RS;
                const uint32_t bytes = (uint32_t)rows * rowbytes;
                if (!mbar_wait(&empty_bar[slot], ph ^ 1u)) break;
                mbar_arrive_expect_tx(&full_bar[slot], bytes);
                bulk_g2s_hint(smem + (size_t)slot * stage_bytes, src, bytes, &full_bar[slot], pol);
                src += (size_t)RS * rowbytes;
                if (++slot == NS) { slot = 0; ph ^= 1u; }
            }
        }
        return;
    }

    bool dead = false;   // a wait ran out: stop waiting, keep going so every warp finishes
    if (p.x_img) {
        if (warp >= CA) return;
        if (!mbar_wait(&x_bar, 0)) dead = true;
    } else {
        rowk::grid_dep_wait();                   // x may be the previous kernel's output
#pragma unroll
        for (int b = 0; b < NB; ++b)
            prep_x_all(b < p.nb_cols ? p.x + (size_t)b * p.k : nullptr, ximg + (size_t)b * CB,
                       ximg + (size_t)b * CB + 2 * p.k, nb, S, warp, CW, lane);
        named_sync(1, CW * 32);
        if (threadIdx.x == 0) mbar_arrive(&x_bar);   // the producer may stream past its window
        if (warp >= CA) return;
    }

    const int gi = warp / G, seg = warp - gi * G;
    const int part = lane % LPB;
    const int h = part >> 2, t = (part >> 1) & 1, j = part & 1;
    // a warp takes four blocks of one parity (segment pair sp covers blocks
    // 8sp..8sp+7): blocks 2 apart start 420 bytes apart, one bank group
    // further, so the 32 lanes' word loads fall in 32 different banks
    const int kb = 8 * (seg >> 1) + 2 * (lane / LPB) + (seg & 1);
    const bool valid = kb < nb;
    const int kbc = valid ? kb : nb - 1;       // idle lanes read a real block, weight 0
    const int sl = 4 * kbc + 2 * h;            // image slice of run t (run t + 2: sl + 1)
    const int ga = 2 * t + j;                  // 16-byte group of the run's xh (xl: ga + 4)

    uint32_t xah[NB][4], xal[NB][4], xbh[NB][4], xbl[NB][4];
    int nxa[NB], nxb[NB];                      // -32 * XS of the two runs
    float u[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const uint8_t *img = ximg + (size_t)b * CB;
        const uint4 ah = *reinterpret_cast<const uint4 *>(img + (ga * S + sl) * 16);
        const uint4 al = *reinterpret_cast<const uint4 *>(img + ((ga + 4) * S + sl) * 16);
        const uint4 bh = *reinterpret_cast<const uint4 *>(img + (ga * S + sl + 1) * 16);
        const uint4 bl = *reinterpret_cast<const uint4 *>(img + ((ga + 4) * S + sl + 1) * 16);
        xah[b][0] = ah.x; xah[b][1] = ah.y; xah[b][2] = ah.z; xah[b][3] = ah.w;
        xal[b][0] = al.x; xal[b][1] = al.y; xal[b][2] = al.z; xal[b][3] = al.w;
        xbh[b][0] = bh.x; xbh[b][1] = bh.y; xbh[b][2] = bh.z; xbh[b][3] = bh.w;
        xbl[b][0] = bl.x; xbl[b][1] = bl.y; xbl[b][2] = bl.z; xbl[b][3] = bl.w;
        int sah = 0, sal = 0, sbh = 0, sbl = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sah = dp4a_ss(xah[b][i], 0x01010101u, sah);
            sal = dp4a_ss(xal[b][i], 0x01010101u, sal);
            sbh = dp4a_ss(xbh[b][i], 0x01010101u, sbh);
            sbl = dp4a_ss(xbl[b][i], 0x01010101u, sbl);
        }
        nxa[b] = -32 * (254 * sah + sal);
        nxb[b] = -32 * (254 * sbh + sbl);
        const uint8_t *meta = img + 2 * p.k;
        u[b] = valid ? *reinterpret_cast<const float *>(meta + sl * 16 + 8) : 0.f;
    }

    // the block starts 2-byte aligned: word loads from the aligned address
    // below it, realigned with one byte permute per word
    const uint32_t blk0 = ring_s + (uint32_t)kbc * (uint32_t)BB;
    const uint32_t delta = blk0 & 2u;
    const uint32_t sel = delta ? 0x5432u : 0x3210u;
    const uint32_t dsh = delta ? 16u : 0u;
    const uint32_t lane_a = blk0 - delta;
    const uint32_t oql = (uint32_t)(64 * h + 32 * t + 16 * j);
    const uint32_t oqh = (uint32_t)(128 + 32 * h + 16 * j);
    const uint32_t osc = (uint32_t)(192 + 8 * h + 2 * t + j) + delta;
    const int sa = 4 - 2 * t, sb = 2 * t;

    // products of one row (block at aligned shared address a) with all NB columns
    auto row_dot = [&](uint32_t a, float (&out)[NB]) {
        uint32_t ql[4], qh[4];
        {
            uint32_t w[5], v[5];
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                w[i] = rowk::lds32(a + oql + 4u * (uint32_t)i);
                v[i] = rowk::lds32(a + oqh + 4u * (uint32_t)i);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ql[i] = __byte_perm(w[i], w[i + 1], sel);
                qh[i] = __byte_perm(v[i], v[i + 1], sel);
            }
        }
        int sc_a, sc_b;
        asm volatile("ld.shared.s8 %0, [%1];" : "=r"(sc_a) : "r"(a + osc));
        asm volatile("ld.shared.s8 %0, [%1];" : "=r"(sc_b) : "r"(a + osc + 4u));
        const float d = h2f(rowk::lds32(a + 208u) >> dsh);
        const float dsa = d * (float)sc_a, dsb = d * (float)sc_b;
        uint32_t qa[4], qb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qa[i] = (ql[i] & 0x0F0F0F0Fu) | ((qh[i] << sa) & 0x30303030u);
            qb[i] = ((ql[i] >> 4) & 0x0F0F0F0Fu) | ((qh[i] >> sb) & 0x30303030u);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            int Ha = 0, La = nxa[b], Hb = 0, Lb = nxb[b];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                Ha = dp4a_us(qa[i], xah[b][i], Ha);
                La = dp4a_us(qa[i], xal[b][i], La);
                Hb = dp4a_us(qb[i], xbh[b][i], Hb);
                Lb = dp4a_us(qb[i], xbl[b][i], Lb);
            }
            // |254 H + L| < 2^26: exact in int32
            const int Da = 254 * Ha + La, Db = 254 * Hb + Lb;
            out[b] = u[b] * fmaf(dsa, (float)Da, dsb * (float)Db);
        }
    };

    const uint32_t rA0 = (uint32_t)gi * rowbytes, rA1 = (uint32_t)(gi + NG) * rowbytes;
    constexpr int SHIFT = 5 - LOGV;                    // lane >> SHIFT = value index after the tree
    const int my_v = lane >> SHIFT;
    const int my_t = my_v / NB, my_b = my_v % NB;      // row slot (0,1 stage A; 2,3 stage B), column
    const int my_rowoff = gi + ((my_t & 1) ? NG : 0);

    int slot = 0;
    uint32_t ph = 0;
    for (int uu = 0; uu < units; uu += 2) {
        const bool hasB = uu + 1 < units;
        const int slotA = slot;
        const uint32_t phA = ph;
        if (++slot == NS) { slot = 0; ph ^= 1u; }
        const int slotB = slot;
        const uint32_t phB = ph;
        if (hasB) {
            if (++slot == NS) { slot = 0; ph ^= 1u; }
        }
        const int nA = nrows - uu * RS < RS ? nrows - uu * RS : RS;
        const int nB = hasB ? (nrows - (uu + 1) * RS < RS ? nrows - (uu + 1) * RS : RS) : 0;
        float v[V];
        float tmp[NB];
        if (!dead && !mbar_wait(&full_bar[slotA], phA)) dead = true;
        {
            const uint32_t sA = lane_a + (uint32_t)slotA * stage_bytes;
            row_dot(sA + rA0, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[b] = gi < nA ? tmp[b] : 0.f;
            row_dot(sA + rA1, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[NB + b] = gi + NG < nA ? tmp[b] : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slotA]);
        if (hasB && !dead && !mbar_wait(&full_bar[slotB], phB)) dead = true;
        {
            const uint32_t sB = lane_a + (uint32_t)slotB * stage_bytes;
            row_dot(sB + rA0, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[2 * NB + b] = gi < nB ? tmp[b] : 0.f;
            row_dot(sB + rA1, tmp);
#pragma unroll
            for (int b = 0; b < NB; ++b) v[3 * NB + b] = gi + NG < nB ? tmp[b] : 0.f;
        }
        __syncwarp();
        if (lane == 0 && hasB) mbar_arrive(&empty_bar[slotB]);
        const float tot = rowsnb::transposed_sum<V, LOGV>(v, lane);
        if ((lane & ((1 << SHIFT) - 1)) == 0 && my_b < p.nb_cols) {
            const int n_here = my_t >= 2 ? nB : nA;
            if (my_rowoff < n_here) {
                const int row = (uu + (my_t >= 2 ? 1 : 0)) * RS + my_rowoff;   // relative to r0
                if (G == 1)
                    p.y[(size_t)my_b * p.ldy + r0 + row] = tot;
                else
                    red[((size_t)row * G + seg) * NB + my_b] = tot;
            }
        }
    }
    if (G > 1) {
        named_sync(2, CA * 32);
        for (int i = warp * 32 + lane; i < nrows * NB; i += CA * 32) {
            const int row = i / NB, b = i % NB;
            if (b >= p.nb_cols) continue;
            float sum = red[((size_t)row * G) * NB + b];
            for (int g2 = 1; g2 < G; ++g2) sum += red[((size_t)row * G + g2) * NB + b];
            p.y[(size_t)b * p.ldy + r0 + row] = sum;
        }
    }
}

template <int NB>
cudaError_t launch(const uint8_t *w, int64_t n_out, int64_t k, const float *x, int nb_cols, float *y, int64_t ldy,
                   int grid, cudaStream_t s) {
    Params p{w, nullptr, x, y, (long long)ldy, (int)n_out, (int)k, nb_cols, 0, 0, 0, 0, 0, weight_prefetch()};
    if (!rows6::plan<NB>(k, n_out, grid, p)) return cudaErrorInvalidValue;
    const int smem = p.nstages * p.RS * (int)(k / 256) * BB + NB * col_bytes(k) + rows6::red_bytes<NB>(p);
    static PerDeviceOnce configured;
    const cudaError_t ce = configured.run([] {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, gemv_q6_k_nb<NB>);
        if (e != cudaSuccess) return e;
        if (fa.sharedSizeBytes > (size_t)kStatic) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(gemv_q6_k_nb<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBudget - kStatic);
    });
    if (ce != cudaSuccess) return ce;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (NB == 2 && k <= rowsnb::kNbConvertMaxK) {
        // x converted by the kernel itself (two columns: Q6_K head 83.5 -> 80.7
        // us, 4096x14336 17.4 -> 16.3 us; four columns convert more slowly than
        // prep_x_nb: 2000x4096 batch 3 9.1 -> 10.1 us, so they keep it)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads<NB>());
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_q6_k_nb<NB>, p);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    cudaMemPool_t pool = scratch_pool();
    if (!pool) return cudaErrorMemoryAllocation;
    void *img = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&img, (size_t)NB * col_bytes(k), pool, s);
    if (e != cudaSuccess) return e;
    p.x_img = static_cast<const uint8_t *>(img);
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3((unsigned)((k / 256 + 7) / 8), NB);
    pcfg.blockDim = dim3(256);
    pcfg.stream = s;
    pcfg.attrs = attr;
    pcfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&pcfg, rowsnb::prep_x_nb<NB>, x, (int)k, nb_cols, static_cast<uint8_t *>(img));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads<NB>());
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gemv_q6_k_nb<NB>, p);
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    const cudaError_t f = cudaFreeAsync(img, s);
    return e != cudaSuccess ? e : f;
}

// Whether this kernel runs Q6_K (k, n_out) at `batch` (2-4) columns.
inline bool takes(int64_t k, int64_t n_out, int batch) {
    Params p{};
    const int grid_est = 132;      // fewer SMs than any sm_103 part: a conservative row count
    const int grid = (int)(n_out < grid_est ? n_out : grid_est);
    if (batch < 2 || batch > 4 || k > (INT64_C(1) << 20)) return false;
    return batch == 2 ? rows6::plan<2>(k, n_out, grid, p) : rows6::plan<4>(k, n_out, grid, p);
}
}  // namespace rows6

// ---------------------------------------------------------------------------
// Q4_K and Q6_K at batch 3-8 for k = 4096 (the decode layer's QKV, O,
// gate+up and 14336-row shapes, and the output head): the products on
// mma.sync (m16n8k16, fp16 in, f32 accumulate) with both operands in
// registers, one launch per call.
//
// Stages are runs of 16 whole rows (one bulk copy per row, rows PITCH bytes
// apart so that the eight rows a warp's lanes read fall in different
// shared-memory banks).  Warp w of the 16 owns super-block w of every row: a
// K range of 256 = 16 MMA steps of 16 positions.
//   B (x): built once per call by each warp for its own super-block: the hi
//     and lo fp16 halves of x' = 2^e x (e per super-block and column, see
//     tc_scale_exponent); per 8 MMA columns (4 x columns x {hi, lo}) a thread
//     holds its 4 positions of every step in 32 registers.
//   A (weights): rows g and g+8 of the stage, positions 4i..4i+3 of the step
//     (lane = 4g + i), in the K slot order of the B fragment.
//   The 16 warps' sums of a stage are added in warp order through shared
//   memory after one barrier (by warps 0-1); after it the last warp's first
//   thread refills the stage's ring slot, which no warp reads any more.
namespace rmma {
constexpr int CWARPS = 16;
constexpr int THREADS = CWARPS * 32;
constexpr int RS = 16;                       // rows per stage
constexpr int K = 4096;

struct Params {
    const uint8_t *w;
    const float *x;
    float *y;
    long long ldy;
    int n_out;
    int nb_cols;     // real columns (the others are zero)
    int early_w;     // stream weights before waiting on the previous kernel
    int epi;         // kEpiNone, kEpiBias (bias[n_out]) or kEpiSwiGLU (n_out = 2 * pairs, gate rows first)
    const float *bias;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma16816_acc(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// two bytes of v chosen by sel (byte_perm nibbles i, 4, j, 4) as the fp16 pair
// (v_i - off, v_j - off): 0x64 above a byte is the fp16 1024 + byte, and the
// subtraction of OFF (an fp16 pair, 1024 + off) is exact
template <uint32_t OFF>
__device__ __forceinline__ uint32_t bytes_h2(uint32_t v, uint32_t sel) {
    const uint32_t p = __byte_perm(v, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(OFF));
    return r;
}
__host__ __device__ constexpr uint32_t pair_sel(uint32_t i, uint32_t j) { return i | 0x40u | (j << 8) | 0x4000u; }

// Stage u (rows_u rows) of this CTA into ring slot `slot`.
template <int ROWB, int PITCH, int STAGE>
__device__ __forceinline__ void issue_stage(uint8_t *smem, uint64_t *full, const uint8_t *src, int rows,
                                            uint64_t pol) {
    mbar_arrive_expect_tx(full, (uint32_t)rows * ROWB);
    for (int r = 0; r < rows; ++r)
        bulk_g2s_hint(smem + (size_t)r * PITCH, src + (size_t)r * ROWB, (uint32_t)ROWB, full, pol);
}

// B fragments of x columns 4t..4t+3 for this warp's super-block (see above);
// optionally the sub-block sums of x' as the fp16 B fragment of the mins
// product (K slots 2i, 2i+1 = sub-blocks 2i, 2i+1).  undo: 2^-e of the
// thread's C column 4t + i.
// The two lanes of a column (hi and lo part, lanes 4g+i and 4(g^1)+i) each
// load half of the column's steps (the hi lane steps 0-7, the lo lane 8-15),
// split their values into both halves, and swap the halves the other needs:
// x is read once per CTA.
template <bool XSUMS>
__device__ __forceinline__ void build_x(const Params &p, int t, int warp, int lane, uint32_t (&xb)[16][2],
                                        uint32_t &xsb, float &undo) {
    const int g = lane >> 2, i4 = lane & 3;
    const int col = 4 * t + (g >> 1);
    const bool lo_part = g & 1;
    const int s0 = lo_part ? 8 : 0;              // the steps this lane loads
    float v[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < p.nb_cols) a = ldg_f4(p.x + (size_t)col * K + warp * 256 + 16 * (s0 + s) + 4 * i4);
        v[s][0] = a.x; v[s][1] = a.y; v[s][2] = a.z; v[s][3] = a.w;
    }
    float m = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fabsf(v[s][j]));
    // NaN never wins fmaxf; a NaN anywhere still reaches y through the products
    uint32_t mb = __float_as_uint(m);
    // the column's eight lanes (4 position groups x the two halves of its steps)
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
    const int e = tc_scale_exponent(mb);
    const float mult = __uint_as_float((uint32_t)(127 + e) << 23);
    const float und = __uint_as_float((uint32_t)(127 - e) << 23);
    float xs[4] = {0.f, 0.f, 0.f, 0.f};          // sums over this lane's part of sub-blocks s0/2 .. s0/2+3
    uint32_t own[8][2], other[8][2];             // this lane's half / the partner's half of the loaded steps
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        float sx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) sx[j] = v[s][j] * mult;
        if (XSUMS) xs[s >> 1] += (sx[0] + sx[1]) + (sx[2] + sx[3]);
        // positions (0, 1) and (2, 3) as fp16 pairs (K slots 2i, 2i+1 and
        // 2i+8, 2i+9): hi parts, then the rest
        const __half2 h01 = __floats2half2_rn(sx[0], sx[1]), h23 = __floats2half2_rn(sx[2], sx[3]);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(sx[0] - f01.x, sx[1] - f01.y);
        const __half2 l23 = __floats2half2_rn(sx[2] - f23.x, sx[3] - f23.y);
        const uint32_t hb0 = *reinterpret_cast<const uint32_t *>(&h01), hb1 = *reinterpret_cast<const uint32_t *>(&h23);
        const uint32_t lb0 = *reinterpret_cast<const uint32_t *>(&l01), lb1 = *reinterpret_cast<const uint32_t *>(&l23);
        own[s][0] = lo_part ? lb0 : hb0;
        own[s][1] = lo_part ? lb1 : hb1;
        other[s][0] = lo_part ? hb0 : lb0;
        other[s][1] = lo_part ? hb1 : lb1;
    }
    // the partner (lane ^ 4) loaded the other eight steps: swap
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint32_t r0 = __shfl_xor_sync(0xffffffffu, other[s][0], 4);
        const uint32_t r1 = __shfl_xor_sync(0xffffffffu, other[s][1], 4);
        // (register indices must be static: select instead of indexing by s0)
        xb[s][0] = lo_part ? r0 : own[s][0];
        xb[s][1] = lo_part ? r1 : own[s][1];
        xb[8 + s][0] = lo_part ? own[s][0] : r0;
        xb[8 + s][1] = lo_part ? own[s][1] : r1;
    }
    if (XSUMS) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            xs[j] += __shfl_xor_sync(0xffffffffu, xs[j], 1);
            xs[j] += __shfl_xor_sync(0xffffffffu, xs[j], 2);
        }
        // sub-blocks 2i, 2i+1: on the hi lane (sub-blocks 0-3) for i < 2, the
        // lo lane (4-7) for i >= 2; |x'| < 2^10, so a sum of 32 fits fp16
        const int jj = 2 * (i4 & 1);
        const float a0 = jj ? xs[2] : xs[0], a1 = jj ? xs[3] : xs[1];
        const int src = 4 * ((g & ~1) + (i4 >> 1)) + i4;
        const float xa = __shfl_sync(0xffffffffu, a0, src), xc = __shfl_sync(0xffffffffu, a1, src);
        const __half2 hp = __floats2half2_rn(xa, xc);
        const float2 fp = __half22float2(hp);
        const __half2 lp = __floats2half2_rn(xa - fp.x, xc - fp.y);
        xsb = lo_part ? *reinterpret_cast<const uint32_t *>(&lp) : *reinterpret_cast<const uint32_t *>(&hp);
    }
    // the C columns of this thread are 2i (hi) and 2i+1 (lo): x column 4t + i
    undo = __shfl_sync(0xffffffffu, und, 8 * i4);
}

// Format policies: ROWB bytes per row, the ring depth for NT B tiles, and the
// products of one stage for this warp's super-block (rows g, g+8 at aligned
// shared addresses ra, rb), giving v[t][0..1] = y parts of rows g, g+8.
struct Q4 {
    // stages per CTA barrier (the partial sums of SPS stages are added after
    // one barrier): 2 (14336x4096 batch 8 15.4 -> 14.8 us; batch 2 9.81 ->
    // 9.52 us once the decode had become cheaper)
    template <int NT> static constexpr int sps() { return 2; }
    static constexpr int ROWB = (K / 256) * 144;          // 2304
    static constexpr int PITCH = ROWB + 16;
    static constexpr bool XSUMS = true;
    template <int NT> static constexpr int stages() { return 5; }
    // The code bytes (low nibbles, sub-block 2c; high nibbles shifted down,
    // sub-block 2c+1) become q * 2^-9 through the e4m3 conversion; at 8
    // columns times sc * 2^9 (an fp16 integer, at most 32256), so that A is
    // sc*q exactly (<= 945, an fp16 integer); at 4 columns sc multiplies the
    // sub-block's f32 sums.  The mins through one product of the 6-bit mins
    // with the sub-block sums; y += 2^-e * (d * (A.x') - dmin * (m.XS'))
    template <int NT>
    static __device__ __forceinline__ void stage(uint32_t ra, uint32_t rb, int warp, int lane,
                                                 const uint32_t (&xb)[NT][16][2], const uint32_t (&xsb)[NT],
                                                 const float (&undo)[NT], float (&v)[NT][2]) {
        (void)warp;
        const int i4 = lane & 3;
        const uint4 ha = lds128(ra), hb = lds128(rb);
        const uint32_t sca[2] = {ha.y & 0x3F3F3F3Fu, (ha.w & 0x0F0F0F0Fu) | ((ha.y >> 2) & 0x30303030u)};
        const uint32_t scb[2] = {hb.y & 0x3F3F3F3Fu, (hb.w & 0x0F0F0F0Fu) | ((hb.y >> 2) & 0x30303030u)};
        float c[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) c[t][0] = c[t][1] = c[t][2] = c[t][3] = 0.f;
        if constexpr (NT == 1) {
            // 4 columns: each sub-block's two MMAs on the unscaled codes into
            // their own f32 sums, scaled by sc in f32 afterwards (no fp16
            // multiplies; 14336x4096 batch 2 / 4 10.14 / 10.55 -> 9.82 / 10.32
            // us).  The 8-column instance has no registers for those sums.
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint32_t sw = (uint32_t)(2 * (cc & 1));
                // 6-bit scales as f32: the byte under the exponent bits of 2^23, minus 2^23
                const float fla = __uint_as_float(__byte_perm(sca[cc >> 1], 0x4B000000u, 0x7650u | sw)) - 8388608.0f;
                const float fha = __uint_as_float(__byte_perm(sca[cc >> 1], 0x4B000000u, 0x7650u | (sw + 1))) - 8388608.0f;
                const float flb = __uint_as_float(__byte_perm(scb[cc >> 1], 0x4B000000u, 0x7650u | sw)) - 8388608.0f;
                const float fhb = __uint_as_float(__byte_perm(scb[cc >> 1], 0x4B000000u, 0x7650u | (sw + 1))) - 8388608.0f;
                float cl[NT][4], ch[NT][4];
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const uint32_t off = 16u + 32u * cc + 16u * pp + 4u * i4;
                    const uint32_t wa = rowk::lds32(ra + off), wb = rowk::lds32(rb + off);
                    uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
                    nibble_bytes_h2(wa & 0x0F0F0F0Fu, l0, l2);
                    nibble_bytes_h2(wb & 0x0F0F0F0Fu, l1, l3);
                    nibble_bytes_h2((wa >> 4) & 0x0F0F0F0Fu, h0, h2);
                    nibble_bytes_h2((wb >> 4) & 0x0F0F0F0Fu, h1, h3);
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (pp == 0) {
                            mma16816(cl[t], l0, l1, l2, l3, xb[t][4 * cc + pp][0], xb[t][4 * cc + pp][1]);
                            mma16816(ch[t], h0, h1, h2, h3, xb[t][4 * cc + pp + 2][0], xb[t][4 * cc + pp + 2][1]);
                        } else {
                            mma16816_acc(cl[t], l0, l1, l2, l3, xb[t][4 * cc + pp][0], xb[t][4 * cc + pp][1]);
                            mma16816_acc(ch[t], h0, h1, h2, h3, xb[t][4 * cc + pp + 2][0], xb[t][4 * cc + pp + 2][1]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    c[t][0] = fmaf(fla, cl[t][0], fmaf(fha, ch[t][0], c[t][0]));
                    c[t][1] = fmaf(fla, cl[t][1], fmaf(fha, ch[t][1], c[t][1]));
                    c[t][2] = fmaf(flb, cl[t][2], fmaf(fhb, ch[t][2], c[t][2]));
                    c[t][3] = fmaf(flb, cl[t][3], fmaf(fhb, ch[t][3], c[t][3]));
                }
            }
        } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint32_t sw = (uint32_t)(2 * (cc & 1));
                // (sc * 2^9) pairs of sub-blocks 2c (l) and 2c+1 (h) of rows a, b
                const uint32_t Sla = hmul2_bits(bytes_h2<0x64006400u>(sca[cc >> 1], pair_sel(sw, sw)), 0x60006000u);
                const uint32_t Slb = hmul2_bits(bytes_h2<0x64006400u>(scb[cc >> 1], pair_sel(sw, sw)), 0x60006000u);
                const uint32_t Sha = hmul2_bits(bytes_h2<0x64006400u>(sca[cc >> 1], pair_sel(sw + 1, sw + 1)), 0x60006000u);
                const uint32_t Shb = hmul2_bits(bytes_h2<0x64006400u>(scb[cc >> 1], pair_sel(sw + 1, sw + 1)), 0x60006000u);
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const uint32_t off = 16u + 32u * cc + 16u * pp + 4u * i4;
                    const uint32_t wa = rowk::lds32(ra + off), wb = rowk::lds32(rb + off);
                    // positions 4i, 4i+1 (l0, l1, h0, h1) and 4i+2, 4i+3 (l2, l3, h2, h3)
                    uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
                    nibble_bytes_h2(wa & 0x0F0F0F0Fu, l0, l2);
                    nibble_bytes_h2(wb & 0x0F0F0F0Fu, l1, l3);
                    nibble_bytes_h2((wa >> 4) & 0x0F0F0F0Fu, h0, h2);
                    nibble_bytes_h2((wb >> 4) & 0x0F0F0F0Fu, h1, h3);
                    l0 = hmul2_bits(l0, Sla); l2 = hmul2_bits(l2, Sla);
                    l1 = hmul2_bits(l1, Slb); l3 = hmul2_bits(l3, Slb);
                    h0 = hmul2_bits(h0, Sha); h2 = hmul2_bits(h2, Sha);
                    h1 = hmul2_bits(h1, Shb); h3 = hmul2_bits(h3, Shb);
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        mma16816_acc(c[t], l0, l1, l2, l3, xb[t][4 * cc + pp][0], xb[t][4 * cc + pp][1]);
                        mma16816_acc(c[t], h0, h1, h2, h3, xb[t][4 * cc + pp + 2][0], xb[t][4 * cc + pp + 2][1]);
                    }
                }
            }
        }
        const float cfix = NT == 1 ? 512.0f : 1.0f;   // the codes' 2^-9 (4 columns: not in the scales)
        // mins: K slots 2i, 2i+1 = sub-blocks 2i, 2i+1 of rows g, g+8
        const uint32_t mwa = (i4 >> 1) ? (((ha.w >> 4) & 0x0F0F0F0Fu) | ((ha.z >> 2) & 0x30303030u)) : (ha.z & 0x3F3F3F3Fu);
        const uint32_t mwb = (i4 >> 1) ? (((hb.w >> 4) & 0x0F0F0F0Fu) | ((hb.z >> 2) & 0x30303030u)) : (hb.z & 0x3F3F3F3Fu);
        const uint32_t ms = (uint32_t)(2 * (i4 & 1));
        const uint32_t ma = bytes_h2<0x64006400u>(mwa, pair_sel(ms, ms + 1));
        const uint32_t mbb = bytes_h2<0x64006400u>(mwb, pair_sel(ms, ms + 1));
        const float da = h2f(ha.x), dma = h2f(ha.x >> 16), db = h2f(hb.x), dmb = h2f(hb.x >> 16);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float cm[4];
            mma16816(cm, ma, mbb, 0u, 0u, xsb[t], 0u);
            v[t][0] = undo[t] * fmaf(da * cfix, c[t][0] + c[t][1], -dma * (cm[0] + cm[1]));
            v[t][1] = undo[t] * fmaf(db * cfix, c[t][2] + c[t][3], -dmb * (cm[2] + cm[3]));
        }
    }
};

struct Q6 {
    template <int NT> static constexpr int sps() { return 1; }   // 2 at 8 columns: head 112 -> 115 us
    static constexpr int ROWB = (K / 256) * 210;          // 3360
    static constexpr int PITCH = ROWB + 16;
    static constexpr bool XSUMS = false;
    template <int NT> static constexpr int stages() { return NT == 1 ? 4 : 3; }
    // q - 32 exact from the ql nibble and the qh bit pair; a step is one
    // 16-weight sub-block, so each product is scaled by its signed 8-bit
    // scale as it is added; y += 2^-e * d * sum(sc * (A.x'))
    template <int NT>
    static __device__ __forceinline__ void stage(uint32_t ra, uint32_t rb, int warp, int lane,
                                                 const uint32_t (&xb)[NT][16][2], const uint32_t (&xsb)[NT],
                                                 const float (&undo)[NT], float (&v)[NT][2]) {
        (void)xsb;
        const int i4 = lane & 3;
        // the super-block starts 2-byte aligned (ra, rb are the aligned
        // addresses below it): word loads realigned by one byte permute
        const uint32_t delta = ((uint32_t)warp * 210u) & 2u;
        const uint32_t sel = delta ? 0x5432u : 0x3210u;
        auto ldw = [&](uint32_t a) { return __byte_perm(rowk::lds32(a), rowk::lds32(a + 4u), sel); };
        uint32_t sc0[4], sc1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sc0[j] = ldw(ra + 192u + 4u * j);
            sc1[j] = ldw(rb + 192u + 4u * j);
        }
        const float d0 = h2f(rowk::lds32(ra + 208u) >> (delta ? 16u : 0u));
        const float d1 = h2f(rowk::lds32(rb + 208u) >> (delta ? 16u : 0u));
        float acc[NT][2];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int sp = 0; sp < 2; ++sp) {
                const uint32_t oh = 128u + 32u * h + 16u * sp + 4u * i4;
                const uint32_t qh0 = ldw(ra + oh), qh1 = ldw(rb + oh);
#pragma unroll
                for (int t1 = 0; t1 < 2; ++t1) {
                    const uint32_t ol = 64u * h + 32u * t1 + 16u * sp + 4u * i4;
                    const uint32_t ql0 = ldw(ra + ol), ql1 = ldw(rb + ol);
#pragma unroll
                    for (int hn = 0; hn < 2; ++hn) {
                        const int r = t1 + 2 * hn;                      // run 0..3 of the half
                        const int s = 8 * h + 2 * r + sp;               // step = scale index
                        const uint32_t lo0 = (hn ? (ql0 >> 4) : ql0) & 0x0F0F0F0Fu;
                        const uint32_t lo1 = (hn ? (ql1 >> 4) : ql1) & 0x0F0F0F0Fu;
                        const uint32_t hb0 = (r < 3 ? (qh0 << (4 - 2 * r)) : (qh0 >> 2)) & 0x30303030u;
                        const uint32_t hb1 = (r < 3 ? (qh1 << (4 - 2 * r)) : (qh1 >> 2)) & 0x30303030u;
                        const uint32_t q0 = lo0 | hb0, q1 = lo1 | hb1;
                        // (q - 32) pairs: subtract the fp16 1056 = 1024 + 32
                        const uint32_t a0 = bytes_h2<0x64206420u>(q0, pair_sel(0, 1));
                        const uint32_t a1 = bytes_h2<0x64206420u>(q1, pair_sel(0, 1));
                        const uint32_t a2 = bytes_h2<0x64206420u>(q0, pair_sel(2, 3));
                        const uint32_t a3 = bytes_h2<0x64206420u>(q1, pair_sel(2, 3));
                        const float sa = (float)(int)(int8_t)(sc0[s >> 2] >> (8 * (s & 3)));
                        const float sb = (float)(int)(int8_t)(sc1[s >> 2] >> (8 * (s & 3)));
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            float c[4];
                            mma16816(c, a0, a1, a2, a3, xb[t][s][0], xb[t][s][1]);
                            acc[t][0] = fmaf(sa, c[0] + c[1], acc[t][0]);
                            acc[t][1] = fmaf(sb, c[2] + c[3], acc[t][1]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            v[t][0] = d0 * undo[t] * acc[t][0];
            v[t][1] = d1 * undo[t] * acc[t][1];
        }
    }
};

template <class F, int NT> constexpr int stage_bytes() { return RS * F::PITCH; }
// partial-sum buffers: two groups of SPS stages, 16 warps x 16 rows x NB columns each
template <int NT, int SPS = 1> constexpr int red_floats() { return 2 * SPS * CWARPS * RS * 4 * NT; }
template <class F, int NT> constexpr int smem_bytes() {
    return F::template stages<NT>() * stage_bytes<F, NT>() + red_floats<NT, F::template sps<NT>()>() * 4 + 128;
}
static_assert(smem_bytes<Q4, 2>() <= kSmemBudget - 512 && smem_bytes<Q6, 1>() <= kSmemBudget - 512 &&
                  smem_bytes<Q6, 2>() <= kSmemBudget - 512,
              "shared memory per CTA");

// With 4 columns (NT = 1) a producer warp streams the stages, released by
// per-slot empty barriers, and the block has 17 warps (96 registers each);
// with 8 (NT = 2) the x fragments need 128 registers, so the block has the
// 16 compute warps only and a thread of the last warp refills each slot
// after the stage's barrier.
template <int NT> constexpr bool has_producer() { return NT == 1; }
template <int NT> constexpr int block_threads() { return has_producer<NT>() ? THREADS + 32 : THREADS; }

template <class F, int NT>
__global__ void __launch_bounds__(block_threads<NT>(), 1) gemv_rows_mma(Params p) {
    constexpr int NS = F::template stages<NT>();
    constexpr int STAGE = stage_bytes<F, NT>();
    constexpr int NB = 4 * NT;                   // x columns
    constexpr bool PROD = has_producer<NT>();
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[NS], empty_bar[NS];
    float *red = reinterpret_cast<float *>(smem + NS * STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, i4 = lane & 3;
    // items: rows, or for SwiGLU (gate, up) row pairs, RS/2 pairs per stage
    // (gate rows in stage rows 0-7, their up rows in 8-15)
    const bool sw = p.epi == kEpiSwiGLU;
    const int64_t n_items = sw ? p.n_out / 2 : p.n_out;
    const int per_stage = sw ? RS / 2 : RS;
    const int64_t r0 = n_items * blockIdx.x / gridDim.x;
    const int nrows = (int)(n_items * (blockIdx.x + 1) / gridDim.x - r0);
    const int units = (nrows + per_stage - 1) / per_stage;
    const uint32_t ring_s = smem_u32(smem);
    uint64_t pol = 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CWARPS);
        }
        fence_mbar_init();
    }
    rowk::grid_dep_launch();
    __syncthreads();
    auto fill = [&](int u) {                     // stage u into slot u % NS
        const int rows = nrows - u * per_stage < per_stage ? nrows - u * per_stage : per_stage;
        uint8_t *dst = smem + (size_t)(u % NS) * STAGE;
        const uint8_t *src = p.w + (r0 + (int64_t)u * per_stage) * F::ROWB;
        if (!sw) {
            issue_stage<F::ROWB, F::PITCH, STAGE>(dst, &full_bar[u % NS], src, rows, pol);
        } else {
            mbar_arrive_expect_tx(&full_bar[u % NS], (uint32_t)(2 * rows) * F::ROWB);
            const size_t up = (size_t)(p.n_out / 2) * F::ROWB;
            for (int r = 0; r < rows; ++r) {
                bulk_g2s_hint(dst + (size_t)r * F::PITCH, src + (size_t)r * F::ROWB, (uint32_t)F::ROWB,
                              &full_bar[u % NS], pol);
                bulk_g2s_hint(dst + (size_t)(r + RS / 2) * F::PITCH, src + up + (size_t)r * F::ROWB,
                              (uint32_t)F::ROWB, &full_bar[u % NS], pol);
            }
        }
    };
    // PROD: the producer warp's first thread issues every copy; else the first
    // thread of the last compute warp
    constexpr int FILLER = PROD ? THREADS : THREADS - 32;
    if (threadIdx.x == FILLER) {
        pol = make_evict_first_policy();
        // the weights may be the previous kernel's output unless the caller
        // declared them static (pq_set_weight_prefetch)
        if (!p.early_w) rowk::grid_dep_wait();
        if (PROD) {
            for (int u = 0; u < units; ++u) {
                if (u >= NS && !mbar_wait(&empty_bar[u % NS], ((uint32_t)(u / NS) & 1u) ^ 1u)) break;
                fill(u);
            }
        } else {
            for (int u = 0; u < NS && u < units; ++u) fill(u);
        }
    }
    if (PROD && warp == CWARPS) return;
    rowk::grid_dep_wait();                       // x is the previous kernel's output
    uint32_t xb[NT][16][2], xsb[NT] = {};
    float undo[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) build_x<F::XSUMS>(p, t, warp, lane, xb[t], xsb[t], undo[t]);

    bool dead = false;
    const uint32_t blk = (uint32_t)warp * (uint32_t)(F::ROWB / 16);   // this warp's super-block in a row
    for (int u = 0; u < units; ++u) {
        const int slot = u % NS;
        const uint32_t ph = (uint32_t)(u / NS) & 1u;
        if (!dead && !mbar_wait(&full_bar[slot], ph)) dead = true;
        const uint32_t ra = (ring_s + (uint32_t)slot * STAGE + (uint32_t)g * F::PITCH + blk) & ~3u;
        const uint32_t rb = ra + 8u * F::PITCH;
        float v[NT][2];
#pragma unroll
        for (int t = 0; t < NT; ++t) v[t][0] = v[t][1] = 0.f;
        if (!dead) F::template stage<NT>(ra, rb, warp, lane, xb, xsb, undo, v);
        if (PROD) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
        }
        constexpr int SPS = F::template sps<NT>();
        float *rw = red + (size_t)(u & (2 * SPS - 1)) * CWARPS * RS * NB + (size_t)warp * RS * NB;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            rw[g * NB + 4 * t + i4] = v[t][0];
            rw[(g + 8) * NB + 4 * t + i4] = v[t][1];
        }
        if (u % SPS != SPS - 1 && u != units - 1) continue;     // one barrier per SPS stages
        named_sync(1, THREADS);
        const int u0 = u - u % SPS;                             // the first stage since the last barrier
        // !PROD: every warp is done with those stages' slots: refill them
        // (after ordering the reads before the copy engine's writes)
        if (!PROD && threadIdx.x == FILLER) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            for (int uu = u0; uu <= u; ++uu)
                if (uu + NS < units) fill(uu + NS);
        }
        // the first warps add the 16 warps' parts in warp order (one thread
        // per stage, row and column) while the others go on with the next stages
        if ((int)threadIdx.x < (u - u0 + 1) * per_stage * NB) {
            const int su = u0 + (int)threadIdx.x / (per_stage * NB);   // the stage this thread adds
            const int tid = (int)threadIdx.x % (per_stage * NB);
            const int row = tid / NB, col = tid % NB;
            const float *rr = red + (size_t)(su & (2 * SPS - 1)) * CWARPS * RS * NB + row * NB + col;
            float sum = rr[0];
#pragma unroll
            for (int w2 = 1; w2 < CWARPS; ++w2) sum += rr[(size_t)w2 * RS * NB];
            const int n_here = nrows - su * per_stage < per_stage ? nrows - su * per_stage : per_stage;
            const int64_t item = r0 + (int64_t)su * per_stage + row;
            if (sw) {
                // the up row of the pair: stage row row + 8
                const float *ru = rr + (RS / 2) * NB;
                float up = ru[0];
#pragma unroll
                for (int w2 = 1; w2 < CWARPS; ++w2) up += ru[(size_t)w2 * RS * NB];
                sum = rowk::silu(sum) * up;
            } else if (p.epi == kEpiBias) {
                if (row < n_here) sum += p.bias[item];
            }
            if (row < n_here && col < p.nb_cols) p.y[(size_t)col * p.ldy + item] = sum;
        }
    }
}

template <class F, int NT>
cudaError_t launch_t(const uint8_t *w, int64_t n_out, const float *x, int nb_cols, float *y, int64_t ldy, int grid,
                     cudaStream_t s, int early_w, const Epilogue &epi) {
    static PerDeviceOnce configured;
    const cudaError_t ce = configured.run([] {
        return cudaFuncSetAttribute(gemv_rows_mma<F, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem_bytes<F, NT>());
    });
    if (ce != cudaSuccess) return ce;
    Params p{w, x, y, (long long)ldy, (int)n_out, nb_cols, early_w, epi.kind,
             epi.kind == kEpiBias ? epi.bias : nullptr};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block_threads<NT>());
    cfg.dynamicSmemBytes = (size_t)smem_bytes<F, NT>();
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_rows_mma<F, NT>, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// grid: CTAs, at most one per row (per row pair for SwiGLU).
cudaError_t launch(int fmt, const uint8_t *w, int64_t n_out, const float *x, int nb_cols, float *y, int64_t ldy,
                   int grid, cudaStream_t s, int early_w, const Epilogue &epi = Epilogue{}) {
    if (fmt == PQ_Q4_K)
        return nb_cols <= 4 ? launch_t<Q4, 1>(w, n_out, x, nb_cols, y, ldy, grid, s, early_w, epi)
                            : launch_t<Q4, 2>(w, n_out, x, nb_cols, y, ldy, grid, s, early_w, epi);
    return nb_cols <= 4 ? launch_t<Q6, 1>(w, n_out, x, nb_cols, y, ldy, grid, s, early_w, epi)
                        : launch_t<Q6, 2>(w, n_out, x, nb_cols, y, ldy, grid, s, early_w, epi);
}

// Whether this kernel runs (fmt, k, n_out) at `batch` columns with epilogue
// `kind`.  Q4_K: k = 4096, batch 2-8, except plain batch-2 calls on tall
// matrices (rowsnb::kNbTallRows, the two-column kernel); Q6_K: k = 4096,
// batch 3-8, and at least one 16-row stage per CTA on a full GPU (at batch
// 2, and on small matrices, the CUDA-core kernel is faster: output head 83.5
// against 93 us at batch 2).
inline bool takes(int fmt, int64_t k, int64_t n_out, int batch, int kind = kEpiNone) {
    if (k != K || batch < 2 || batch > 8 || n_out < 1) return false;
    if (fmt == PQ_Q4_K) return !(batch == 2 && kind == kEpiNone && n_out >= rowsnb::kNbTallRows);
    return fmt == PQ_Q6_K && batch >= 3 && n_out >= 152 * RS;
}
}  // namespace rmma

}  // namespace

unsigned stream_wait_timeouts(bool reset) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) return 0;
    if (reset) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_wait_timeouts, &z, sizeof(z));
    }
    return v;
}

bool stream_epilogue_fused(int fmt, int64_t n_out, int64_t k, int batch, int kind) {
    if (batch > 1) return rmma::takes(fmt, k, n_out, batch, kind);
    return batch == 1 && n_out >= 1 && k <= (INT64_C(1) << 20) && rowk::takes(fmt, k, n_out, kind == kEpiSwiGLU);
}

bool stream_mma_takes(int fmt, int64_t n_out, int64_t k, int batch) { return rmma::takes(fmt, k, n_out, batch); }

bool stream_supported(int fmt, int64_t n_out, int64_t k, int batch) {
    if (batch == 1 && n_out >= 1 && k <= (INT64_C(1) << 20) && rowk::takes(fmt, k, n_out)) return true;
    if (rmma::takes(fmt, k, n_out, batch)) return true;
    if (fmt == PQ_Q6_K && batch >= 2) return rows6::takes(k, n_out, batch);
    if (fmt != PQ_Q4_K || batch < 1 || batch > 4 || n_out < 1) return false;
    if (k % 256 || k > (INT64_C(1) << 20)) return false;
    return plan_stages(k, batch) >= 2;
}

cudaError_t launch_gemv_stream_epi(int fmt, const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch,
                                   float *y, int64_t ldy, cudaStream_t s, const DeviceInfo &dev, const Epilogue &epi) {
    if (!stream_epilogue_fused(fmt, n_out, k, batch, epi.kind)) return cudaErrorInvalidValue;
    const int64_t items = epi.kind == kEpiSwiGLU ? n_out / 2 : n_out;
    const int grid = (int)(items < dev.sm_count ? items : dev.sm_count);
    if (batch > 1) return rmma::launch(fmt, w, n_out, x, batch, y, ldy, grid, s, weight_prefetch(), epi);
    switch (fmt) {
    case PQ_Q4_K: return rowk::launch_epi<rowk::Q4K>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    case PQ_Q6_K: return rowk::launch_epi<rowk::Q6K>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    case PQ_Q8_0: return rowk::launch_epi<rowk::Q80>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    case PQ_Q5_K: return rowk::launch_epi<rowk::Q5K>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    case PQ_I4_ROW: return rowk::launch_epi<rowk::I4R>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    case PQ_Q2_K: return rowk::launch_epi<rowk::Q2K>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    case PQ_Q3_K: return rowk::launch_epi<rowk::Q3K>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    default: return rowk::launch_epi<rowk::I8R>(w, n_out, k, x, y, grid, s, weight_prefetch(), epi);
    }
}

cudaError_t launch_gemv_stream(int fmt, const uint8_t *w, int64_t n_out, int64_t k,
                               const float *x, int batch, float *y, int64_t ldy,
                               cudaStream_t s, const DeviceInfo &dev) {
    if (!stream_supported(fmt, n_out, k, batch)) return cudaErrorInvalidValue;
    Params p{w, x, y, (long long)ldy, (int)n_out, (int)k, 0};
    const int grid = (int)(n_out < dev.sm_count ? n_out : dev.sm_count);
    if (batch == 1 && rowk::takes(fmt, k, n_out))
        return launch_gemv_stream_epi(fmt, w, n_out, k, x, 1, y, ldy, s, dev, Epilogue{});
    if (rmma::takes(fmt, k, n_out, batch))
        return rmma::launch(fmt, w, n_out, x, batch, y, ldy, grid, s, weight_prefetch());
    if (fmt == PQ_Q4_K && rowsnb::takes(k, n_out, batch))
        return rowsnb::launch<2>(w, n_out, k, x, 2, y, ldy, grid, s);
    if (fmt == PQ_Q6_K)
        return batch == 2 ? rows6::launch<2>(w, n_out, k, x, 2, y, ldy, grid, s)
                          : rows6::launch<4>(w, n_out, k, x, batch, y, ldy, grid, s);
    switch (batch) {
    case 1: return launch_nb<1>(p, grid, s);
    case 2: return launch_nb<2>(p, grid, s);
    case 3: return launch_nb<3>(p, grid, s);
    default: return launch_nb<4>(p, grid, s);
    }
}

}  // namespace pqk

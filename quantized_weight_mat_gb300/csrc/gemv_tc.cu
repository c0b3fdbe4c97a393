// Tensor-core fused dequant + mat-vec for Q4_K at batch 5..16 (tcgen05).
//
// The operation is the same mat-vec with the decoding of W fused into it
// (ember pull request, quant.rs description) on GGUF-style Q4_K super-blocks (PESTI README, "What
// This Is"), for several x columns at once.  At batch 8-16 each weight feeds
// 8-16 multiply-adds, too many for CUDA cores at HBM speed, so the products go
// to the 5th-generation tensor cores while the weights still stream once.
//
// Exactness: a tile entry is the integer sc_j*q (q in 0..15, sc_j in 0..63,
// so <= 945), exactly representable in fp16; x enters as two fp16 columns
// (x_hi = fp16(x'), x_lo = fp16(x' - x_hi)) of x' = 2^e * x, where the power
// of two e is chosen per super-block and column so that max|x'| lies in
// [2^9, 2^10): every x' and every sum of 32 of them fits fp16's range, for
// any finite x.  Every product is exact in the f32 accumulator and only
// accumulation rounds.  The sub-block mins enter through a second, K=16
// product of the 6-bit mins with the fp16 hi/lo sums of x' over each
// 32-element sub-block.  Per super-block, row and column the epilogue forms
// y += 2^-e * (d*(A.x') - dmin*(m.XS')) in f32 (multiplying by 2^-e is
// exact).
//
// Work split: the (128-row tile, super-block) items of the matrix, in
// tile-major order, are cut into one contiguous, equal-sized range per CTA
// (one CTA per SM).  A tile whose items are spread over several CTAs is
// split-K: each writes its partial sums to scratch, and a small kernel that
// runs after the main one (resident beside it, waiting on it) adds the parts
// in CTA order and writes y, so the result does not depend on timing.
//
// Pipeline inside a CTA:
//   warp 20 producer: a 2-D TMA load (tensor map over W as [n_out][row bytes])
//           brings one 128-row x 144-byte super-block column per stage, and a
//           1-D bulk copy brings that super-block's x tile;
//   warps 0-15 decoders: thread (c, r) turns the 64 weights of chunk c of
//           row r into fp16 sc*q (one mask per four codes, their e4m3
//           conversion to q * 2^-9, one HMUL2 by sc * 2^9 per two weights) and
//           writes them straight into tensor memory (tcgen05.st; TMEM lane =
//           row, two K values per column), a ring of eight slots (two
//           super-blocks); the chunk-0 threads also write the row's mins;
//   warps 21-24 MMA issuers (one thread each): for super-blocks g with
//           g % 2 == buf, thread (buf, half) issues the eight tcgen05.mma
//           (M=128, N=2*NBP, K=16, A from tensor memory, x from shared memory)
//           of chunks 2*half, 2*half+1 into its own TMEM accumulator (half 0
//           also the mins product), then commits;
//   warps 16-19 epilogue: tcgen05.ld of the three accumulators (warp w reads
//           TMEM lanes 32(w%4).. = its rows), d and dmin from the raw block,
//           f32 scaling; frees the stage and the accumulators.
// Accumulators are double-buffered in TMEM; every mbarrier wait is bounded.
//
// x is converted once per call by a small kernel into a per-super-block image
// (the operand layout the MMA reads, plus the sub-block sums), in scratch
// memory that also holds the split-K partial sums.

#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "pq_device.cuh"
#include "pq_internal.h"
#include "pq_ptx.cuh"

namespace pqk {
namespace {

constexpr int TM = 128;                       // rows per tile = MMA M
constexpr int RAW_BYTES = TM * 144;           // one super-block column of a tile
#ifndef PQ_TC_ABUFS
#define PQ_TC_ABUFS 2
#endif
constexpr int A_BUFS = PQ_TC_ABUFS;           // super-blocks in flight between decoders, MMA and epilogue
constexpr int TMEM_COLS = 512;
constexpr int DEC_WARPS = 16, EPI_WARPS = 4;
constexpr int PRODUCER_WARP = DEC_WARPS + EPI_WARPS;
constexpr int MMA_WARP = PRODUCER_WARP + 1;   // MMA_WARP + 2*buf + half: see the issuer role

// Per column count: the 32-column kernel keeps one super-block in flight (its
// three 64-column accumulators and A slots fill the 512 TMEM columns), the
// others two.
template <int NBP> __host__ __device__ constexpr int tc_abufs() { return NBP == 32 ? 1 : A_BUFS; }
template <int NBP> __host__ __device__ constexpr int tc_threads() { return (MMA_WARP + 2 * tc_abufs<NBP>()) * 32; }
// TMEM column of A slot 0 (32 columns per 64-weight slot, four slots per
// buffer) and of the mins operand of buffer b (8 columns at tc_amin_col + 8b)
template <int NBP> __host__ __device__ constexpr int tc_a_col() { return TMEM_COLS - 32 * 4 * tc_abufs<NBP>(); }
template <int NBP> __host__ __device__ constexpr int tc_amin_col() { return tc_a_col<NBP>() - 8 * tc_abufs<NBP>(); }
constexpr int kMaxGrid = 160;                 // CTAs at most (partial-sum slots are sized for it)

// x image of one super-block for NBP columns (N' = 2*NBP MMA columns, the hi
// parts then the lo parts): N' x 256 fp16, K-major 8x8 core matrices, 8-row
// groups 4096 bytes apart; then the mins operand N' x 16 fp16 (K = j < 8: the
// hi or lo part of the sum of x' over sub-block j; K = 8..15: zero), 8-row
// groups 256 bytes apart; then 128 bytes holding, per column, the f32 factor
// 2^-e that undoes the column's scale.
template <int NBP> __host__ __device__ constexpr int xmain_bytes() { return 2 * NBP * 256 * 2; }
template <int NBP> __host__ __device__ constexpr int xmins_bytes() { return 2 * NBP * 16 * 2; }
template <int NBP> __host__ __device__ constexpr int xscale_off() { return xmain_bytes<NBP>() + xmins_bytes<NBP>(); }
template <int NBP> __host__ __device__ constexpr int btile_bytes() { return xscale_off<NBP>() + 128; }
static_assert(16 * 4 <= 128, "one f32 factor per column fits the scale area");
template <int NBP> __host__ __device__ constexpr int raw_stages() { return NBP == 32 ? 4 : NBP == 16 ? 6 : 8; }
template <int NBP> __host__ __device__ constexpr int stage_bytes() { return RAW_BYTES + btile_bytes<NBP>(); }
template <int NBP> __host__ __device__ constexpr int smem_bytes() { return raw_stages<NBP>() * stage_bytes<NBP>() + 1024; }
static_assert(stage_bytes<8>() % 128 == 0 && stage_bytes<16>() % 128 == 0 && stage_bytes<32>() % 128 == 0,
              "stage alignment");
static_assert(smem_bytes<32>() <= 227 * 1024 && smem_bytes<16>() <= 227 * 1024, "shared memory per CTA");

// Scratch of one call: x image, then partial sums [grid][2][TM][NBP] (slot
// 2c: CTA c's first tile, 2c+1: its last tile, when split).
template <int NBP> size_t scratch_img_bytes(int64_t k) { return (size_t)(k / 256) * btile_bytes<NBP>(); }
template <int NBP> size_t scratch_part_bytes(int grid) { return (size_t)grid * 2 * NBP * TM * 4; }
template <int NBP> size_t scratch_bytes(int64_t k, int grid) {
    return scratch_img_bytes<NBP>(k) + scratch_part_bytes<NBP>(grid);
}

// K order inside a super-block: chunk e of A-column a (8 fp16 per 16 bytes)
// holds weight position pos(a, e).  It follows how two qs words turn into
// four half2 pairs: bytes (0,1), then (2,3), of each word -- their low
// nibbles in the chunk's first half, their high nibbles in the second.
__host__ __device__ constexpr int kpos(int a, int e) {
    return 64 * (a / 8) + 32 * ((a % 8) / 4) + 8 * (a % 4) + e;
}

// byte offset of element (n, K) in a K-major no-swizzle operand whose 8-row
// groups are `sbo` bytes apart (core matrices of 8 rows x 16 bytes, K-adjacent
// core matrices 128 bytes apart)
__host__ __device__ constexpr int kmaj_off(int n, int K, int sbo) {
    return (n / 8) * sbo + (K / 8) * 128 + (n % 8) * 16 + (K % 8) * 2;
}

// ---------------------------------------------------------------- x image
// One block per super-block.  Launched with programmatic dependent launch: it
// may become resident while the previous kernel on the stream finishes, and
// waits for that kernel before anything else.  Only then does it let the main
// kernel launch, so that the weights the main kernel starts streaming at once
// are complete even when the previous kernel wrote them; the main kernel waits
// for this one only before its first x tile.
//
// Scale of column b: x' = 2^e * x with e = tc_scale_exponent(max|x| over the
// super-block's 256 values of the column); see that function.

template <int NBP>
__global__ void __launch_bounds__(256) prep_x_tc(const float *__restrict__ x, int k, int nb_cols,
                                                 uint8_t *__restrict__ img) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int sb = blockIdx.x;
    constexpr int NP = 2 * NBP;
    uint8_t *tile = img + (size_t)sb * btile_bytes<NBP>();
    __half *out = reinterpret_cast<__half *>(tile);
    __half *om = reinterpret_cast<__half *>(tile + xmain_bytes<NBP>());
    float *undo = reinterpret_cast<float *>(tile + xscale_off<NBP>());
    __shared__ uint32_t wmax[8][NBP];
    __shared__ float mult[NBP];
    __shared__ float xs[NBP][8];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    // main part: thread t = K index; all column loads in flight together
    const int K = t;
    const int pos = kpos(K / 8, K % 8);
    float v[NBP];
#pragma unroll
    for (int b = 0; b < NBP; ++b) v[b] = b < nb_cols ? __ldg(x + (size_t)b * k + sb * 256 + pos) : 0.f;
    // sub-block sums: thread (column, sub-block) for t < NBP * 8, 8 vector loads
    const int sbc = t / 8, sbj = t % 8;
    float4 sv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < NBP * 8 && sbc < nb_cols) {
        const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)sbc * k + sb * 256 + 32 * sbj);
#pragma unroll
        for (int i = 0; i < 8; ++i) sv[i] = __ldg(xb + i);
    }
    // max |x| per column: the bit patterns of non-negative floats order like
    // their values (NaN above inf), so an integer reduction gives it
#pragma unroll
    for (int b = 0; b < NBP; ++b) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(v[b]) & 0x7fffffffu);
        if (lane == 0) wmax[warp][b] = m;
    }
    __syncthreads();
    if (t < NBP) {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) m = max(m, wmax[w][t]);
        const int e = tc_scale_exponent(m);
        mult[t] = __uint_as_float((uint32_t)(127 + e) << 23);    // 2^e
        undo[t] = __uint_as_float((uint32_t)(127 - e) << 23);    // 2^-e
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < NBP; ++b) {
        const float s = v[b] * mult[b];
        const __half hi = __float2half_rn(s);
        const __half lo = __float2half_rn(s - __half2float(hi));
        out[kmaj_off(b, K, 4096) / 2] = hi;
        out[kmaj_off(NBP + b, K, 4096) / 2] = lo;
    }
    if (t < NBP * 8) {
        // fixed order; |x'| < 2^10, so |sum| < 2^15 stays in fp16's range
        const float m = mult[sbc];
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s = s + sv[i].x * m + sv[i].y * m + sv[i].z * m + sv[i].w * m;
        xs[sbc][sbj] = s;
    }
    __syncthreads();
    // mins operand: K = j < 8 holds the sums (hi part for n < NBP, lo part after), K = 8..15 zero
    for (int i = t; i < NP * 16; i += 256) {
        const int n = i / 16, Kk = i % 16;
        float val = 0.f;
        if (Kk < 8) {
            const float s = xs[n % NBP][Kk];
            const __half hi = __float2half_rn(s);
            val = n < NBP ? __half2float(hi) : __half2float(__float2half_rn(s - __half2float(hi)));
        }
        om[kmaj_off(n, Kk, 256) / 2] = __float2half_rn(val);
    }
}

// ---------------------------------------------------------------- tcgen05 helpers
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version for tcgen05; no swizzle, base offset 0
    return d;
}

// kind::f16 instruction descriptor: f32 accumulator, fp16 A and B, both K-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Same with the A operand in tensor memory (column address a_tmem).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Each thread writes 32 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// Each thread writes 8 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// x image for the register-operand kernel (gemv_mma_q4_k): the same scaled
// hi/lo halves as prep_x_tc, stored in the order the warps load them as
// mma.sync A fragments.  Per 16-position step s of the super-block and group
// mt of 8 columns, lane L = 4g + i holds 16 bytes {a0, a1, a2, a3}: column
// 8mt + g, positions 16s + 4i + {0, 1} (a0 hi, a1 lo) and + {2, 3} (a2 hi, a3
// lo) -- the K slots 2i, 2i+1 and 2i+8, 2i+9 of the fragment, matching the
// weights a thread decodes from one 4-byte qs word.  Then per group, lane L:
// 8 bytes {hi, lo} of the sums over sub-blocks 2i and 2i+1 of column 8mt + g
// (the mins operand; K slots 8..15 are zero); then the factors 2^-e.  The
// tile has the size of prep_x_tc's.
template <int NBP>
__global__ void __launch_bounds__(256) prep_x_mma(const float *__restrict__ x, int k, int nb_cols,
                                                  uint8_t *__restrict__ img) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int MT = NBP / 8;
    const int sb = blockIdx.x;
    uint8_t *tile = img + (size_t)sb * btile_bytes<NBP>();
    float *undo = reinterpret_cast<float *>(tile + xscale_off<NBP>());
    __shared__ uint32_t wmax[8][NBP];
    __shared__ float mult[NBP];
    __shared__ float xs[NBP][8];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    float v[NBP];
#pragma unroll
    for (int b = 0; b < NBP; ++b) v[b] = b < nb_cols ? __ldg(x + (size_t)b * k + sb * 256 + t) : 0.f;
    const int sbc = t / 8, sbj = t % 8;
    float4 sv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < NBP * 8 && sbc < nb_cols) {
        const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)sbc * k + sb * 256 + 32 * sbj);
#pragma unroll
        for (int i = 0; i < 8; ++i) sv[i] = __ldg(xb + i);
    }
#pragma unroll
    for (int b = 0; b < NBP; ++b) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(v[b]) & 0x7fffffffu);
        if (lane == 0) wmax[warp][b] = m;
    }
    __syncthreads();
    if (t < NBP) {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) m = max(m, wmax[w][t]);
        const int e = tc_scale_exponent(m);
        mult[t] = __uint_as_float((uint32_t)(127 + e) << 23);    // 2^e
        undo[t] = __uint_as_float((uint32_t)(127 - e) << 23);    // 2^-e
    }
    __syncthreads();
    // position t: step t/16, lane slot i = (t%16)/4, r = t%4 -> registers
    // 0 (hi) and 1 (lo) for r < 2, 2 and 3 for r >= 2, low half for r even
    const int st = t >> 4, i4 = (t >> 2) & 3, r = t & 3;
    const int hreg = (r >> 1) ? 2 : 0, half = r & 1;
#pragma unroll
    for (int b = 0; b < NBP; ++b) {
        const float sx = v[b] * mult[b];
        const __half hi = __float2half_rn(sx);
        const __half lo = __float2half_rn(sx - __half2float(hi));
        const int L = 4 * (b % 8) + i4;
        __half *frag = reinterpret_cast<__half *>(tile + ((size_t)(st * MT + b / 8) * 32 + L) * 16);
        frag[2 * hreg + half] = hi;
        frag[2 * (hreg + 1) + half] = lo;
    }
    if (t < NBP * 8) {
        const float m = mult[sbc];
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s = s + sv[i].x * m + sv[i].y * m + sv[i].z * m + sv[i].w * m;
        xs[sbc][sbj] = s;
    }
    __syncthreads();
    // mins operand: thread (column b, sub-block j) writes its hi and lo halves
    if (t < NBP * 8) {
        const int b = sbc, j = sbj;
        const float s = xs[b][j];
        const __half hi = __float2half_rn(s);
        const __half lo = __float2half_rn(s - __half2float(hi));
        const int L = 4 * (b % 8) + (j >> 1);
        __half *frag = reinterpret_cast<__half *>(tile + xmain_bytes<NBP>() + ((size_t)(b / 8) * 32 + L) * 8);
        frag[j & 1] = hi;
        frag[2 + (j & 1)] = lo;
    }
}


__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// Wait for the preceding tcgen05.ld; the registers are passed through so that
// no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
          "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<const uint32_t *>(&v); }
__device__ __forceinline__ __half2 h2_of(uint32_t bits) { return *reinterpret_cast<const __half2 *>(&bits); }
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) { return h2_bits(__hmul2(h2_of(a), h2_of(b))); }

// Each thread reads 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
        :
        : "memory");
}

struct TcParams {
    const uint8_t *x_img;      // x image, one tile per super-block
    float *y;
    float *partials;           // [grid][2][NBP][TM] split-K partial sums
    long long ldy;
    long long total;           // work items: tiles x super-blocks per row
    int n_out;
    int k;
    int nb_cols;
    const float *bias;         // bias epilogue: bias[n_out], else null
    // SwiGLU epilogue (n_ff > 0): tile 2i is rows [128i, 128i+128) of the gate
    // half, tile 2i+1 the same rows of the up half (rows n_ff + ...); every
    // tile's sums go to ytmp [tiles][TM][NBP] or to the partial sums, and a
    // finishing kernel forms h = silu(gate) * up
    int n_ff;
    float *ytmp;
};

// First matrix row of tile t (see TcParams).
__host__ __device__ __forceinline__ long long tile_row0(int t, int n_ff) {
    return n_ff > 0 ? (long long)(t & 1) * n_ff + (long long)(t >> 1) * TM : (long long)t * TM;
}

// First work item of CTA c when `total` items are split over `grid` CTAs, and
// the CTA that owns item i (the largest c with item_begin(c) <= i).
__device__ __forceinline__ long long item_begin(long long c, long long total, int grid) { return c * total / grid; }
__device__ __forceinline__ int item_owner(long long i, long long total, int grid) {
    return (int)(((i + 1) * grid - 1) / total);
}

template <int NBP>
__global__ void __launch_bounds__(tc_threads<NBP>(), 1)
    gemv_tc_q4_k(const __grid_constant__ CUtensorMap wmap, TcParams p) {
    constexpr int NP = 2 * NBP;
    constexpr int NSR = raw_stages<NBP>();
    constexpr int STAGE = stage_bytes<NBP>();
    constexpr uint32_t IDESC = instr_desc(TM, NP);
    constexpr int A_BUFS = tc_abufs<NBP>();
    constexpr int A_COL = tc_a_col<NBP>(), AMIN_COL = tc_amin_col<NBP>();
    static_assert(3 * A_BUFS * NP <= AMIN_COL, "accumulators below the A operands");
    static_assert(A_COL + 32 * 4 * A_BUFS <= TMEM_COLS, "A slots fit in the allocation");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t raw_full[NSR], raw_empty[NSR];
    __shared__ __align__(8) uint64_t a_full[A_BUFS][2];
    __shared__ __align__(8) uint64_t item_done[A_BUFS], acc_empty[A_BUFS];
    __shared__ uint32_t tmem_base_sh;

    // 1024-aligned working area
    uint8_t *ring = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int grid = (int)gridDim.x;
    const long long i0 = item_begin(blockIdx.x, p.total, grid);
    const int count = (int)(item_begin(blockIdx.x + 1, p.total, grid) - i0);   // items of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSR; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], EPI_WARPS);
        }
        for (int s = 0; s < A_BUFS; ++s) {
            mbar_init(&a_full[s][0], DEC_WARPS / 2);
            mbar_init(&a_full[s][1], DEC_WARPS / 2);
            mbar_init(&item_done[s], 2);
            mbar_init(&acc_empty[s], EPI_WARPS);
        }
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_sh)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // the split-K finishing kernel may be scheduled now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == PRODUCER_WARP) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = make_evict_first_policy();
            int tile = (int)(i0 / nb), sb = (int)(i0 % nb);
            for (int g = 0; g < count; ++g) {
                const int slot = g % NSR;
                const uint32_t ph = (uint32_t)(g / NSR) & 1u;
                if (!mbar_wait(&raw_empty[slot], ph ^ 1u)) break;
                uint8_t *st = ring + slot * STAGE;
                mbar_arrive_expect_tx(&raw_full[slot], (uint32_t)STAGE);
                tma_load_2d(st, &wmap, sb * 144, (int)tile_row0(tile, p.n_ff), &raw_full[slot]);
                // the weights were complete before the x-prep kernel let this kernel
                // launch; the x image is that kernel's output: wait for it once,
                // before its first use
                if (g == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                bulk_g2s_hint(st + RAW_BYTES, p.x_img + (size_t)sb * btile_bytes<NBP>(), (uint32_t)btile_bytes<NBP>(),
                              &raw_full[slot], pol);
                if (++sb == nb) { sb = 0; ++tile; }
            }
        }
    } else if (warp >= MMA_WARP) {
        // ---------------- MMA issuers ----------------
        // Thread (buf, half) issues, for the super-blocks g with g % A_BUFS ==
        // buf, the eight products of chunks 2*half and 2*half+1 into its own
        // accumulator.  Several issuing threads keep the tensor core busy: one
        // thread's tcgen05 instructions and waits go out one after another.
        const int buf = (warp - MMA_WARP) >> 1, half = (warp - MMA_WARP) & 1;
        if (lane == 0) {
            bool dead = false;
            for (int g = buf; g < count; g += A_BUFS) {
                const int slot = g % NSR;
                const uint32_t par = (uint32_t)(g / A_BUFS) & 1u;
                // accumulator free (epilogue done with super-block g - A_BUFS), then
                // the two A chunks decoded; the decoders saw the stage (weights and
                // x tile) complete before they arrived
                if (!dead && !mbar_wait(&acc_empty[buf], par ^ 1u)) dead = true;
                if (!dead && !mbar_wait(&a_full[buf][half], par)) dead = true;
                tc_fence_after();
                if (!dead) {
                    // eight products back to back, no branch between them
                    const uint32_t d_acc = tmem + (uint32_t)((3 * buf + half) * NP);
                    const uint32_t a0 = tmem + (uint32_t)(A_COL + 32 * (4 * buf + 2 * half));
                    const uint32_t bst = smem_u32(ring + slot * STAGE + RAW_BYTES);
                    const uint64_t b0 = smem_desc(bst + 2048 * half, 128u, 4096u);
#pragma unroll
                    for (int cl = 0; cl < 2; ++cl)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_f16_ta(d_acc, a0 + (uint32_t)(32 * cl + 8 * ks), b0 + (uint64_t)(16 * (4 * cl + ks)),
                                       IDESC, (cl | ks) ? 1u : 0u);
                    if (half == 0)
                        mma_f16_ta(tmem + (uint32_t)((3 * buf + 2) * NP), tmem + (uint32_t)(AMIN_COL + 8 * buf),
                                   smem_desc(bst + xmain_bytes<NBP>(), 128u, 256u), IDESC, 0u);
                }
                mma_commit(&item_done[buf]);
            }
        }
    } else if (warp >= DEC_WARPS) {
        // ---------------- epilogue (warps 16-19) ----------------
        const int r = 32 * (warp & 3) + lane;                              // row within the tile = TMEM lane
        const uint32_t row_taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const int first_tile = (int)(i0 / nb);
        float yacc[NBP];
#pragma unroll
        for (int b = 0; b < NBP; ++b) yacc[b] = 0.f;
        bool dead = false;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // before any store of y or partials
        int tile = first_tile, sb = (int)(i0 % nb);
        for (int g = 0; g < count; ++g) {
            const int slot = g % NSR;
            const int buf = g % A_BUFS;
            const uint32_t par = (uint32_t)(g / A_BUFS) & 1u;
            // d and dmin of row r (the stage is held until this warp frees it)
            const uint8_t *st = ring + slot * STAGE;
            if (!dead && !mbar_wait(&item_done[buf], par)) dead = true;
            tc_fence_after();
            const uint32_t dd = *reinterpret_cast<const uint32_t *>(st + r * 144);
            // lane b < NBP keeps column b's factor 2^-e (read before the stage is freed)
            const float undo = *reinterpret_cast<const float *>(st + RAW_BYTES + xscale_off<NBP>() + 4 * (lane % NBP));
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[slot]);
            const float d = h2f(dd), dmin = h2f(dd >> 16);
            // the super-block's three accumulators (two halves of the products,
            // the mins product), each with hi and lo x columns, in scaled units
            if constexpr (NBP == 8) {
                float v[NBP];
#pragma unroll
                for (int part = 0; part < 3; ++part) {
                    const uint32_t taddr = row_taddr + (uint32_t)((3 * buf + part) * NP);
                    const float sc = part < 2 ? d : -dmin;
                    uint32_t t[16];
                    tmem_ld16(taddr, t);
                    tmem_ld_wait(t);
#pragma unroll
                    for (int b = 0; b < NBP; ++b) {
                        const float pr = __uint_as_float(t[b]) + __uint_as_float(t[NBP + b]);
                        v[b] = part == 0 ? sc * pr : fmaf(sc, pr, v[b]);
                    }
                }
#pragma unroll
                for (int b = 0; b < NBP; ++b) yacc[b] = fmaf(v[b], __shfl_sync(0xffffffffu, undo, b), yacc[b]);
            } else {
                // 16 columns at a time: their hi columns, then their lo
                // columns, 16 registers each (the 800- and 736-thread blocks
                // leave 72 and 80 registers per thread)
#pragma unroll
                for (int grp = 0; grp < NBP / 16; ++grp) {
                    float v[16];
#pragma unroll
                    for (int part = 0; part < 3; ++part) {
                        const uint32_t taddr = row_taddr + (uint32_t)((3 * buf + part) * NP + 16 * grp);
                        const float sc = part < 2 ? d : -dmin;
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl) {
                            uint32_t t[16];
                            tmem_ld16(taddr + (uint32_t)(NBP * hl), t);
                            tmem_ld_wait(t);
#pragma unroll
                            for (int b = 0; b < 16; ++b)
                                v[b] = (part == 0 && hl == 0) ? sc * __uint_as_float(t[b])
                                                              : fmaf(sc, __uint_as_float(t[b]), v[b]);
                        }
                    }
#pragma unroll
                    for (int b = 0; b < 16; ++b)
                        yacc[16 * grp + b] = fmaf(v[b], __shfl_sync(0xffffffffu, undo, 16 * grp + b), yacc[16 * grp + b]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);

            if (sb == nb - 1 || g == count - 1) {
                // the CTA's part of this tile is complete
                const long long t0i = (long long)tile * nb;
                const int cf = item_owner(t0i, p.total, grid), cl = item_owner(t0i + nb - 1, p.total, grid);
                const int row = tile * TM + r;
                if (cf == cl && p.n_ff > 0) {
                    // SwiGLU: the finishing kernel pairs this tile with its partner
                    float4 *mine = reinterpret_cast<float4 *>(p.ytmp + ((size_t)tile * TM + r) * NBP);
#pragma unroll
                    for (int b4 = 0; b4 < NBP / 4; ++b4)
                        mine[b4] = make_float4(yacc[4 * b4], yacc[4 * b4 + 1], yacc[4 * b4 + 2], yacc[4 * b4 + 3]);
                } else if (cf == cl) {
                    if (row < p.n_out) {
                        const float bias = p.bias ? p.bias[row] : 0.f;
#pragma unroll
                        for (int b = 0; b < NBP; ++b)
                            if (b < p.nb_cols) p.y[(size_t)b * p.ldy + row] = p.bias ? yacc[b] + bias : yacc[b];
                    }
                } else {
                    // split tile: this CTA's part, added up by the finishing kernel
                    const int side = tile == first_tile ? 0 : 1;
                    float4 *mine = reinterpret_cast<float4 *>(p.partials + ((size_t)(blockIdx.x * 2 + side) * TM + r) * NBP);
#pragma unroll
                    for (int b4 = 0; b4 < NBP / 4; ++b4)
                        mine[b4] = make_float4(yacc[4 * b4], yacc[4 * b4 + 1], yacc[4 * b4 + 2], yacc[4 * b4 + 3]);
                }
#pragma unroll
                for (int b = 0; b < NBP; ++b) yacc[b] = 0.f;
            }
            if (++sb == nb) { sb = 0; ++tile; }
        }
    } else {
        // ---------------- decoders (warps 0-15) ----------------
        // thread (c, r): chunk c (weights 64c..64c+63: sub-blocks 2c, 2c+1) of row r
        const int c = warp >> 2;
        const int r = 32 * (warp & 3) + lane;
        const int h = c >> 1, cc = c & 1;
        const uint32_t mA = h ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
        const uint32_t mB = h ? 0x30303030u : 0u;
        const uint32_t a_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's TMEM lanes
        bool dead = false;
        for (int g = 0; g < count; ++g) {
            const int slot = g % NSR;
            const uint32_t ph = (uint32_t)(g / NSR) & 1u;
            const int buf = g % A_BUFS;
            const uint32_t par = (uint32_t)(g / A_BUFS) & 1u;
            if (!dead && !mbar_wait(&raw_full[slot], ph)) dead = true;
            const uint8_t *blk = ring + slot * STAGE + r * 144;
            const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
            const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
            const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
            // 6-bit scales of sub-blocks 2c (low nibbles) and 2c+1 (high nibbles)
            const uint32_t sc4 = ((h ? hd.w : hd.y) & mA) | ((hd.y >> 2) & mB);
            // (sc * 2^9) pairs: the codes come as q * 2^-9 from the e4m3
            // conversion, and sc*q <= 945 is exact in fp16
            const __half slo = __int2half_rn((int)((sc4 >> (16 * cc)) & 0xFF) * 512);
            const __half shi = __int2half_rn((int)((sc4 >> (16 * cc + 8)) & 0xFF) * 512);
            const uint32_t Slo = h2_bits(__halves2half2(slo, slo));
            const uint32_t Shi = h2_bits(__halves2half2(shi, shi));
            const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            // the chunk's 64 K values of row r: TMEM column j holds K = 2j, 2j+1
            uint32_t R[32];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const uint32_t w0 = w[2 * a], w1 = w[2 * a + 1];
                nibble_bytes_h2(w0 & 0x0F0F0F0Fu, R[4 * a + 0], R[4 * a + 1]);
                nibble_bytes_h2(w1 & 0x0F0F0F0Fu, R[4 * a + 2], R[4 * a + 3]);
                nibble_bytes_h2((w0 >> 4) & 0x0F0F0F0Fu, R[16 + 4 * a + 0], R[16 + 4 * a + 1]);
                nibble_bytes_h2((w1 >> 4) & 0x0F0F0F0Fu, R[16 + 4 * a + 2], R[16 + 4 * a + 3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    R[4 * a + j] = hmul2_u(R[4 * a + j], Slo);
                    R[16 + 4 * a + j] = hmul2_u(R[16 + 4 * a + j], Shi);
                }
            }
            // this buffer's slots are free once the products of the super-block
            // that used them before are complete
            if (!dead && !mbar_wait(&item_done[buf], par ^ 1u)) dead = true;
            tc_fence_after();
            tmem_st32(a_lane + (uint32_t)(A_COL + 32 * (4 * buf + c)), R);
            if (c == 0) {
                // the row's mins product operand: m_0..m_7 at K = 0..7, zero at K = 8..15
                const uint32_t mlo = hd.z & 0x3F3F3F3Fu;
                const uint32_t mhi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
                uint32_t M[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t src = i < 2 ? mlo : mhi;
                    const int sh = 16 * (i & 1);
                    M[i] = h2_bits(__halves2half2(__int2half_rn((int)((src >> sh) & 0xFFu)),
                                                  __int2half_rn((int)((src >> (sh + 8)) & 0xFFu))));
                    M[4 + i] = 0u;
                }
                tmem_st8(a_lane + (uint32_t)(AMIN_COL + 8 * buf), M);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[buf][h]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------- register-operand kernel
// The same work split, stages and split-K as gemv_tc_q4_k, with the products
// on mma.sync (m16n8k16, fp16 in, f32 accumulate) fed from registers: the
// decoded weights never leave the registers of the warp that decodes them
// (the tensor-memory kernel above writes 64 KB of fp16 per super-block item
// into tensor memory, and that store bounds it).  A = x (16 rows = hi and lo
// parts of 8 columns), B = the exact fp16 sc*q of 8 weight rows.
//
//   warp 16 producer (as above);
//   warps 0-15: group q = warp/4 takes items q, q+4, ...; warp w%4 of a group
//           rows 32(w%4)..+31 of the item's 128-row tile, in four n8 blocks.
//           Per item: the 256 K of the super-block in 16 steps; each qs word
//           gives a thread's four weights of two steps (low and high
//           nibbles), decoded with one mask per four codes, the e4m3
//           conversion (q * 2^-9) and one HMUL2 by sc * 2^9 per two weights;
//           one K=16 product of the mins per n8 block; then, per row and column,
//           y += 2^-e * (d*(x'.A) - dmin*(XS'.m)) in registers.
//           At the end of a tile the four groups' sums are added in group
//           order through shared memory and stored (or written as split-K
//           parts / SwiGLU halves, as above).
constexpr int MMA_GROUPS = 4;
constexpr int MMA_COMPUTE_WARPS = 16;
constexpr int MMA_THREADS = (MMA_COMPUTE_WARPS + 1) * 32;
template <int NBP> __host__ __device__ constexpr int mma_stages() { return NBP == 8 ? 7 : 5; }
template <int NBP> __host__ __device__ constexpr int mma_red_bytes() { return MMA_GROUPS * TM * NBP * 4; }
template <int NBP> __host__ __device__ constexpr int mma_smem_bytes() {
    return mma_stages<NBP>() * stage_bytes<NBP>() + mma_red_bytes<NBP>() + 1024;
}
static_assert(mma_smem_bytes<8>() <= 227 * 1024 && mma_smem_bytes<16>() <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// fp16 pairs as bit patterns, so that the arithmetic below takes them as
// immediate: 1024
constexpr uint32_t kH2_1024 = 0x64006400u;

// byte i (0..3) of v as an exact fp16 value, duplicated in both halves
__device__ __forceinline__ uint32_t byte_h2(uint32_t v, int i) {
    // (0x64 << 8 | byte) is the fp16 1024 + byte; subtracting 1024 is exact
    const uint32_t sel = (uint32_t)i | 0x40u | ((uint32_t)i << 8) | 0x4000u;
    const uint32_t p = __byte_perm(v, 0x64646464u, sel);
    return h2_bits(__hsub2(h2_of(p), h2_of(kH2_1024)));
}
// bytes i and i+1 of v as exact fp16 values (low half: byte i); i may vary
__device__ __forceinline__ uint32_t bytes_h2(uint32_t v, uint32_t i) {
    const uint32_t sel = i | 0x40u | ((i + 1u) << 8) | 0x4000u;
    const uint32_t p = __byte_perm(v, 0x64646464u, sel);
    return h2_bits(__hsub2(h2_of(p), h2_of(kH2_1024)));
}
constexpr uint32_t kH2_512 = 0x60006000u;

// Wait until the producer has issued item g (the counter it advances after
// each issue), bounded like the mbarrier waits.  A group that takes every
// fourth item may reach item g's slot while the slot still holds, or has not
// yet been given, the item before it (the ring is not a multiple of four
// stages); waiting on the full barrier's parity then would see that older
// phase complete.  Once item g is issued, the slot's previous phase has
// completed and the parity wait is exact.
__device__ __forceinline__ bool wait_issued(const volatile int *issued, int g) {
    if (*issued <= g) {
        const unsigned long long t0 = globaltimer_ns();
        while (*issued <= g) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicAdd(&g_wait_timeouts, 1u);
                return false;
            }
        }
    }
    __threadfence_block();   // pairs with the producer's fence before its store
    return true;
}

template <int NBP>
__global__ void __launch_bounds__(MMA_THREADS, 1)
    gemv_mma_q4_k(const __grid_constant__ CUtensorMap wmap, TcParams p) {
    constexpr int MT = NBP / 8;
    constexpr int NSR = mma_stages<NBP>();
    constexpr int STAGE = stage_bytes<NBP>();

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t raw_full[NSR], raw_empty[NSR];
    __shared__ int issued_sh;                                       // items the producer has issued
    volatile int *issued = &issued_sh;
    uint8_t *ring = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    float *red = reinterpret_cast<float *>(ring + NSR * STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int grid = (int)gridDim.x;
    const long long i0 = item_begin(blockIdx.x, p.total, grid);
    const int count = (int)(item_begin(blockIdx.x + 1, p.total, grid) - i0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSR; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 4);
        }
        *issued = 0;
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == MMA_COMPUTE_WARPS) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = make_evict_first_policy();
            int tile = (int)(i0 / nb), sb = (int)(i0 % nb);
            for (int g = 0; g < count; ++g) {
                const int slot = g % NSR;
                const uint32_t ph = (uint32_t)(g / NSR) & 1u;
                if (!mbar_wait(&raw_empty[slot], ph ^ 1u)) break;
                uint8_t *st = ring + slot * STAGE;
                mbar_arrive_expect_tx(&raw_full[slot], (uint32_t)STAGE);
                tma_load_2d(st, &wmap, sb * 144, (int)tile_row0(tile, p.n_ff), &raw_full[slot]);
                if (g == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                bulk_g2s_hint(st + RAW_BYTES, p.x_img + (size_t)sb * btile_bytes<NBP>(), (uint32_t)btile_bytes<NBP>(),
                              &raw_full[slot], pol);
                __threadfence_block();
                *issued = g + 1;
                if (++sb == nb) { sb = 0; ++tile; }
            }
        }
        return;
    }

    // ---------------- compute warps ----------------
    const int q = warp >> 2, r4 = warp & 3;
    const int g8 = lane >> 2, tig = lane & 3;
    float yacc[MT][4][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) yacc[mt][nt][0] = yacc[mt][nt][1] = 0.f;
    bool dead = false;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // before any store of y or partials
    const int first_tile = (int)(i0 / nb);
    int tile = first_tile, sb = (int)(i0 % nb);
    for (int g = 0; g < count; ++g) {
        if ((g & (MMA_GROUPS - 1)) == q) {
            const int slot = g % NSR;
            const uint32_t ph = (uint32_t)(g / NSR) & 1u;
            if (!dead && !wait_issued(issued, g)) dead = true;
            if (!dead && !mbar_wait(&raw_full[slot], ph)) dead = true;
            const uint8_t *st = ring + slot * STAGE;
            const uint8_t *xt = st + RAW_BYTES;
            if (!dead) {
                // B rows of this thread: 32 r4 + 8 nt + g8, 1152 bytes apart
                const uint8_t *rb = st + (32 * r4 + g8) * 144;
                uint32_t scw[4][2], mnw[4][2];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const uint4 hd = *reinterpret_cast<const uint4 *>(rb + nt * 1152);
                    // 6-bit scales and mins of sub-blocks 0-3 and 4-7
                    scw[nt][0] = hd.y & 0x3F3F3F3Fu;
                    scw[nt][1] = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
                    mnw[nt][0] = hd.z & 0x3F3F3F3Fu;
                    mnw[nt][1] = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
                }
                float acc[MT][4][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // (sc * 2^9) pairs of sub-blocks 2c (low nibbles) and 2c+1
                    // (high nibbles): the codes come as q * 2^-9 from the e4m3
                    // conversion, and sc*q <= 945 is exact in fp16
                    uint32_t Slo[4], Shi[4];
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        const uint32_t w = scw[nt][c >> 1];
                        Slo[nt] = hmul2_u(byte_h2(w, 2 * (c & 1)), kH2_512);
                        Shi[nt] = hmul2_u(byte_h2(w, 2 * (c & 1) + 1), kH2_512);
                    }
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        const int slo = 4 * c + pp, shi = slo + 2;
                        uint4 alo[MT], ahi[MT];
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            alo[mt] = *reinterpret_cast<const uint4 *>(xt + ((size_t)(slo * MT + mt) * 32 + lane) * 16);
                            ahi[mt] = *reinterpret_cast<const uint4 *>(xt + ((size_t)(shi * MT + mt) * 32 + lane) * 16);
                        }
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
                            const uint32_t w = *reinterpret_cast<const uint32_t *>(rb + nt * 1152 + 16 + 32 * c + 16 * pp + 4 * tig);
                            // positions 4tig, 4tig+1 (b0, b2) and 4tig+2, 4tig+3 (b1, b3)
                            uint32_t b0, b1, b2, b3;
                            nibble_bytes_h2(w & 0x0F0F0F0Fu, b0, b1);
                            nibble_bytes_h2((w >> 4) & 0x0F0F0F0Fu, b2, b3);
                            b0 = hmul2_u(b0, Slo[nt]);
                            b1 = hmul2_u(b1, Slo[nt]);
                            b2 = hmul2_u(b2, Shi[nt]);
                            b3 = hmul2_u(b3, Shi[nt]);
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                mma_16816(acc[mt][nt], alo[mt], b0, b1);
                                mma_16816(acc[mt][nt], ahi[mt], b2, b3);
                            }
                        }
                    }
                }
                // mins: K slots 2tig, 2tig+1 = sub-blocks 2tig, 2tig+1; slots 8..15 zero
                float mins[MT][4][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint2 am = *reinterpret_cast<const uint2 *>(xt + xmain_bytes<NBP>() + ((size_t)mt * 32 + lane) * 8);
                    const uint4 a = make_uint4(am.x, am.y, 0u, 0u);
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        mins[mt][nt][0] = mins[mt][nt][1] = mins[mt][nt][2] = mins[mt][nt][3] = 0.f;
                        const uint32_t bm = bytes_h2((tig >> 1) ? mnw[nt][1] : mnw[nt][0], 2u * (uint32_t)(tig & 1));
                        mma_16816(mins[mt][nt], a, bm, 0u);
                    }
                }
                // y += 2^-e * (d * main - dmin * mins) for rows 2tig, 2tig+1 of each n8 block
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int rc = 32 * r4 + 8 * nt + 2 * tig;
                    const uint32_t dd0 = *reinterpret_cast<const uint32_t *>(st + rc * 144);
                    const uint32_t dd1 = *reinterpret_cast<const uint32_t *>(st + (rc + 1) * 144);
                    const float d0 = h2f(dd0), m0 = h2f(dd0 >> 16), d1 = h2f(dd1), m1 = h2f(dd1 >> 16);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const float undo = *reinterpret_cast<const float *>(xt + xscale_off<NBP>() + 4 * (8 * mt + g8));
                        const float v0 = fmaf(d0, acc[mt][nt][0] + acc[mt][nt][2], -m0 * (mins[mt][nt][0] + mins[mt][nt][2]));
                        const float v1 = fmaf(d1, acc[mt][nt][1] + acc[mt][nt][3], -m1 * (mins[mt][nt][1] + mins[mt][nt][3]));
                        yacc[mt][nt][0] = fmaf(v0, undo, yacc[mt][nt][0]);
                        yacc[mt][nt][1] = fmaf(v1, undo, yacc[mt][nt][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[slot]);
        }

        if (sb == nb - 1 || g == count - 1) {
            // the CTA's part of this tile is complete: add the groups' sums
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int rc = 32 * r4 + 8 * nt + 2 * tig, col = 8 * mt + g8;
                    red[((size_t)q * TM + rc) * NBP + col] = yacc[mt][nt][0];
                    red[((size_t)q * TM + rc + 1) * NBP + col] = yacc[mt][nt][1];
                    yacc[mt][nt][0] = yacc[mt][nt][1] = 0.f;
                }
            named_sync(1, MMA_COMPUTE_WARPS * 32);
            const long long t0i = (long long)tile * nb;
            const int cf = item_owner(t0i, p.total, grid), cl = item_owner(t0i + nb - 1, p.total, grid);
            for (int idx = threadIdx.x; idx < TM * NBP; idx += MMA_COMPUTE_WARPS * 32) {
                const int r = idx / NBP, b = idx % NBP;
                float v = red[(size_t)r * NBP + b];
#pragma unroll
                for (int qq = 1; qq < MMA_GROUPS; ++qq) v += red[((size_t)qq * TM + r) * NBP + b];
                if (cf == cl && p.n_ff > 0) {
                    p.ytmp[((size_t)tile * TM + r) * NBP + b] = v;
                } else if (cf == cl) {
                    const int row = tile * TM + r;
                    if (row < p.n_out && b < p.nb_cols)
                        p.y[(size_t)b * p.ldy + row] = p.bias ? v + p.bias[row] : v;
                } else {
                    const int side = tile == first_tile ? 0 : 1;
                    p.partials[((size_t)(blockIdx.x * 2 + side) * TM + r) * NBP + b] = v;
                }
            }
            named_sync(1, MMA_COMPUTE_WARPS * 32);
        }
        if (++sb == nb) { sb = 0; ++tile; }
    }
}

// Split-K finish: block c adds up the tile whose first contributor is CTA c
// (the last tile of c's range, when later CTAs share it), parts in CTA order.
// Launched after the main kernel with programmatic dependent launch: it can be
// resident beside it and waits for the main grid to complete.
template <int NBP>
__global__ void __launch_bounds__(TM) tc_finish(const float *__restrict__ partials, float *__restrict__ y,
                                               long long ldy, long long total, int nb, int n_out, int nb_cols,
                                               const float *__restrict__ bias) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int grid = (int)gridDim.x, c = (int)blockIdx.x;
    const long long last_item = item_begin(c + 1, total, grid) - 1;
    const int tile = (int)(last_item / nb);
    const long long t0 = (long long)tile * nb;
    if (item_owner(t0, total, grid) != c) return;                  // c is not the tile's first contributor
    const int cl = item_owner(t0 + nb - 1, total, grid);
    if (cl == c) return;                                            // not split
    const int r = threadIdx.x, row = tile * TM + r;
    float sum[NBP];
#pragma unroll
    for (int b = 0; b < NBP; ++b) sum[b] = 0.f;
    // four contributors' parts in flight at a time, added in CTA order
    for (int c0 = c; c0 <= cl; c0 += 4) {
        float4 v[4][NBP / 4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int cc = c0 + u;
            if (cc <= cl) {
                const int side = tile == (int)(item_begin(cc, total, grid) / nb) ? 0 : 1;
                const float4 *part = reinterpret_cast<const float4 *>(partials + ((size_t)(cc * 2 + side) * TM + r) * NBP);
#pragma unroll
                for (int b4 = 0; b4 < NBP / 4; ++b4) v[u][b4] = part[b4];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (c0 + u <= cl) {
#pragma unroll
                for (int b4 = 0; b4 < NBP / 4; ++b4) {
                    sum[4 * b4 + 0] += v[u][b4].x;
                    sum[4 * b4 + 1] += v[u][b4].y;
                    sum[4 * b4 + 2] += v[u][b4].z;
                    sum[4 * b4 + 3] += v[u][b4].w;
                }
            }
        }
    }
    if (row < n_out) {
        const float bv = bias ? bias[row] : 0.f;
#pragma unroll
        for (int b = 0; b < NBP; ++b)
            if (b < nb_cols) y[(size_t)b * ldy + row] = bias ? sum[b] + bv : sum[b];
    }
}

// The sums of row r of tile t for all NBP columns: from ytmp when one CTA
// computed the whole tile, else its CTAs' partial sums added in CTA order
// (the loads of up to four parts in flight at a time).
template <int NBP>
__device__ __forceinline__ void tile_sums(float (&sum)[NBP], int t, int r, const float *__restrict__ partials,
                                          const float *__restrict__ ytmp, long long total, int nb, int grid) {
    const long long t0 = (long long)t * nb;
    const int cf = item_owner(t0, total, grid), cl = item_owner(t0 + nb - 1, total, grid);
    if (cf == cl) {
        const float4 *v = reinterpret_cast<const float4 *>(ytmp + ((size_t)t * TM + r) * NBP);
#pragma unroll
        for (int b4 = 0; b4 < NBP / 4; ++b4) {
            const float4 q = v[b4];
            sum[4 * b4] = q.x; sum[4 * b4 + 1] = q.y; sum[4 * b4 + 2] = q.z; sum[4 * b4 + 3] = q.w;
        }
        return;
    }
#pragma unroll
    for (int b = 0; b < NBP; ++b) sum[b] = 0.f;
    for (int c0 = cf; c0 <= cl; c0 += 4) {
        float4 v[4][NBP / 4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int cc = c0 + u;
            if (cc <= cl) {
                const int side = t == (int)(item_begin(cc, total, grid) / nb) ? 0 : 1;
                const float4 *part = reinterpret_cast<const float4 *>(partials + ((size_t)(cc * 2 + side) * TM + r) * NBP);
#pragma unroll
                for (int b4 = 0; b4 < NBP / 4; ++b4) v[u][b4] = part[b4];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (c0 + u <= cl) {
#pragma unroll
                for (int b4 = 0; b4 < NBP / 4; ++b4) {
                    sum[4 * b4] += v[u][b4].x; sum[4 * b4 + 1] += v[u][b4].y;
                    sum[4 * b4 + 2] += v[u][b4].z; sum[4 * b4 + 3] += v[u][b4].w;
                }
            }
        }
    }
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z) with CUDA's expf (PESTI README,
// "Conformance": the MLP multiplies silu of the gate projection by the up
// projection).
__device__ __forceinline__ float silu_tc(float z) { return z / (1.0f + expf(-z)); }

// SwiGLU finish: block i forms h[b][128i + r] = silu(gate) * up from tiles 2i
// (gate rows) and 2i+1 (up rows).  Launched after the main kernel with
// programmatic dependent launch, like tc_finish.
template <int NBP>
__global__ void __launch_bounds__(2 * TM) tc_finish_swiglu(const float *__restrict__ partials,
                                                      const float *__restrict__ ytmp, float *__restrict__ h,
                                                      long long ldh, long long total, int nb, int grid, int n_ff,
                                                      int nb_cols) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // threads 0..127 sum the gate tile's row r, threads 128..255 the up tile's;
    // the up sums reach the gate thread through shared memory
    __shared__ float up_s[TM][NBP + 1];
    const int i = (int)blockIdx.x, r = threadIdx.x % TM, half = threadIdx.x / TM;
    float v[NBP];
    tile_sums<NBP>(v, 2 * i + half, r, partials, ytmp, total, nb, grid);
    if (half) {
#pragma unroll
        for (int b = 0; b < NBP; ++b) up_s[r][b] = v[b];
    }
    __syncthreads();
    const int j = i * TM + r;
    if (!half && j < n_ff) {
#pragma unroll
        for (int b = 0; b < NBP; ++b)
            if (b < nb_cols) h[(size_t)b * ldh + j] = silu_tc(v[b]) * up_s[r][b];
    }
}

// Whether any tile is split over several CTAs (same arithmetic as item_begin/item_owner).
bool any_split(long long total, int nb, int grid) {
    for (int c = 0; c < grid; ++c) {
        const long long last_item = ((long long)(c + 1) * total) / grid - 1;
        const long long t0 = last_item / nb * nb;
        const int cf = (int)(((t0 + 1) * grid - 1) / total), cl = (int)(((t0 + nb) * grid - 1) / total);
        if (cf == c && cl != c) return true;
    }
    return false;
}

// ---------------------------------------------------------------- host side
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(ptr);
    });
    return fn;
}


// CTAs for a call: one per SM, at most one per work item.  When there are no
// more row tiles than CTAs, one whole tile per CTA avoids the split-K
// finishing kernel (about four super-blocks' time per call); that is chosen
// when it costs each CTA at most five super-blocks more than an even split
// (14336x4096: 16 instead of 12 super-blocks per CTA).
// Row tiles of a call: 128-row tiles of the matrix, or for the SwiGLU
// epilogue a gate tile and an up tile per 128 pairs.
long long tc_tiles(int64_t n_out, const Epilogue &epi) {
    return epi.kind == kEpiSwiGLU ? 2 * ((n_out / 2 + TM - 1) / TM) : (n_out + TM - 1) / TM;
}

int tc_grid(int64_t n_out, int64_t k, const DeviceInfo &dev, const Epilogue &epi = Epilogue{}) {
    const long long ntiles = tc_tiles(n_out, epi), nb = k / 256;
    const long long total = ntiles * nb;
    long long g = dev.sm_count < kMaxGrid ? dev.sm_count : kMaxGrid;
    if (g > total) g = total;
    if (g < 1) g = 1;
    if (ntiles <= g && nb - (total + g - 1) / g <= 5) g = ntiles;
    return (int)g;
}

// Scratch of one call: x image, split-K partial sums, and for the SwiGLU
// epilogue the whole tiles' sums [tiles][TM][NBP].
template <int NBP> size_t scratch_bytes_epi(int64_t n_out, int64_t k, int grid, const Epilogue &epi) {
    return scratch_bytes<NBP>(k, grid) + (epi.kind == kEpiSwiGLU ? (size_t)tc_tiles(n_out, epi) * TM * NBP * 4 : 0);
}

// The register-operand kernel for 1-8 columns (PQ_TC_MMA=0 builds the
// tensor-memory kernel there instead); 9-32 columns take the tensor-memory
// kernel (at 16 columns the register-operand kernel is slower: 24.6 against
// 19.3 us at 14336x4096, its accumulators spill at 96 registers).
#ifndef PQ_TC_MMA
#define PQ_TC_MMA 1
#endif
template <int NBP> constexpr bool use_mma() { return PQ_TC_MMA && NBP == 8; }

template <int NBP>
cudaError_t launch_nbp(const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch, float *y,
                       int64_t ldy, cudaStream_t s, int grid, uint8_t *scratch, const Epilogue &epi = Epilogue{}) {
    constexpr bool MMA = use_mma<NBP>();
    const int nb = (int)(k / 256);
    uint8_t *img = scratch;
    float *partials = reinterpret_cast<float *>(scratch + scratch_img_bytes<NBP>(k));
    float *ytmp = reinterpret_cast<float *>(scratch + scratch_bytes<NBP>(k, grid));
    const bool swiglu = epi.kind == kEpiSwiGLU;
    const int n_ff = swiglu ? (int)(n_out / 2) : 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3(nb);
    pcfg.blockDim = dim3(256);
    pcfg.stream = s;
    pcfg.attrs = attr;
    pcfg.numAttrs = 1;
    cudaError_t e;
    if constexpr (MMA)
        e = cudaLaunchKernelEx(&pcfg, prep_x_mma<NBP>, x, (int)k, batch, img);
    else
        e = cudaLaunchKernelEx(&pcfg, prep_x_tc<NBP>, x, (int)k, batch, img);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    EncodeTiled enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)(nb * 144), (cuuint64_t)n_out};
    const cuuint64_t gstride[1] = {(cuuint64_t)(nb * 144)};
    const cuuint32_t box[2] = {144u, (cuuint32_t)TM};
    const cuuint32_t estride[2] = {1u, 1u};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w), gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    static PerDeviceOnce configured;
    e = configured.run([] {
        if constexpr (MMA)
            return cudaFuncSetAttribute(gemv_mma_q4_k<NBP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        mma_smem_bytes<NBP>());
        else
            return cudaFuncSetAttribute(gemv_tc_q4_k<NBP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_bytes<NBP>());
    });
    static_assert(tc_threads<NBP>() <= 1024, "block size");
    if (e != cudaSuccess) return e;
    const long long ntiles = tc_tiles(n_out, epi);
    const long long total = ntiles * nb;
    TcParams p{img, y, partials, (long long)ldy, total, (int)n_out, (int)k, batch,
               epi.kind == kEpiBias ? epi.bias : nullptr, n_ff, swiglu ? ytmp : nullptr};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(MMA ? MMA_THREADS : tc_threads<NBP>());
    cfg.dynamicSmemBytes = (size_t)(MMA ? mma_smem_bytes<NBP>() : smem_bytes<NBP>());
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (MMA)
        e = cudaLaunchKernelEx(&cfg, gemv_mma_q4_k<NBP>, map, p);
    else
        e = cudaLaunchKernelEx(&cfg, gemv_tc_q4_k<NBP>, map, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(TM);
    cfg.dynamicSmemBytes = 0;
    if (swiglu) {
        cfg.gridDim = dim3((unsigned)(ntiles / 2));
        cfg.blockDim = dim3(2 * TM);
        e = cudaLaunchKernelEx(&cfg, tc_finish_swiglu<NBP>, (const float *)partials, (const float *)ytmp, y,
                               (long long)ldy, total, nb, grid, n_ff, batch);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    if (!any_split(total, nb, grid)) return e;
    cfg.gridDim = dim3(grid);
    e = cudaLaunchKernelEx(&cfg, tc_finish<NBP>, (const float *)partials, y, (long long)ldy, total, nb, (int)n_out,
                           batch, p.bias);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Fixed scratch for the allocation-free entry point (pq_gemv_noalloc): x image
// for k up to kNoAllocMaxK at up to 16 columns and split-K partial sums for up
// to kMaxGrid CTAs: 3,743,744 bytes.  Every GPU that loads
// this library keeps it until the process exits.  In host code the name is
// only a stand-in for the device array; its device address comes from
// cudaGetSymbolAddress, once per device.
constexpr int kNoAllocMaxK = 16384;
constexpr size_t kNoAllocScratchBytes =
    (size_t)(kNoAllocMaxK / 256) * (size_t)btile_bytes<16>() + (size_t)kMaxGrid * 2 * 16 * TM * 4;
static_assert(kNoAllocScratchBytes == 3743744, "stated size");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

uint8_t *noalloc_scratch_ptr() {
    static uint8_t *ptrs[64] = {};
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::call_once(once[dev], [dev] {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) == cudaSuccess) ptrs[dev] = static_cast<uint8_t *>(ptr);
    });
    return ptrs[dev];
}

}  // namespace

int noalloc_max_k() { return kNoAllocMaxK; }

cudaError_t launch_gemv_tc_noalloc(const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch,
                                   float *y, int64_t ldy, cudaStream_t s, const DeviceInfo &dev) {
    if (!tc_supported(PQ_Q4_K, n_out, k, batch) || batch > 16 || k > kNoAllocMaxK) return cudaErrorInvalidValue;
    uint8_t *scratch = noalloc_scratch_ptr();
    if (!scratch) return cudaErrorInvalidSymbol;
    const int grid = tc_grid(n_out, k, dev);
    return batch <= 8 ? launch_nbp<8>(w, n_out, k, x, batch, y, ldy, s, grid, scratch)
                      : launch_nbp<16>(w, n_out, k, x, batch, y, ldy, s, grid, scratch);
}

unsigned tc_wait_timeouts(bool reset) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) return 0;
    if (reset) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_wait_timeouts, &z, sizeof(z));
    }
    return v;
}

bool tc_supported(int fmt, int64_t n_out, int64_t k, int batch) {
    return fmt == PQ_Q4_K && batch >= 1 && batch <= 32 && n_out >= 1 && k % 256 == 0 && k >= 256 &&
           k <= 65536;
}

cudaError_t launch_gemv_tc(int fmt, const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch,
                           float *y, int64_t ldy, cudaStream_t s, const DeviceInfo &dev, const Epilogue &epi) {
    if (!tc_supported(fmt, n_out, k, batch)) return cudaErrorInvalidValue;
    if (epi.kind == kEpiSwiGLU && (n_out % 2 || n_out < 2)) return cudaErrorInvalidValue;
    const int grid = tc_grid(n_out, k, dev, epi);
    const size_t bytes = batch <= 8    ? scratch_bytes_epi<8>(n_out, k, grid, epi)
                         : batch <= 16 ? scratch_bytes_epi<16>(n_out, k, grid, epi)
                                       : scratch_bytes_epi<32>(n_out, k, grid, epi);
    cudaMemPool_t pool = scratch_pool();
    if (!pool) return cudaErrorMemoryAllocation;
    void *scratch = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&scratch, bytes, pool, s);
    if (e != cudaSuccess) return e;
    e = batch <= 8    ? launch_nbp<8>(w, n_out, k, x, batch, y, ldy, s, grid, (uint8_t *)scratch, epi)
        : batch <= 16 ? launch_nbp<16>(w, n_out, k, x, batch, y, ldy, s, grid, (uint8_t *)scratch, epi)
                      : launch_nbp<32>(w, n_out, k, x, batch, y, ldy, s, grid, (uint8_t *)scratch, epi);
    const cudaError_t f = cudaFreeAsync(scratch, s);
    return e != cudaSuccess ? e : f;
}

}  // namespace pqk

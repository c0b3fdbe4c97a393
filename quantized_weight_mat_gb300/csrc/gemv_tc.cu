// Tensor-core fused dequant + mat-vec for Q4_K at batch 5..16 (tcgen05).
//
// The operation is the same fused "dequantize + mat-vec" (ember pull request,
// quant.rs description) on GGUF-style Q4_K super-blocks (PESTI README, "What
// This Is"), for several x columns at once.  At batch 8-16 each weight feeds
// 8-16 multiply-adds, too many for CUDA cores at HBM speed, so the products go
// to the 5th-generation tensor cores while the weights still stream once.
//
// Exactness: a tile entry is the integer sc_j*q (q in 0..15, sc_j in 0..63,
// so <= 945), exactly representable in fp16; x enters as two fp16 columns
// (x_hi = fp16(x), x_lo = fp16(x - x_hi)), so every product is exact in the
// f32 accumulator and only accumulation rounds.  The sub-block mins enter
// through a second, K=16 product of the 6-bit mins with the fp16 hi/lo sums
// of x over each 32-element sub-block.  Per super-block and row the epilogue
// forms y += d*(A.x) - dmin*(m.XS) in f32.
//
// Pipeline (one CTA per SM, persistent over 128-row tiles):
//   warp 12 producer: a 2-D TMA load (tensor map over W as [n_out][row bytes])
//           brings one 128-row x 144-byte super-block column per stage, and a
//           1-D bulk copy brings that super-block's fp16 x tile;
//   warps 0-7 decoders: thread (r, h) turns the 128 weights of row r, half h
//           of the super-block into fp16 sc*q (one LOP3 + one HFMA2 per two
//           weights), 64 weights per slot, and write them straight into
//           tensor memory (tcgen05.st; TMEM lane = row, two K values per
//           column), a ring of eight slots (two super-blocks);
//   warp 13 MMA issuer (one thread): per super-block the K=16 mins product
//           (A from shared memory), then four tcgen05.mma (M=128, N=2*NBP,
//           K=16, A from tensor memory, x from shared memory) per slot into a
//           TMEM accumulator;
//   warps 8-11 epilogue: tcgen05.ld of the accumulators (warp w reads TMEM
//           lanes 32(w%4).. = its rows), d and dmin from a small ring the
//           decoders fill, f32 scaling.
// Accumulators are double-buffered in TMEM; every mbarrier wait is bounded.
//
// x is converted once per call by a small kernel into a per-super-block fp16
// image (the operand layout the MMA reads), in a stream-ordered scratch
// buffer.

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
constexpr int A_SLOTS = 8;                    // two super-blocks of 64-weight slots, in TMEM
constexpr int A_COL = 256;                    // TMEM column of A slot 0 (32 columns per slot)
constexpr int TMEM_COLS = 512;
constexpr int AMIN_BYTES = TM * 16 * 2;
constexpr int THREADS = 14 * 32;              // 8 decoder, 4 epilogue, producer, MMA warps

// x image of one super-block for N' = 2*NBP columns: main part N' x 256 fp16
// (K-major, 8x8 core matrices), then the mins part N' x 16.
template <int NP> __host__ __device__ constexpr int btile_bytes() { return NP * 256 * 2 + NP * 16 * 2; }
template <int NP> __host__ __device__ constexpr int raw_stages() { return NP == 32 ? 5 : 7; }
template <int NP> __host__ __device__ constexpr int stage_bytes() { return RAW_BYTES + btile_bytes<NP>(); }
template <int NP> __host__ __device__ constexpr int smem_bytes() {
    return raw_stages<NP>() * stage_bytes<NP>() + 2 * AMIN_BYTES + 1024;
}

// K order inside a super-block: chunk e of A-column a (8 fp16 per 16 bytes)
// holds weight position pos(a, e).  It follows how two qs words turn into
// four half2 pairs: low nibbles of bytes (0,2), then (1,3), of each word.
__host__ __device__ constexpr int perm8(int e) { return (e & 4) | ((e & 1) << 1) | ((e >> 1) & 1); }
__host__ __device__ constexpr int kpos(int a, int e) {
    return 64 * (a / 8) + 32 * ((a % 8) / 4) + 8 * (a % 4) + perm8(e);
}

// byte offset of element (n, K) in a K-major no-swizzle operand whose 8-row
// groups are `sbo` bytes apart (core matrices of 8 rows x 16 bytes, K-adjacent
// core matrices 128 bytes apart)
__host__ __device__ constexpr int kmaj_off(int n, int K, int sbo) {
    return (n / 8) * sbo + (K / 8) * 128 + (n % 8) * 16 + (K % 8) * 2;
}

// ---------------------------------------------------------------- x image
// One block per super-block.  Lets the main kernel launch at once
// (programmatic dependent launch): it sets up and streams weights while this
// runs, and waits for it only before its first x tile.
template <int NBP>
__global__ void __launch_bounds__(256) prep_x_tc(const float *__restrict__ x, int k, int nb_cols,
                                                 uint8_t *__restrict__ img) {
    constexpr int NP = 2 * NBP;
    asm volatile("griddepcontrol.launch_dependents;");
    const int sb = blockIdx.x;
    __half *out = reinterpret_cast<__half *>(img + (size_t)sb * btile_bytes<NP>());
    __shared__ float xs[NBP][8];
    const int t = threadIdx.x;
    // sub-block sums, fixed order (thread per (column, sub-block), 8 vector loads)
    if (t < NBP * 8) {
        const int b = t / 8, j = t % 8;
        float s = 0.f;
        if (b < nb_cols) {
            const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)b * k + sb * 256 + 32 * j);
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __ldg(xb + i);
#pragma unroll
            for (int i = 0; i < 8; ++i) s = s + v[i].x + v[i].y + v[i].z + v[i].w;
        }
        xs[b][j] = s;
    }
    // main part: thread t = K index; all column loads in flight together
    {
        const int K = t;
        const int pos = kpos(K / 8, K % 8);
        float v[NBP];
#pragma unroll
        for (int b = 0; b < NBP; ++b) v[b] = b < nb_cols ? __ldg(x + (size_t)b * k + sb * 256 + pos) : 0.f;
#pragma unroll
        for (int b = 0; b < NBP; ++b) {
            const __half hi = __float2half_rn(v[b]);
            const __half lo = __float2half_rn(v[b] - __half2float(hi));
            out[kmaj_off(b, K, 4096) / 2] = hi;
            out[kmaj_off(NBP + b, K, 4096) / 2] = lo;
        }
    }
    __syncthreads();
    // mins part: K = j < 8 holds the sums, K = 8..15 zero
    __half *om = out + NP * 256;
    for (int i = t; i < NP * 16; i += 256) {
        const int n = i / 16, K = i % 16;
        const int b = n % NBP;
        float v = 0.f;
        if (K < 8) {
            const float s = xs[b][K];
            const __half hi = __float2half_rn(s);
            v = n < NBP ? __half2float(hi) : __half2float(__float2half_rn(s - __half2float(hi)));
        }
        om[kmaj_off(n, K, 256) / 2] = __float2half_rn(v);
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
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b),
                              *reinterpret_cast<const __half2 *>(&c));
    return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<const uint32_t *>(&v); }

struct TcParams {
    const uint8_t *w;          // for L2 prefetch of whole tiles (rows are contiguous)
    const uint8_t *x_img;
    float *y;
    long long ldy;
    int n_out;
    int k;
    int nb_cols;
};

template <int NBP>
__global__ void __launch_bounds__(THREADS, 1)
    gemv_tc_q4_k(const __grid_constant__ CUtensorMap wmap, TcParams p) {
    constexpr int NP = 2 * NBP;
    constexpr int NSR = raw_stages<NP>();
    constexpr int STAGE = stage_bytes<NP>();
    constexpr uint32_t IDESC = instr_desc(TM, NP);
    static_assert(4 * NP <= A_COL, "accumulators below the A slots");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t raw_full[NSR], raw_empty[NSR];
    __shared__ __align__(8) uint64_t a_full[A_SLOTS], a_empty[A_SLOTS];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ __align__(8) uint64_t dmeta_full[4];
    __shared__ float2 dmeta[4][TM];      // (d, dmin) of each row, per super-block
    __shared__ uint32_t tmem_base_sh;

    // 1024-aligned working area
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *ring = smem;
    uint8_t *amin = ring + NSR * STAGE;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = p.k / 256;
    const int ntiles = (p.n_out + TM - 1) / TM;
    const int my_tiles = ntiles > (int)blockIdx.x ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_tiles * nb;    // super-block steps of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSR; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 1);
        }
        for (int s = 0; s < 4; ++s) mbar_init(&dmeta_full[s], 4);
        for (int s = 0; s < A_SLOTS; ++s) {
            mbar_init(&a_full[s], 4);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 4);
        }
        fence_mbar_init();
    }
    // zero the unused K = 8..15 half of both mins tiles (never rewritten)
    for (int i = threadIdx.x; i < 2 * TM; i += THREADS) {
        const int buf = i / TM, r = i % TM;
        *reinterpret_cast<uint4 *>(amin + buf * AMIN_BYTES + kmaj_off(r, 8, 256)) = make_uint4(0, 0, 0, 0);
    }
    if (warp == 13) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_sh)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 12) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = make_evict_first_policy();
            bool dead = false;
            for (int g = 0; g < total && !dead; ++g) {
                const int slot = g % NSR;
                const uint32_t ph = (uint32_t)(g / NSR) & 1u;
                const int tile = (int)blockIdx.x + (g / nb) * (int)gridDim.x, sb = g % nb;
                if (!mbar_wait(&raw_empty[slot], ph ^ 1u)) { dead = true; break; }
                uint8_t *st = ring + slot * STAGE;
                mbar_arrive_expect_tx(&raw_full[slot], (uint32_t)STAGE);
                tma_load_2d(st, &wmap, sb * 144, tile * TM, &raw_full[slot]);
                // the weights were complete before the x-prep kernel started; the x
                // image is that kernel's output: wait for it once, before its first use
                if (g == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                bulk_g2s_hint(st + RAW_BYTES, p.x_img + (size_t)sb * btile_bytes<NP>(), (uint32_t)btile_bytes<NP>(),
                              &raw_full[slot], pol);
            }
        }
    } else if (warp == 13) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            bool dead = false;
            for (int g = 0; g < total; ++g) {
                const int slot = g % NSR;
                const uint32_t ph = (uint32_t)(g / NSR) & 1u;
                const int buf = g & 1;
                const int a0 = 4 * buf;                       // A slots of this super-block
                const uint32_t aph = (uint32_t)(g >> 1) & 1u;
                if (!dead && !mbar_wait(&acc_empty[buf], ((uint32_t)(g >> 1) & 1u) ^ 1u)) dead = true;
                if (!dead && !mbar_wait(&raw_full[slot], ph)) dead = true;
                // the mins rows are complete once both halves' first slots are
                if (!dead && !mbar_wait(&a_full[a0], aph)) dead = true;
                if (!dead && !mbar_wait(&a_full[a0 + 2], aph)) dead = true;
                tc_fence_after();
                const uint32_t d_main = tmem + (uint32_t)(buf * 2 * NP);
                const uint32_t d_min = d_main + NP;
                const uint32_t bbase = smem_u32(ring + slot * STAGE + RAW_BYTES);
                {
                    const uint64_t ad = smem_desc(smem_u32(amin + buf * AMIN_BYTES), 128u, 256u);
                    const uint64_t bd = smem_desc(bbase + NP * 256 * 2, 128u, 256u);
                    if (!dead) mma_f16(d_min, ad, bd, IDESC, 0u);
                }
                for (int c = 0; c < 4; ++c) {
                    if ((c & 1) && !dead && !mbar_wait(&a_full[a0 + c], aph)) dead = true;
                    tc_fence_after();
                    const uint32_t acol = tmem + (uint32_t)(A_COL + 32 * (a0 + c));
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t bd = smem_desc(bbase + 256u * (4 * c + ks), 128u, 4096u);
                        if (!dead) mma_f16_ta(d_main, acol + 8u * ks, bd, IDESC, (c | ks) ? 1u : 0u);
                    }
                    mma_commit(&a_empty[a0 + c]);
                }
                mma_commit(&acc_full[buf]);
                mma_commit(&raw_empty[slot]);
            }
        }
    } else if (warp >= 8) {
        // ---------------- epilogue (warps 8-11) ----------------
        const int r = 32 * (warp - 8) + lane;           // row within the tile = TMEM lane
        const uint32_t row_taddr = tmem + ((uint32_t)(32 * (warp - 8)) << 16);
        float yacc[NBP];
#pragma unroll
        for (int b = 0; b < NBP; ++b) yacc[b] = 0.f;
        bool dead = false;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // before any store of y
        for (int g = 0; g < total; ++g) {
            const int buf = g & 1;
            if (!dead && !mbar_wait(&acc_full[buf], (uint32_t)(g >> 1) & 1u)) dead = true;
            tc_fence_after();
            uint32_t v[2 * NP];
            {
                uint32_t t0[32];
                tmem_ld32(row_taddr + (uint32_t)(buf * 2 * NP), t0);
                if constexpr (NP == 32) {
                    uint32_t t1[32];
                    tmem_ld32(row_taddr + (uint32_t)(buf * 2 * NP + 32), t1);
                    tmem_ld_wait(t1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[32 + i] = t1[i];
                }
                tmem_ld_wait(t0);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = t0[i];
            }
            tc_fence_before();
            if (!dead && !mbar_wait(&dmeta_full[g & 3], (uint32_t)(g >> 2) & 1u)) dead = true;
            const float2 dm = dmeta[g & 3][r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            const float d = dm.x, dmin = dm.y;
#pragma unroll
            for (int b = 0; b < NBP; ++b) {
                const float dot = __uint_as_float(v[b]) + __uint_as_float(v[NBP + b]);
                const float mn = __uint_as_float(v[NP + b]) + __uint_as_float(v[NP + NBP + b]);
                yacc[b] = fmaf(d, dot, fmaf(-dmin, mn, yacc[b]));
            }
            if (g % nb == nb - 1) {
                const int tile = (int)blockIdx.x + (g / nb) * (int)gridDim.x;
                const int row = tile * TM + r;
                if (row < p.n_out) {
#pragma unroll
                    for (int b = 0; b < NBP; ++b)
                        if (b < p.nb_cols) p.y[(size_t)b * p.ldy + row] = yacc[b];
                }
#pragma unroll
                for (int b = 0; b < NBP; ++b) yacc[b] = 0.f;
            }
        }
    } else {
        // ---------------- decoders (warps 0-7) ----------------
        const int r = threadIdx.x & 127;        // row within the tile
        const int h = threadIdx.x >> 7;         // half of the super-block: sub-blocks 4h..4h+3
        const uint32_t mA = h ? 0x0F0F0F0Fu : 0x3F3F3F3Fu;
        const uint32_t mB = h ? 0x30303030u : 0u;
        const uint32_t a_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's TMEM lanes
        bool dead = false;
        for (int g = 0; g < total; ++g) {
            const int slot = g % NSR;
            const uint32_t ph = (uint32_t)(g / NSR) & 1u;
            const int buf = g & 1;
            const uint32_t aph = (uint32_t)(g >> 1) & 1u;
            if (!dead && !mbar_wait(&raw_full[slot], ph)) dead = true;
            const uint8_t *blk = ring + slot * STAGE + r * 144;
            const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
            uint4 qw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qw[i] = *reinterpret_cast<const uint4 *>(blk + 16 + 64 * h + 16 * i);
            // 6-bit scales / mins of sub-blocks 4h..4h+3, one per byte
            const uint32_t sc4 = ((h ? hd.w : hd.y) & mA) | ((hd.y >> 2) & mB);
            const uint32_t m4 = ((h ? (hd.w >> 4) : hd.z) & mA) | ((hd.z >> 2) & mB);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * h + cc;           // 64-weight chunk of the super-block
                const int as = 4 * buf + c;         // its A slot
                if (!dead && !mbar_wait(&a_empty[as], aph ^ 1u)) dead = true;
                if (cc == 0 && h == 0) {
                    // (d, dmin) for the epilogue.  Slot g&3 was last read by the
                    // epilogue four super-blocks ago; the wait above implies the
                    // MMAs two super-blocks ago were issued, which waited for
                    // that epilogue to finish.
                    dmeta[g & 3][r] = make_float2(h2f(hd.x), h2f(hd.x >> 16));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dmeta_full[g & 3]);
                }
                if (cc == 0) {
                    // mins row of the K=16 product: m_{4h..4h+3} at K = 4h..4h+3.
                    // The wait above covers every product issued before this slot
                    // was last read, which includes the mins product that last
                    // read this buffer (two super-blocks ago): it is issued first.
                    const __half2 m01 = __halves2half2(__int2half_rn((int)(m4 & 0xFF)),
                                                       __int2half_rn((int)((m4 >> 8) & 0xFF)));
                    const __half2 m23 = __halves2half2(__int2half_rn((int)((m4 >> 16) & 0xFF)),
                                                       __int2half_rn((int)(m4 >> 24)));
                    *reinterpret_cast<uint2 *>(amin + buf * AMIN_BYTES + kmaj_off(r, 4 * h, 256)) =
                        make_uint2(h2_bits(m01), h2_bits(m23));
                }
                // scale pairs: low nibbles -> (1024+q)*sc - 1024*sc, high nibbles -> (1024+16q)*sc/16 - 64*sc
                const __half slo = __int2half_rn((int)((sc4 >> (16 * cc)) & 0xFF));
                const __half shi = __int2half_rn((int)((sc4 >> (16 * cc + 8)) & 0xFF));
                const uint32_t Slo = h2_bits(__halves2half2(slo, slo));
                const uint32_t Clo = h2_bits(__hmul2(__halves2half2(slo, slo), __float2half2_rn(-1024.0f)));
                const uint32_t Shi = h2_bits(__hmul2(__halves2half2(shi, shi), __float2half2_rn(0.0625f)));
                const uint32_t Chi = h2_bits(__hmul2(__halves2half2(shi, shi), __float2half2_rn(-64.0f)));
                const uint32_t w[8] = {qw[2 * cc].x, qw[2 * cc].y, qw[2 * cc].z, qw[2 * cc].w,
                                       qw[2 * cc + 1].x, qw[2 * cc + 1].y, qw[2 * cc + 1].z, qw[2 * cc + 1].w};
                // the slot's 64 K values of row r: TMEM column j holds K = 2j, 2j+1
                uint32_t R[32];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const uint32_t w0 = w[2 * a], w1 = w[2 * a + 1];
                    const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
                    R[4 * a + 0] = hfma2_u((w0 & 0x000F000Fu) | 0x64006400u, Slo, Clo);
                    R[4 * a + 1] = hfma2_u((s0 & 0x000F000Fu) | 0x64006400u, Slo, Clo);
                    R[4 * a + 2] = hfma2_u((w1 & 0x000F000Fu) | 0x64006400u, Slo, Clo);
                    R[4 * a + 3] = hfma2_u((s1 & 0x000F000Fu) | 0x64006400u, Slo, Clo);
                    R[16 + 4 * a + 0] = hfma2_u((w0 & 0x00F000F0u) | 0x64006400u, Shi, Chi);
                    R[16 + 4 * a + 1] = hfma2_u((s0 & 0x00F000F0u) | 0x64006400u, Shi, Chi);
                    R[16 + 4 * a + 2] = hfma2_u((w1 & 0x00F000F0u) | 0x64006400u, Shi, Chi);
                    R[16 + 4 * a + 3] = hfma2_u((s1 & 0x00F000F0u) | 0x64006400u, Shi, Chi);
                }
                tmem_st32(a_lane + (uint32_t)(A_COL + 32 * as), R);
                tmem_st_wait();
                if (cc == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // mins row
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[as]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
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

// Stream-ordered scratch for the x image: a library-owned memory pool per
// device that keeps freed memory for reuse.
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

template <int NBP>
cudaError_t launch_nbp(const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch, float *y,
                       int64_t ldy, cudaStream_t s, const DeviceInfo &dev, uint8_t *img) {
    constexpr int NP = 2 * NBP;
    const int nb = (int)(k / 256);
    prep_x_tc<NBP><<<nb, 256, 0, s>>>(x, (int)k, batch, img);
    cudaError_t e = cudaGetLastError();
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

    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(gemv_tc_q4_k<NBP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<NP>());
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int ntiles = (int)((n_out + TM - 1) / TM);
    const int grid = ntiles < dev.sm_count ? ntiles : dev.sm_count;
    TcParams p{w, img, y, (long long)ldy, (int)n_out, (int)k, batch};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = (size_t)smem_bytes<NP>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_tc_q4_k<NBP>, map, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Fixed scratch for the allocation-free entry point (pq_gemv_noalloc): the
// fp16 x image for k up to kNoAllocMaxK at up to 16 columns, 1,114,112 bytes.
// Every GPU that loads this library keeps it until the process exits.  In
// host code the name is only a stand-in for the device array; its device
// address comes from cudaGetSymbolAddress, once per device.
constexpr int kNoAllocMaxK = 16384;
constexpr size_t kNoAllocScratchBytes = (size_t)(kNoAllocMaxK / 256) * (size_t)btile_bytes<32>();
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
    if (!tc_supported(PQ_Q4_K, n_out, k, batch) || k > kNoAllocMaxK) return cudaErrorInvalidValue;
    uint8_t *img = noalloc_scratch_ptr();
    if (!img) return cudaErrorInvalidSymbol;
    return batch <= 8 ? launch_nbp<8>(w, n_out, k, x, batch, y, ldy, s, dev, img)
                      : launch_nbp<16>(w, n_out, k, x, batch, y, ldy, s, dev, img);
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
    return fmt == PQ_Q4_K && batch >= 1 && batch <= 16 && n_out >= 1 && k % 256 == 0 && k >= 256 &&
           k <= 65536;
}

cudaError_t launch_gemv_tc(int fmt, const uint8_t *w, int64_t n_out, int64_t k, const float *x, int batch,
                           float *y, int64_t ldy, cudaStream_t s, const DeviceInfo &dev) {
    if (!tc_supported(fmt, n_out, k, batch)) return cudaErrorInvalidValue;
    const int NP = batch <= 8 ? 16 : 32;
    const size_t bytes = (size_t)(k / 256) * (size_t)(NP * 256 * 2 + NP * 16 * 2);
    cudaMemPool_t pool = scratch_pool();
    if (!pool) return cudaErrorMemoryAllocation;
    void *img = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&img, bytes, pool, s);
    if (e != cudaSuccess) return e;
    e = batch <= 8 ? launch_nbp<8>(w, n_out, k, x, batch, y, ldy, s, dev, (uint8_t *)img)
                   : launch_nbp<16>(w, n_out, k, x, batch, y, ldy, s, dev, (uint8_t *)img);
    const cudaError_t f = cudaFreeAsync(img, s);
    return e != cudaSuccess ? e : f;
}

}  // namespace pqk

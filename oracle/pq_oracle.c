/*
 * pq_oracle.c -- plain, slow CPU oracle for the block-quantized mat-vec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  The CUDA
 * library never includes, links or calls anything here, and this file
 * includes nothing of the CUDA library.
 *
 * What it computes (the definition the GPU path is checked against):
 *   1. decode every quantized block to f32 by the layout rules below;
 *   2. y[b][r] = sum_i (double)w[r][i] * (double)x[b][i], summed in f64 in
 *      index order and returned in f64.
 * Source of the operation: the ember pull request ("Project scaffold:
 * modules, CLI, and correctness harness", quant.rs description) fuses the
 * decoding of W into the mat-vec so that no f32 copy of W is made; the
 * mat-vec is the row-major one that costs the most in a decode step (same
 * page, tensor.rs description); the block formats are the K family whose
 * decoding the PESTI README ("What This Is", "Architecture") reports as
 * exact to the byte.
 *
 * The pages never print a block's byte layout.  The layouts below are the
 * public GGUF layouts, read as a byte specification (sizes: Q8_0 34 B per
 * 32 weights, Q4_K 144 B per 256, Q6_K 210 B per 256, and for the rest of
 * the K family the PESTI README names, Q5_K 176 B, Q3_K 110 B, Q2_K 84 B
 * per 256).  Per-row int8 has
 * no published layout; the one used here is: int8 q[n_out*k] row-major,
 * then, at the next 16-byte boundary, float scale[n_out].  Per-row int4 (the
 * ember page lists int4 beside int8) likewise: two signed 4-bit codes per byte, weight
 * 2i in the low nibble of byte i and weight 2i+1 in the high nibble, rows of
 * k/2 bytes (k even), then float scale[n_out] at the next 16-byte boundary.
 *
 * Quantizers: the pages give none (PESTI dequantizes files made by other
 * tools).  The ones here are a plain, deterministic, non-iterative reading
 * (round to nearest, ties away from zero, f64 arithmetic, fp16 stored by
 * round-to-nearest-even).  They only make test inputs.
 *
 * Built with -O2 -ffp-contract=off so that every product and sum rounds
 * exactly as written.  Parity of the quantizers' f64->f16 step and of the
 * decoders is pinned by the CPU tests (library routines, closed forms,
 * brute force, bit flips).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { PQO_Q8_0 = 0, PQO_Q4_K = 1, PQO_Q6_K = 2, PQO_I8_ROW = 3, PQO_Q5_K = 4, PQO_Q3_K = 5, PQO_Q2_K = 6,
       PQO_I4_ROW = 7 };

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16                                                   */
/* ------------------------------------------------------------------ */

/* binary16 -> binary32, exact.  Written from the format's definition:
 * sign(1) exponent(5, bias 15) fraction(10); exponent 0 = zero/subnormal
 * (value = fraction * 2^-24), exponent 31 = inf/NaN. */
float pqo_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        if (f == 0)
            v = INFINITY;
        else
            return sign ? -NAN : NAN;
    } else {
        v = ldexp((double)(f + 1024), e - 25);
    }
    return (float)(sign ? -v : v);
}

/* binary64 -> binary16, round to nearest, ties to even; overflow -> inf.
 * Written from the definition: find the binary16 quantum for |v|'s binade
 * (2^(e-10) for normals, 2^-24 for subnormals), scale v to units of that
 * quantum (exact: a power-of-two scaling), round that to the nearest
 * integer with ties to even (nearbyint in the default rounding mode), and
 * re-assemble. */
uint16_t pqo_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7e00);
    if (isinf(a))
        return (uint16_t)(sign | 0x7c00);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);            /* a = m * 2^e2, m in [0.5,1): unbiased exp = e2-1 */
    int e = e2 - 1;
    if (e < -14)
        e = -14;              /* subnormal binade shares the 2^-24 quantum */
    double units = nearbyint(ldexp(a, 10 - e));   /* integer count of quanta */
    /* units in [1024, 2048] for normals (2048 = carried into next binade),
     * [0, 1024] for the subnormal range. */
    if (units >= 2048.0) {
        units = 1024.0;
        e += 1;
    }
    if (units < 1024.0) {      /* subnormal (only possible when e == -14) */
        return (uint16_t)(sign | (uint16_t)units);
    }
    if (e > 15)
        return (uint16_t)(sign | 0x7c00);
    uint16_t bits = (uint16_t)(((e + 15) << 10) | ((int)units - 1024));
    return (uint16_t)(sign | bits);
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* ------------------------------------------------------------------ */
/* Layout constants                                                    */
/* ------------------------------------------------------------------ */

int pqo_block_weights(int fmt)
{
    switch (fmt) {
    case PQO_Q8_0: return 32;
    case PQO_Q4_K: return 256;
    case PQO_Q6_K: return 256;
    case PQO_I8_ROW: return 1;
    case PQO_Q5_K: return 256;
    case PQO_Q3_K: return 256;
    case PQO_Q2_K: return 256;
    case PQO_I4_ROW: return 2;
    }
    return -1;
}

int pqo_block_bytes(int fmt)
{
    switch (fmt) {
    case PQO_Q8_0: return 34;
    case PQO_Q4_K: return 144;
    case PQO_Q6_K: return 210;
    case PQO_I8_ROW: return 1;
    case PQO_Q5_K: return 176;
    case PQO_Q3_K: return 110;
    case PQO_Q2_K: return 84;
    case PQO_I4_ROW: return 1;
    }
    return -1;
}

/* Bytes of one whole matrix.  For per-row int8 the f32 scales follow the
 * n_out*k codes at the next 16-byte boundary. */
int64_t pqo_weight_bytes(int fmt, int64_t n_out, int64_t k)
{
    if (fmt == PQO_I8_ROW) {
        int64_t q = n_out * k;
        int64_t off = (q + 15) / 16 * 16;
        return off + 4 * n_out;
    }
    int qk = pqo_block_weights(fmt), bb = pqo_block_bytes(fmt);
    if (qk <= 0 || k % qk)
        return -1;
    if (fmt == PQO_I4_ROW)
        return (n_out * (k / 2) + 15) / 16 * 16 + 4 * n_out;
    return n_out * (k / qk) * bb;
}

static int64_t i8row_scale_offset(int64_t n_out, int64_t k)
{
    return (n_out * k + 15) / 16 * 16;
}

static int64_t i4row_scale_offset(int64_t n_out, int64_t k)
{
    return (n_out * (k / 2) + 15) / 16 * 16;
}

/* Signed value of the 4-bit two's-complement code c (0..15): -8..7. */
static int i4_value(int c) { return c >= 8 ? c - 16 : c; }

/* ------------------------------------------------------------------ */
/* Block decoders (one block -> f32)                                   */
/* ------------------------------------------------------------------ */

/* Q8_0: f16 d at bytes 0-1, int8 q[32] at bytes 2-33.  w[i] = d * q[i]. */
void pqo_decode_q8_0(const uint8_t *blk, float *w)
{
    float d = pqo_half_to_float(rd16(blk));
    for (int i = 0; i < 32; ++i)
        w[i] = d * (float)(int8_t)blk[2 + i];
}

/* The 6-bit scale and min of sub-block j (0..7) of a Q4_K super-block,
 * from the 12 packed bytes s[0..11]:
 *   j < 4 : sc = low 6 bits of s[j],   m = low 6 bits of s[j+4]
 *   j >= 4: sc = low nibble of s[j+4] with the top 2 bits of s[j-4] above it,
 *           m  = high nibble of s[j+4] with the top 2 bits of s[j] above it. */
void pqo_q4_k_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 0x0f) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Q4_K (144 B): f16 d @0, f16 dmin @2, 12 scale bytes @4, qs[128] @16.
 * The 256 weights form 4 chunks of 64; in chunk c, weight 64c+l (l<32) is the
 * low nibble of qs[32c+l] and belongs to sub-block 2c, weight 64c+32+l is
 * the high nibble of the same byte and belongs to sub-block 2c+1.
 * w = (d*sc_j)*q - dmin*m_j in f32: both products are exact in f32, only the
 * subtraction rounds. */
void pqo_decode_q4_k(const uint8_t *blk, float *w)
{
    float d = pqo_half_to_float(rd16(blk));
    float dmin = pqo_half_to_float(rd16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < 256; ++i) {
        int c = i / 64, p = i % 64;
        int j, q;
        if (p < 32) {
            j = 2 * c;
            q = qs[32 * c + p] & 0x0f;
        } else {
            j = 2 * c + 1;
            q = qs[32 * c + p - 32] >> 4;
        }
        int sc, m;
        pqo_q4_k_scale_min(scales, j, &sc, &m);
        float dl = d * (float)sc;
        float ml = dmin * (float)m;
        w[i] = dl * (float)q - ml;
    }
}

/* Q6_K (210 B): ql[128] @0, qh[64] @128, int8 sc[16] @192, f16 d @208.
 * Two halves of 128 weights; half h reads ql+64h and qh+32h.  For l<32 the
 * four 6-bit codes of column l are
 *   weight 128h+l     : low nibble of ql[l]     | bits 0-1 of qh[l] << 4
 *   weight 128h+l+32  : low nibble of ql[l+32]  | bits 2-3 of qh[l] << 4
 *   weight 128h+l+64  : high nibble of ql[l]    | bits 4-5 of qh[l] << 4
 *   weight 128h+l+96  : high nibble of ql[l+32] | bits 6-7 of qh[l] << 4
 * each minus 32.  Weight n uses sc[n/16].  w = (d*sc)*(q-32), exact in f32. */
void pqo_decode_q6_k(const uint8_t *blk, float *w)
{
    const uint8_t *ql0 = blk, *qh0 = blk + 128;
    const int8_t *sc = (const int8_t *)(blk + 192);
    float d = pqo_half_to_float(rd16(blk + 208));
    for (int n = 0; n < 256; ++n) {
        int h = n / 128, r = n % 128;
        int t = r / 32, l = r % 32;
        const uint8_t *ql = ql0 + 64 * h, *qh = qh0 + 32 * h;
        int lo4, hi2;
        switch (t) {
        case 0: lo4 = ql[l] & 0x0f;      hi2 = (qh[l] >> 0) & 3; break;
        case 1: lo4 = ql[l + 32] & 0x0f; hi2 = (qh[l] >> 2) & 3; break;
        case 2: lo4 = ql[l] >> 4;        hi2 = (qh[l] >> 4) & 3; break;
        default: lo4 = ql[l + 32] >> 4;  hi2 = (qh[l] >> 6) & 3; break;
        }
        int q = (lo4 | (hi2 << 4)) - 32;
        float ds = d * (float)sc[n / 16];
        w[n] = ds * (float)q;
    }
}

/* Q5_K (176 B): f16 d @0, f16 dmin @2, 12 scale bytes @4 (packed exactly as
 * Q4_K's), qh[32] @16, qs[128] @48.  As in Q4_K, chunk c of 64 weights holds
 * sub-block 2c (low nibbles of qs[32c..32c+31]) then sub-block 2c+1 (high
 * nibbles of the same bytes); the fifth bit of weight 64c+32h+l (h = 0, 1,
 * l < 32) is bit 2c+h of qh[l].  q = nibble + 16*bit, in 0..31.
 * w = (d*sc_j)*q - dmin*m_j in f32: both products are exact, the subtraction
 * rounds. */
void pqo_decode_q5_k(const uint8_t *blk, float *w)
{
    float d = pqo_half_to_float(rd16(blk));
    float dmin = pqo_half_to_float(rd16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    for (int i = 0; i < 256; ++i) {
        int c = i / 64, p = i % 64;
        int h = p / 32, l = p % 32;
        int j = 2 * c + h;
        int lo4 = h == 0 ? (qs[32 * c + l] & 0x0f) : (qs[32 * c + l] >> 4);
        int q = lo4 + 16 * ((qh[l] >> j) & 1);
        int sc, m;
        pqo_q4_k_scale_min(scales, j, &sc, &m);
        float dl = d * (float)sc;
        float ml = dmin * (float)m;
        w[i] = dl * (float)q - ml;
    }
}

/* The signed 6-bit scale of group s (0..15, 16 weights each) of a Q3_K
 * super-block, from the 12 packed bytes t[0..11]: the low four bits are the
 * low nibble of t[s] (s < 8) or the high nibble of t[s-8] (s >= 8); the top two
 * bits are bits 2*(s/4), 2*(s/4)+1 of t[8 + s%4]; the stored value is offset
 * by 32. */
int pqo_q3_k_scale(const uint8_t *t, int s)
{
    int lo4 = s < 8 ? (t[s] & 0x0f) : (t[s - 8] >> 4);
    int hi2 = (t[8 + s % 4] >> (2 * (s / 4))) & 3;
    return (lo4 | (hi2 << 4)) - 32;
}

/* Q3_K (110 B): hmask[32] @0, qs[64] @32, 12 scale bytes @96, f16 d @108.
 * Two halves of 128 weights; in half n, weight 128n+32j+l (j = 0..3, l < 32)
 * takes bits 2j, 2j+1 of qs[32n+l] as a 2-bit code and bit 4n+j of hmask[l]
 * as its high bit: value = code - 4 when that bit is clear, code when set
 * (range -4..3).  Weight i uses scale group i/16.  w = (d*sc)*value, exact in
 * f32. */
void pqo_decode_q3_k(const uint8_t *blk, float *w)
{
    const uint8_t *hmask = blk, *qs = blk + 32, *scales = blk + 96;
    float d = pqo_half_to_float(rd16(blk + 108));
    for (int i = 0; i < 256; ++i) {
        int n = i / 128, r = i % 128;
        int j = r / 32, l = r % 32;
        int code = (qs[32 * n + l] >> (2 * j)) & 3;
        int high = (hmask[l] >> (4 * n + j)) & 1;
        int value = code - (high ? 0 : 4);
        float ds = d * (float)pqo_q3_k_scale(scales, i / 16);
        w[i] = ds * (float)value;
    }
}

/* Q2_K (84 B): scales[16] @0 (low nibble: scale, high nibble: min, one byte
 * per group of 16 weights), qs[64] @16, f16 d @80, f16 dmin @82.  Weight
 * 128n+32j+l takes bits 2j, 2j+1 of qs[32n+l] (code 0..3) and group i/16.
 * w = (d*sc)*code - dmin*m in f32: both products exact, the subtraction
 * rounds. */
void pqo_decode_q2_k(const uint8_t *blk, float *w)
{
    const uint8_t *scales = blk, *qs = blk + 16;
    float d = pqo_half_to_float(rd16(blk + 80));
    float dmin = pqo_half_to_float(rd16(blk + 82));
    for (int i = 0; i < 256; ++i) {
        int n = i / 128, r = i % 128;
        int j = r / 32, l = r % 32;
        int code = (qs[32 * n + l] >> (2 * j)) & 3;
        int g = scales[i / 16];
        float dl = d * (float)(g & 0x0f);
        float ml = dmin * (float)(g >> 4);
        w[i] = dl * (float)code - ml;
    }
}

/* Decode row r of a whole matrix into w[0..k). */
static void decode_row(int fmt, const uint8_t *W, int64_t n_out, int64_t k, int64_t r, float *w)
{
    if (fmt == PQO_I8_ROW) {
        const int8_t *q = (const int8_t *)W + r * k;
        float s;
        memcpy(&s, W + i8row_scale_offset(n_out, k) + 4 * r, 4);
        for (int64_t i = 0; i < k; ++i)
            w[i] = s * (float)q[i];
        return;
    }
    if (fmt == PQO_I4_ROW) {
        const uint8_t *q = W + r * (k / 2);
        float s;
        memcpy(&s, W + i4row_scale_offset(n_out, k) + 4 * r, 4);
        for (int64_t i = 0; i < k; ++i) {
            int c = (i % 2 == 0) ? (q[i / 2] & 0x0f) : (q[i / 2] >> 4);
            w[i] = s * (float)i4_value(c);
        }
        return;
    }
    int qk = pqo_block_weights(fmt), bb = pqo_block_bytes(fmt);
    int64_t nb = k / qk;
    const uint8_t *row = W + r * nb * bb;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = row + b * bb;
        float *o = w + b * qk;
        switch (fmt) {
        case PQO_Q8_0: pqo_decode_q8_0(blk, o); break;
        case PQO_Q4_K: pqo_decode_q4_k(blk, o); break;
        case PQO_Q6_K: pqo_decode_q6_k(blk, o); break;
        case PQO_Q5_K: pqo_decode_q5_k(blk, o); break;
        case PQO_Q3_K: pqo_decode_q3_k(blk, o); break;
        default: pqo_decode_q2_k(blk, o); break;
        }
    }
}

static int nthreads_or_default(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of threads an OpenMP region with this request actually gets. */
int pqo_threads(int nthreads)
{
    int used = 1;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads_or_default(nthreads))
    {
#pragma omp single
        used = omp_get_num_threads();
    }
#else
    (void)nthreads;
#endif
    return used;
}

/* out[r][i] (f32, row-major n_out x k) = decoded weight. */
int pqo_dequant(int fmt, const uint8_t *W, int64_t n_out, int64_t k, float *out, int nthreads)
{
    if (pqo_weight_bytes(fmt, n_out, k) < 0)
        return -1;
    int nt = nthreads_or_default(nthreads);
    (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t r = 0; r < n_out; ++r)
        decode_row(fmt, W, n_out, k, r, out + r * k);
    return 0;
}

/* y[b][j] for the listed rows (rows[j], j < nrows): decode the row to f32,
 * then sum (double)w*(double)x over i in index order.  y is [batch][nrows]. */
int pqo_gemv_rows(int fmt, const uint8_t *W, int64_t n_out, int64_t k,
                  const float *x, int64_t batch, const int64_t *rows, int64_t nrows,
                  double *y, int nthreads)
{
    if (pqo_weight_bytes(fmt, n_out, k) < 0)
        return -1;
    int nt = nthreads_or_default(nthreads);
    int failed = 0;
#pragma omp parallel num_threads(nt)
    {
        float *w = (float *)malloc(sizeof(float) * (size_t)k);
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t j = 0; j < nrows; ++j) {
            if (!w)
                continue;
            decode_row(fmt, W, n_out, k, rows[j], w);
            for (int64_t b = 0; b < batch; ++b) {
                const float *xb = x + b * k;
                double acc = 0.0;
                for (int64_t i = 0; i < k; ++i)
                    acc += (double)w[i] * (double)xb[i];
                y[b * nrows + j] = acc;
            }
        }
        free(w);
    }
    return failed ? -2 : 0;
}

/* y[b][r] for every row: y is [batch][n_out]. */
int pqo_gemv(int fmt, const uint8_t *W, int64_t n_out, int64_t k,
             const float *x, int64_t batch, double *y, int nthreads)
{
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_out > 0 ? n_out : 1));
    if (!rows)
        return -2;
    for (int64_t r = 0; r < n_out; ++r)
        rows[r] = r;
    int rc = pqo_gemv_rows(fmt, W, n_out, k, x, batch, rows, n_out, y, nthreads);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Epilogues on the decode-layer mat-vecs                              */
/* ------------------------------------------------------------------ */

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z), in f64 (the PESTI README,
 * "Conformance": the MLP's SwiGLU multiplies the sigmoid-based silu of the
 * gate projection by the up projection).  Written as z / (1 + exp(-z)) for z >= 0 and as
 * z * e^z / (1 + e^z) for z < 0, so that neither form overflows. */
double pqo_silu(double z)
{
    if (z >= 0.0)
        return z / (1.0 + exp(-z));
    double e = exp(z);
    return z * e / (1.0 + e);
}

/* SwiGLU on a fused gate+up matrix: W has 2*n_ff rows, rows [0, n_ff) the
 * gate projection and rows [n_ff, 2*n_ff) the up projection (the order the
 * name gate+up gives).  h[b][j] = silu(g) * u with g, u the f64 mat-vec rows
 * j and n_ff + j.  h is [batch][n_ff]. */
int pqo_gemv_swiglu(int fmt, const uint8_t *W, int64_t n_ff, int64_t k,
                    const float *x, int64_t batch, double *h, int nthreads)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)(batch * 2 * n_ff > 0 ? batch * 2 * n_ff : 1));
    if (!y)
        return -2;
    int rc = pqo_gemv(fmt, W, 2 * n_ff, k, x, batch, y, nthreads);
    if (rc == 0)
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t j = 0; j < n_ff; ++j) {
                double g = y[b * 2 * n_ff + j], u = y[b * 2 * n_ff + n_ff + j];
                h[b * n_ff + j] = pqo_silu(g) * u;
            }
    free(y);
    return rc;
}

/* y[b][r] = (W x_b)[r] + bias[r] in f64 (the PESTI README, "Conformance":
 * the QKV projections carry a bias). */
int pqo_gemv_bias(int fmt, const uint8_t *W, int64_t n_out, int64_t k,
                  const float *x, int64_t batch, const float *bias, double *y, int nthreads)
{
    int rc = pqo_gemv(fmt, W, n_out, k, x, batch, y, nthreads);
    if (rc == 0)
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t r = 0; r < n_out; ++r)
                y[b * n_out + r] += (double)bias[r];
    return rc;
}

/* ------------------------------------------------------------------ */
/* Quantizers (make test inputs)                                       */
/* ------------------------------------------------------------------ */

static int clampi(double v, int lo, int hi)
{
    if (v < lo) return lo;
    if (v > hi) return hi;
    return (int)v;
}

/* Q8_0: d = f16(max|v| / 127), q = clamp(round(v/d), -127, 127); q = 0 if d = 0. */
static void quantize_q8_0_block(const float *v, uint8_t *blk)
{
    double amax = 0.0;
    for (int i = 0; i < 32; ++i)
        if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
    uint16_t dh = pqo_double_to_half(amax / 127.0);
    double d = (double)pqo_half_to_float(dh);
    wr16(blk, dh);
    for (int i = 0; i < 32; ++i) {
        int q = d > 0.0 ? clampi(round((double)v[i] / d), -127, 127) : 0;
        blk[2 + i] = (uint8_t)(int8_t)q;
    }
}

/* Q4_K, per super-block of 256 values, sub-blocks of 32:
 *   mn_j = min(0, min v), s_j = (max v - mn_j)/15, mneg_j = -mn_j;
 *   d = f16(max_j s_j / 63), dmin = f16(max_j mneg_j / 63);
 *   sc_j = clamp(round(s_j/d), 0, 63), m_j = clamp(round(mneg_j/dmin), 0, 63)
 *   (0 when the divisor is 0);
 *   q = clamp(round((v + dmin*m_j)/(d*sc_j)), 0, 15) (0 when d*sc_j = 0).
 * Then packed: 6-bit (sc, m) pairs into 12 bytes, nibbles into qs. */
static void quantize_q4_k_block(const float *v, uint8_t *blk)
{
    double s[8], mneg[8];
    double smax = 0.0, mmax = 0.0;
    for (int j = 0; j < 8; ++j) {
        double mn = 0.0, mx = -INFINITY;
        for (int i = 0; i < 32; ++i) {
            double t = (double)v[32 * j + i];
            if (t < mn) mn = t;
            if (t > mx) mx = t;
        }
        s[j] = (mx - mn) / 15.0;
        mneg[j] = -mn;
        if (s[j] > smax) smax = s[j];
        if (mneg[j] > mmax) mmax = mneg[j];
    }
    uint16_t dh = pqo_double_to_half(smax / 63.0);
    uint16_t mh = pqo_double_to_half(mmax / 63.0);
    double d = (double)pqo_half_to_float(dh);
    double dmin = (double)pqo_half_to_float(mh);
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0 ? clampi(round(s[j] / d), 0, 63) : 0;
        m[j] = dmin > 0.0 ? clampi(round(mneg[j] / dmin), 0, 63) : 0;
    }
    memset(blk, 0, 144);
    wr16(blk, dh);
    wr16(blk + 2, mh);
    uint8_t *sb = blk + 4;
    for (int j = 0; j < 4; ++j) {
        sb[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        sb[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        sb[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t *qs = blk + 16;
    for (int i = 0; i < 256; ++i) {
        int j = i / 32;
        double step = d * (double)sc[j];
        double off = dmin * (double)m[j];
        int q = step > 0.0 ? clampi(round(((double)v[i] + off) / step), 0, 15) : 0;
        int c = i / 64, p = i % 64;
        if (p < 32)
            qs[32 * c + p] |= (uint8_t)q;
        else
            qs[32 * c + p - 32] |= (uint8_t)(q << 4);
    }
}

/* Q6_K, per super-block of 256 values, sub-blocks of 16:
 *   s_t = max|v|/31, d = f16(max_t s_t / 127), sc_t = clamp(round(s_t/d), -128, 127),
 *   q = clamp(round(v/(d*sc_t)), -32, 31) + 32 (32 when d*sc_t = 0).
 * Then the 6-bit codes are split into ql (low 4 bits) and qh (high 2 bits)
 * by the layout rule of the decoder. */
static void quantize_q6_k_block(const float *v, uint8_t *blk)
{
    double s[16], smax = 0.0;
    for (int t = 0; t < 16; ++t) {
        double amax = 0.0;
        for (int i = 0; i < 16; ++i)
            if (fabs((double)v[16 * t + i]) > amax) amax = fabs((double)v[16 * t + i]);
        s[t] = amax / 31.0;
        if (s[t] > smax) smax = s[t];
    }
    uint16_t dh = pqo_double_to_half(smax / 127.0);
    double d = (double)pqo_half_to_float(dh);
    int sc[16];
    for (int t = 0; t < 16; ++t)
        sc[t] = d > 0.0 ? clampi(round(s[t] / d), -128, 127) : 0;
    memset(blk, 0, 210);
    uint8_t *ql0 = blk, *qh0 = blk + 128;
    for (int t = 0; t < 16; ++t)
        blk[192 + t] = (uint8_t)(int8_t)sc[t];
    wr16(blk + 208, dh);
    for (int n = 0; n < 256; ++n) {
        double step = d * (double)sc[n / 16];
        int q = step != 0.0 ? clampi(round((double)v[n] / step), -32, 31) + 32 : 32;
        int h = n / 128, r = n % 128, t = r / 32, l = r % 32;
        uint8_t *ql = ql0 + 64 * h, *qh = qh0 + 32 * h;
        int lo4 = q & 15, hi2 = q >> 4;
        switch (t) {
        case 0: ql[l] |= (uint8_t)lo4;             qh[l] |= (uint8_t)(hi2 << 0); break;
        case 1: ql[l + 32] |= (uint8_t)lo4;        qh[l] |= (uint8_t)(hi2 << 2); break;
        case 2: ql[l] |= (uint8_t)(lo4 << 4);      qh[l] |= (uint8_t)(hi2 << 4); break;
        default: ql[l + 32] |= (uint8_t)(lo4 << 4); qh[l] |= (uint8_t)(hi2 << 6); break;
        }
    }
}

/* Quantize an f32 matrix v[n_out][k] (row-major) into out
 * (pqo_weight_bytes(fmt, n_out, k) bytes). */
int pqo_quantize(int fmt, const float *v, int64_t n_out, int64_t k, uint8_t *out, int nthreads)
{
    int64_t total = pqo_weight_bytes(fmt, n_out, k);
    if (total < 0)
        return -1;
    /* no quantizer for Q5_K / Q3_K / Q2_K: their test inputs are random
     * records (every field bit pattern), which need none */
    if (fmt == PQO_Q5_K || fmt == PQO_Q3_K || fmt == PQO_Q2_K)
        return -1;
    int nt = nthreads_or_default(nthreads);
    (void)nt;
    if (fmt == PQO_I8_ROW) {
        /* per-row symmetric: s = max|v_r|/127 (f32), q = clamp(round(v/s), -127, 127) */
        int64_t soff = i8row_scale_offset(n_out, k);
        memset(out, 0, (size_t)total);
#pragma omp parallel for schedule(static) num_threads(nt)
        for (int64_t r = 0; r < n_out; ++r) {
            const float *vr = v + r * k;
            double amax = 0.0;
            for (int64_t i = 0; i < k; ++i)
                if (fabs((double)vr[i]) > amax) amax = fabs((double)vr[i]);
            float s = (float)(amax / 127.0);
            for (int64_t i = 0; i < k; ++i) {
                int q = s > 0.0f ? clampi(round((double)vr[i] / (double)s), -127, 127) : 0;
                out[r * k + i] = (uint8_t)(int8_t)q;
            }
            memcpy(out + soff + 4 * r, &s, 4);
        }
        return 0;
    }
    if (fmt == PQO_I4_ROW) {
        /* per-row symmetric: s = max|v_r|/7 (f32), q = clamp(round(v/s), -7, 7) */
        int64_t soff = i4row_scale_offset(n_out, k);
        memset(out, 0, (size_t)total);
#pragma omp parallel for schedule(static) num_threads(nt)
        for (int64_t r = 0; r < n_out; ++r) {
            const float *vr = v + r * k;
            double amax = 0.0;
            for (int64_t i = 0; i < k; ++i)
                if (fabs((double)vr[i]) > amax) amax = fabs((double)vr[i]);
            float s = (float)(amax / 7.0);
            for (int64_t i = 0; i < k; ++i) {
                int q = s > 0.0f ? clampi(round((double)vr[i] / (double)s), -7, 7) : 0;
                out[r * (k / 2) + i / 2] |= (uint8_t)((q & 0x0f) << (4 * (int)(i % 2)));
            }
            memcpy(out + soff + 4 * r, &s, 4);
        }
        return 0;
    }
    int qk = pqo_block_weights(fmt), bb = pqo_block_bytes(fmt);
    int64_t nb = k / qk;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t r = 0; r < n_out; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *vb = v + r * k + b * qk;
            uint8_t *blk = out + (r * nb + b) * bb;
            if (fmt == PQO_Q8_0)
                quantize_q8_0_block(vb, blk);
            else if (fmt == PQO_Q4_K)
                quantize_q4_k_block(vb, blk);
            else
                quantize_q6_k_block(vb, blk);
        }
    }
    return 0;
}

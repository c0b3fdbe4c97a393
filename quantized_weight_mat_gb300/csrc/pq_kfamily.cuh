// Decoders of the Q5_K, Q3_K and Q2_K super-blocks (256 weights each), the
// rest of the K family that the PESTI README ("What This Is") decodes.  The
// pages print no layout; these are the public GGUF ones, read as a byte
// specification:
//   Q5_K 176 B: f16 d @0, f16 dmin @2, 12 bytes of packed 6-bit (scale, min)
//        pairs @4 (packed as in Q4_K), qh[32] @16, qs[128] @48.  Chunk c of
//        64 weights: sub-block 2c from the low nibbles of qs[32c..32c+31],
//        sub-block 2c+1 from the high nibbles; the fifth bit of weight
//        64c+32h+l is bit 2c+h of qh[l].  w = (d*sc)*q - dmin*m.
//   Q3_K 110 B: hmask[32] @0, qs[64] @32, 12 bytes of 16 packed signed 6-bit
//        scales @96, f16 d @108.  Weight 128n+32j+l: bits 2j..2j+1 of
//        qs[32n+l], minus 4 unless bit 4n+j of hmask[l] is set; scale group
//        i/16.  w = (d*sc)*value, exact.
//   Q2_K 84 B: scales[16] @0 (low nibble scale, high nibble min, group i/16),
//        qs[64] @16, f16 d @80, f16 dmin @82.  Weight 128n+32j+l: bits
//        2j..2j+1 of qs[32n+l].  w = (d*sc)*code - dmin*m.
//
// Each function decodes the eight consecutive weights 8*lane .. 8*lane+7 of
// one super-block (lane 0..31) through a loader L with u8/u16/u32/f16 reads
// at byte offsets of the block.  Every product is exact in f32 and the only
// rounding (the subtraction of the min term) is explicit, so the result is
// bit-identical to the plain decode.  The block alignments differ (176 B
// blocks keep 16-byte alignment, 84 B blocks 4-byte, 110 B blocks only
// 2-byte), and the reads follow them: u32 only for Q5_K and Q2_K, u16 at
// even offsets for Q3_K.
#pragma once

#include <cstdint>

namespace pqk {

__host__ __device__ inline float kf_mul(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}
__host__ __device__ inline float kf_sub(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}

// byte e (0..7) of the little-endian pair of words (a, b)
__host__ __device__ inline uint32_t byte_of2(uint32_t a, uint32_t b, int e) {
    return ((e < 4 ? a : b) >> (8 * (e & 3))) & 0xffu;
}

// 6-bit (scale, min) of sub-block j from the 12 packed bytes at `base`
template <class L>
__host__ __device__ inline void kf_scale_min_k4(const L &ld, int base, int j, int &sc, int &m) {
    if (j < 4) {
        sc = (int)(ld.u8(base + j) & 63u);
        m = (int)(ld.u8(base + j + 4) & 63u);
    } else {
        const uint32_t b = ld.u8(base + j + 4);
        sc = (int)((b & 15u) | ((ld.u8(base + j - 4) >> 6) << 4));
        m = (int)((b >> 4) | ((ld.u8(base + j) >> 6) << 4));
    }
}

template <class L>
__host__ __device__ inline void q5k_lane(const L &ld, int lane, float (&w)[8]) {
    const int c = lane >> 3, h = (lane >> 2) & 1, l0 = 8 * (lane & 3);
    const int j = 2 * c + h;
    int sc, m;
    kf_scale_min_k4(ld, 4, j, sc, m);
    const float dl = kf_mul(ld.f16(0), (float)sc), ml = kf_mul(ld.f16(2), (float)m);
    const uint32_t qa = ld.u32(48 + 32 * c + l0), qb = ld.u32(48 + 32 * c + l0 + 4);
    const uint32_t ha = ld.u32(16 + l0), hb = ld.u32(16 + l0 + 4);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t nib = (byte_of2(qa, qb, e) >> (4 * h)) & 15u;
        const uint32_t q = nib + 16u * ((byte_of2(ha, hb, e) >> j) & 1u);
        w[e] = kf_sub(kf_mul(dl, (float)q), ml);
    }
}

// signed scale of group s (0..15) from the 12 packed bytes at `base`
template <class L>
__host__ __device__ inline int kf_scale_q3k(const L &ld, int base, int s) {
    const uint32_t lo4 = s < 8 ? (ld.u8(base + s) & 15u) : (ld.u8(base + s - 8) >> 4);
    const uint32_t hi2 = (ld.u8(base + 8 + (s & 3)) >> (2 * (s >> 2))) & 3u;
    return (int)(lo4 | (hi2 << 4)) - 32;
}

template <class L>
__host__ __device__ inline void q3k_lane(const L &ld, int lane, float (&w)[8]) {
    const int n = lane >> 4, j = (lane & 15) >> 2, l0 = 8 * (lane & 3);
    const float ds = kf_mul(ld.f16(108), (float)kf_scale_q3k(ld, 96, lane >> 1));
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const uint32_t q2 = ld.u16(32 + 32 * n + l0 + e), h2 = ld.u16(l0 + e);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int code = (int)((q2 >> (8 * t + 2 * j)) & 3u);
            const int high = (int)((h2 >> (8 * t + 4 * n + j)) & 1u);
            w[e + t] = kf_mul(ds, (float)(code - (high ? 0 : 4)));
        }
    }
}

template <class L>
__host__ __device__ inline void q2k_lane(const L &ld, int lane, float (&w)[8]) {
    const int n = lane >> 4, j = (lane & 15) >> 2, l0 = 8 * (lane & 3);
    const uint32_t g = ld.u8(lane >> 1);
    const float dl = kf_mul(ld.f16(80), (float)(g & 15u)), ml = kf_mul(ld.f16(82), (float)(g >> 4));
    const uint32_t qa = ld.u32(16 + 32 * n + l0), qb = ld.u32(16 + 32 * n + l0 + 4);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t code = (byte_of2(qa, qb, e) >> (2 * j)) & 3u;
        w[e] = kf_sub(kf_mul(dl, (float)code), ml);
    }
}

}  // namespace pqk

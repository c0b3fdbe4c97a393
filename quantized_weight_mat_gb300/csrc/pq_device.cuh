// Device-side helpers shared by the kernels of this library.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "pq.h"
#include "pq_kfamily.cuh"

namespace pqk {

// IEEE binary16 bits -> f32 (exact hardware conversion).
__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}

__device__ __forceinline__ uint32_t ldg_u32(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ uint4 ldg_u128(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ float4 ldg_f4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// Power-of-two scale of x for the fp16 operands of the tensor-core kernels.
// With E the binary exponent of m = max|x| over a block of x (m in
// [2^E, 2^(E+1))), x' = 2^e * x with e = 9 - E, capped at 126 so that 2^e and
// 2^-e are normal f32 numbers (a cap that only applies when m < 2^-117);
// e = 0 when m is 0, inf or NaN (non-finite values then reach y as they would
// unscaled).  Scaling by a power of two is exact, so x' = x_hi + x_lo (two
// fp16 halves) holds x to a relative 2^-21 plus an absolute 2^-25 in scaled
// units, i.e. about 2^-34 of the block's maximum; every x' and every sum of
// 32 of them fits fp16's range.  Argument: the bits of m (sign cleared).
__device__ __forceinline__ int tc_scale_exponent(uint32_t max_abs_bits) {
    const int eb = (int)(max_abs_bits >> 23);           // biased exponent; 0 for zero and subnormals
    if (max_abs_bits == 0u || eb == 255) return 0;
    const int e = 9 - ((eb > 0 ? eb : 1) - 127);
    return e < 126 ? e : 126;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The 6-bit (scale, min) pair of sub-block j (0..7) of a Q4_K super-block.
// s0, s1, s2 are the 12 packed bytes as three little-endian words:
//   j < 4 : sc = bits 0-5 of byte j,          m = bits 0-5 of byte j+4
//   j >= 4: sc = low nibble of byte j+4 | (bits 6-7 of byte j-4) << 4
//           m  = high nibble of byte j+4 | (bits 6-7 of byte j) << 4
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j,
                                              int &sc, int &m) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        m = (s1 >> (8 * j)) & 63;
    } else {
        const int b = 8 * (j - 4);
        sc = ((s2 >> b) & 15) | (((s0 >> (b + 6)) & 3) << 4);
        m = ((s2 >> (b + 4)) & 15) | (((s1 >> (b + 6)) & 3) << 4);
    }
}

// Value of a 4-bit two's-complement code (0..15 -> -8..7), as f32.
__device__ __forceinline__ float i4_value(uint32_t nib) { return (float)((int)(nib ^ 8u) - 8); }

// Read-only loads at byte offsets of one block, for the K-family decoders
// (pq_kfamily.cuh); the decoders keep every access aligned to its width.
struct BlockLoad {
    const uint8_t *p;
    __device__ __forceinline__ uint32_t u8(int o) const { return __ldg(p + o); }
    __device__ __forceinline__ uint32_t u16(int o) const { return ldg_u16(p + o); }
    __device__ __forceinline__ uint32_t u32(int o) const { return ldg_u32(p + o); }
    __device__ __forceinline__ float f16(int o) const { return h2f(ldg_u16(p + o)); }
};

// Weights 8*lane .. 8*lane+7 of one Q5_K / Q3_K / Q2_K super-block.
template <int FMT>
__device__ __forceinline__ void kfamily_lane(const uint8_t *blk, int lane, float (&w)[8]) {
    static_assert(FMT == PQ_Q5_K || FMT == PQ_Q3_K || FMT == PQ_Q2_K, "K-family format");
    const BlockLoad ld{blk};
    if constexpr (FMT == PQ_Q5_K)
        q5k_lane(ld, lane, w);
    else if constexpr (FMT == PQ_Q3_K)
        q3k_lane(ld, lane, w);
    else
        q2k_lane(ld, lane, w);
}

}  // namespace pqk

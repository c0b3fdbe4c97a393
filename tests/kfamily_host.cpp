// Host build of the library's Q5_K / Q3_K / Q2_K lane decoders
// (pq_kfamily.cuh, the functions the CUDA kernels run), for a CPU test that
// compares them bit for bit with the oracle.  Compiled by the test with g++
// and -ffp-contract=off, so every product and difference rounds once, as
// the device's _rn intrinsics do.
#define __host__
#define __device__
#include <cmath>
#include <cstdint>
#include <cstring>

#include "pq_kfamily.cuh"

namespace {

// IEEE binary16 -> binary32 from the format's definition (exact).
float half_bits_to_float(uint32_t h) {
    const uint32_t s = h >> 15, e = (h >> 10) & 31u, f = h & 1023u;
    float v;
    if (e == 0)
        v = std::ldexp((float)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = std::ldexp((float)(1024u + f), (int)e - 25);
    return s ? -v : v;
}

struct HostLoad {
    const uint8_t *p;
    uint32_t u8(int o) const { return p[o]; }
    uint32_t u16(int o) const { return p[o] | (p[o + 1] << 8); }
    uint32_t u32(int o) const {
        return p[o] | (p[o + 1] << 8) | (p[o + 2] << 16) | ((uint32_t)p[o + 3] << 24);
    }
    float f16(int o) const { return half_bits_to_float(u16(o)); }
};

}  // namespace

// Decode one super-block of format fmt (4 = Q5_K, 5 = Q3_K, 6 = Q2_K) into
// out[256], lane by lane as the kernels do.  Returns -1 for another format.
extern "C" int kf_host_decode(int fmt, const uint8_t *blk, float *out) {
    const HostLoad ld{blk};
    for (int lane = 0; lane < 32; ++lane) {
        float w[8];
        if (fmt == 4)
            pqk::q5k_lane(ld, lane, w);
        else if (fmt == 5)
            pqk::q3k_lane(ld, lane, w);
        else if (fmt == 6)
            pqk::q2k_lane(ld, lane, w);
        else
            return -1;
        std::memcpy(out + 8 * lane, w, sizeof w);
    }
    return 0;
}

"""The arithmetic facts the kernels' precision rests on, checked on the CPU.

1. Tensor-core decode: a 4-bit code q and a 6-bit scale sc become the fp16
   value sc*q through one fused multiply-add on a biased operand, (1024+q)*sc
   - 1024*sc for low nibbles and (1024+16q)*(sc/16) - 64*sc for high nibbles.
   Every operand is an exact fp16 value and the exact result sc*q <= 945 is
   an fp16 integer, so the single rounding of the fused operation is exact.
   The register-operand kernel instead converts the code bytes as e4m3 values
   (q * 2^-9 exactly for 0 <= q < 16) and multiplies by the fp16 integer
   sc * 2^9: again one rounding of an exactly representable product.
2. Tensor-core x operand: x' = x_hi + x_lo with x_hi = fp16(x') and x_lo =
   fp16(x' - x_hi) leaves a residual of at most 2^-21 |x'| + 2^-25 (x_lo turns
   subnormal below 2^-14, where fp16 has a fixed step of 2^-24); every
   product (sc*q) * x_hi and (sc*q) * x_lo is exact in the f32 accumulator.
   The pair alone overflows at |x'| >= 65520, so x' = 2^e * x is first scaled
   per super-block and column by a power of two chosen from the column's
   maximum: every x' and every sum of 32 of them then stays inside fp16's
   range for any finite x, and 2^e and 2^-e are normal f32 numbers.
3. Batch-1 x limbs: per 256 values, x ~= u*(254*xh + xl) with int8 limbs
   made by the 1.5*2^23 round-to-nearest shift.  Both limbs stay in
   [-127, 127] without any clamp (the kernel relies on it), and the error is
   at most about max|x|/64516.
The emulation rounds each step exactly as the kernel does: fused operations
are computed exactly with rationals and rounded once to f32.
"""
import zlib
from fractions import Fraction

import numpy as np
import pytest


def f16_exact(v) -> bool:
    return Fraction(float(np.float16(float(v)))) == Fraction(v)


def f32(v) -> np.float32:
    """Round an exact value (Fraction or float) to f32, nearest-even."""
    if isinstance(v, Fraction):
        # f64 first is exact enough only for short rationals; go through
        # numpy's correctly rounded conversion of the nearest f64 when exact
        d = float(v)
        if Fraction(d) == v:
            return np.float32(d)
        # not representable in f64: pick the nearer f32 neighbour exactly
        lo = np.float32(d)
        cands = [lo, np.nextafter(lo, np.float32(np.inf)), np.nextafter(lo, np.float32(-np.inf))]
        best = min(cands, key=lambda c: (abs(Fraction(float(c)) - v), int(np.float32(c).view(np.uint32)) & 1))
        return np.float32(best)
    return np.float32(v)


def fma32(a, b, c) -> np.float32:
    """fmaf: a*b + c computed exactly, rounded once to f32."""
    return f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


# ------------------------------------------------------------------ 1


@pytest.mark.parametrize("sc", range(64))
def test_fp16_bias_trick_is_exact(sc):
    for q in range(16):
        # low nibble: (1024+q)*sc - 1024*sc
        a, b, c = 1024 + q, sc, -1024 * sc
        assert f16_exact(a) and f16_exact(b) and f16_exact(c)
        exact = Fraction(a) * b + c
        assert exact == sc * q and f16_exact(exact)
        # high nibble: the byte's high nibble is kept in place, (1024+16q)*(sc/16) - 64*sc
        a, b, c = 1024 + 16 * q, Fraction(sc, 16), -64 * sc
        assert f16_exact(a) and f16_exact(b) and f16_exact(c)
        exact = Fraction(a) * b + c
        assert exact == sc * q and f16_exact(exact)


def e4m3_value(b: int) -> Fraction:
    """An OCP e4m3 byte by its definition: sign, 4 exponent bits (bias 7), 3
    mantissa bits, subnormals at exponent 0 (S.1111.111 is NaN)."""
    sign = -1 if b & 0x80 else 1
    e, m = (b >> 3) & 0xF, b & 7
    assert not (e == 15 and m == 7), "NaN"
    if e == 0:
        return sign * Fraction(m, 8) * Fraction(1, 2 ** 6)
    return sign * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


@pytest.mark.parametrize("sc", range(64))
def test_e4m3_nibble_decode_times_scale_is_exact(sc):
    # the register-operand kernel: code bytes 0-15 through the e4m3 -> fp16
    # conversion give q * 2^-9, multiplied by the fp16 sc * 2^9 in one rounding
    s512 = sc * 512
    assert f16_exact(s512)
    for q in range(16):
        v = e4m3_value(q)
        assert v == Fraction(q, 512) and f16_exact(v)
        assert v * s512 == sc * q and f16_exact(sc * q)
        # the same product in numpy's fp16 arithmetic
        assert float(np.float16(float(v)) * np.float16(s512)) == sc * q


def test_byte_under_2_pow_23_gives_the_byte():
    # the 4-column register-operand path reads a 6-bit scale byte b as the
    # f32 with bits 0x4B000000 | b (= 2^23 + b) minus 2^23
    for b in range(256):
        f = np.array([0x4B000000 | b], dtype=np.uint32).view(np.float32)[0]
        assert float(np.float32(f) - np.float32(8388608.0)) == b


# ------------------------------------------------------------------ 2


def test_x_hi_lo_split_residual_and_exact_products():
    g = np.random.default_rng(60)
    x = np.concatenate([g.normal(0, 1, 4000), g.normal(0, 1e-3, 1000), g.normal(0, 30, 1000)]).astype(np.float32)
    x_hi = x.astype(np.float16)
    x_lo = (x - x_hi.astype(np.float32)).astype(np.float16)
    for xi, h, l in zip(x[:2000], x_hi[:2000], x_lo[:2000]):
        res = abs(Fraction(float(xi)) - Fraction(float(h)) - Fraction(float(l)))
        assert res <= Fraction(abs(float(xi))) / 2 ** 21 + Fraction(1, 2 ** 25)
        for scq in (1, 7, 945):
            # fp16 * fp16 with |sc*q| <= 945: at most 10 + 11 significant bits
            for part in (h, l):
                p = Fraction(scq) * Fraction(float(part))
                assert Fraction(float(np.float32(float(p)))) == p


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_x_hi_lo_range_limits():
    # the largest value the bare pair holds, and the first one it cannot: the
    # reason x is scaled before the split
    assert np.isfinite(np.float16(np.float32(65519.0)))
    assert np.isinf(np.float16(np.float32(65520.0)))
    # below the smallest fp16 subnormal (2^-24) half-way point, x is lost
    tiny = np.float32(2.0 ** -26)
    hi = np.float16(tiny)
    assert float(hi) == 0.0 and float(np.float16(tiny - np.float32(hi))) == 0.0


def tc_scale_exponent(max_abs_bits: int) -> int:
    """The tensor-core x prep's choice of e from the bits of max|x| (sign
    cleared): e = 9 - E for max|x| in [2^E, 2^(E+1)), at most 126; 0 for a
    zero, infinite or NaN maximum."""
    eb = max_abs_bits >> 23
    if max_abs_bits == 0 or eb == 255:
        return 0
    return min(9 - (max(eb, 1) - 127), 126)


def pow2_f32(e: int) -> np.float32:
    """2^e built from its bit pattern, as the kernel does (e + 127 in 1..254)."""
    assert 1 <= e + 127 <= 254
    return np.array([(e + 127) << 23], dtype=np.uint32).view(np.float32)[0]


def tc_columns(case: str, g: np.random.Generator) -> np.ndarray:
    if case == "normal":
        return g.normal(0, 1, 256)
    if case == "huge":
        return g.normal(0, 1, 256) * 1e30
    if case == "large":
        return g.uniform(-1e6, 1e6, 256)
    if case == "tiny":
        return g.normal(0, 1e-30, 256)
    if case == "denormal":
        return g.normal(0, 1e-39, 256)
    if case == "wide":
        return g.normal(0, 1, 256) * 10.0 ** g.uniform(-30, 30, 256)
    if case == "spike":
        v = g.normal(0, 1e-3, 256)
        v[g.integers(0, 256)] = 3.0e38
        return v
    if case == "max":
        return np.full(256, 3.4e38) * g.choice([-1, 1], 256)
    if case == "zero":
        return np.zeros(256)
    raise ValueError(case)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("case", ["normal", "huge", "large", "tiny", "denormal", "wide", "spike", "max", "zero"])
def test_tc_x_scale_keeps_the_pair_and_sums_in_range(case):
    g = np.random.default_rng(zlib.crc32(case.encode()))
    for _ in range(8):
        v = tc_columns(case, g).astype(np.float32)
        m = int((v.view(np.uint32) & np.uint32(0x7FFFFFFF)).max())
        e = tc_scale_exponent(m)
        mult, undo = pow2_f32(e), pow2_f32(-e)
        assert float(mult) * float(undo) == 1.0                       # both normal, exact inverses
        xs = (v * mult).astype(np.float32)
        amax = float(np.max(np.abs(xs)))
        assert amax < 2.0 ** 10
        if m and 1 <= (m >> 23) and 9 - ((m >> 23) - 127) <= 126:
            assert amax >= 2.0 ** 9                                   # no cap: the max lands in [2^9, 2^10)
        # scaling by 2^e is exact wherever the result stays a normal f32
        normal = np.abs(xs) >= np.float32(2.0 ** -126)
        assert np.array_equal((xs[normal].astype(np.float64) / float(mult)), v[normal].astype(np.float64))
        hi = xs.astype(np.float16)
        lo = (xs - hi.astype(np.float32)).astype(np.float16)
        assert np.all(np.isfinite(hi)) and np.all(np.isfinite(lo))
        for x, h, l in zip(xs[:64], hi[:64], lo[:64]):
            res = abs(Fraction(float(x)) - Fraction(float(h)) - Fraction(float(l)))
            assert res <= Fraction(abs(float(x))) / 2 ** 21 + Fraction(1, 2 ** 25)
        # the eight 32-value sub-block sums (fixed order, f32) and their pairs
        for j in range(8):
            s = np.float32(0.0)
            for val in xs[32 * j:32 * j + 32]:
                s = np.float32(s + val)
            assert abs(float(s)) < 2.0 ** 15 < 65504.0
            sh = np.float16(s)
            assert np.isfinite(sh) and np.isfinite(np.float16(s - np.float32(sh)))


def test_tc_x_scale_exponent_edges():
    bits = lambda f: int(np.float32(f).view(np.uint32))
    assert tc_scale_exponent(bits(1.0)) == 9             # 1 -> 512
    assert tc_scale_exponent(bits(1023.9)) == 0          # already in [2^9, 2^10)
    assert tc_scale_exponent(bits(512.0)) == 0
    assert tc_scale_exponent(bits(1024.0)) == -1
    assert tc_scale_exponent(bits(3.4e38)) == 9 - 127
    assert tc_scale_exponent(bits(1e-38)) == 126         # capped: 2^126 and 2^-126 stay normal
    assert tc_scale_exponent(1) == 126                   # smallest subnormal
    assert tc_scale_exponent(0) == 0
    assert tc_scale_exponent(0x7F800000) == 0            # inf: no scaling
    assert tc_scale_exponent(0x7FC00000) == 0            # NaN: no scaling


# ------------------------------------------------------------------ 3

K_MAGIC = np.float32(12582912.0)   # 1.5 * 2^23


def limbs(v: np.ndarray):
    """The batch-1 conversion of one 256-value block, step by step in f32."""
    amax = np.float32(np.max(np.abs(v)))
    s = np.float32(amax * np.float32(1.0 / 127.0))
    rcp = np.float32(1.0) / amax if amax > np.float32(1e-30) else np.float32(0.0)
    inv = np.float32(np.float32(127.0) * rcp)
    inv2 = np.float32(np.float32(254.0 * 127.0) * rcp)
    hi, lo = [], []
    for x in v:
        t = fma32(x, inv, K_MAGIC)
        h = np.float32(t - K_MAGIC)                       # exact
        r = fma32(-s, h, x)
        tl = fma32(r, inv2, K_MAGIC)
        hi.append(int(np.float32(t - K_MAGIC)))
        lo.append(int(np.float32(tl - K_MAGIC)))
        assert float(h) == hi[-1]
    return np.array(hi), np.array(lo), s, amax


@pytest.mark.parametrize("case", ["normal", "wide", "edge", "tiny", "spiky"])
def test_int8_limbs_stay_in_range_and_meet_the_bound(case):
    g = np.random.default_rng({"normal": 61, "wide": 62, "edge": 63, "tiny": 64, "spiky": 65}[case])
    for _ in range(12):
        if case == "normal":
            v = g.normal(0, 1, 256)
        elif case == "wide":
            v = g.normal(0, 1, 256) * 10.0 ** g.uniform(-6, 6, 256)
        elif case == "edge":
            amax = g.uniform(0.5, 2.0)
            v = g.choice([-1, 1], 256) * amax * (np.arange(256) % 128) / 127.0
            v[0] = amax                                    # exact multiples of s and the extremes
        elif case == "tiny":
            v = g.normal(0, 1e-20, 256)
        else:
            v = g.normal(0, 1e-3, 256)
            v[g.integers(0, 256)] = 5.0                    # one large value sets the scale
        v = v.astype(np.float32)
        hi, lo, s, amax = limbs(v)
        # no clamp needed: both limbs are int8 values
        assert np.all(np.abs(hi) <= 127) and np.all(np.abs(lo) <= 127), (case, hi.max(), lo.max())
        u = Fraction(float(s)) / 254
        for x, h, l in zip(v, hi, lo):
            err = abs(Fraction(float(x)) - u * (254 * int(h) + int(l)))
            assert err <= Fraction(float(amax)) / 64516 * Fraction(1001, 1000) + Fraction(1, 2 ** 140)

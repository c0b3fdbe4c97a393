"""Pins for the CPU oracle, checked against things other than the oracle itself.

Every function of the oracle is tied here to a library routine (numpy's
float16 and float64 matmul), a closed form on hand-built blocks, single-bit
flips that must change exactly the weights the layout predicts, exact
rational sums, or brute force over all codes.  A mistake such as a swapped
nibble, a wrong shift of the 6-bit scales, a dropped min term or a transposed
operand fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f16_bits(v: float) -> int:
    return int(np.array(v, dtype=np.float16).view(np.uint16))


# ---------------------------------------------------------------- fp16

def test_half_to_float_exhaustive_vs_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = oracle.half_to_float_array(h)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_double_to_half_vs_numpy():
    g = np.random.default_rng(123)
    mags = 10.0 ** g.uniform(-9, 5.5, size=20000)
    vals = list(mags * np.where(g.random(20000) < 0.5, -1, 1))
    # edge values: signed zero, subnormal ties, min normal, max finite, overflow ties
    q = 2.0 ** -24
    vals += [0.0, -0.0, q, q / 2, 3 * q / 2, 5 * q / 2, q * 1023.5, q * 1024, 2.0 ** -14,
             65504.0, 65519.99, 65520.0, -65520.0, 1e300, -1e-300,
             1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2049.0, 2051.0, 0.1, 1 / 3]
    for v in vals:
        want = int(np.array(v, dtype=np.float64).astype(np.float16).view(np.uint16))
        assert oracle.double_to_half(v) == want, v


# ---------------------------------------------------------------- Q8_0

def test_q8_0_closed_form():
    blk = np.zeros(34, dtype=np.uint8)
    blk[0:2] = np.array([f16_bits(0.5)], dtype="<u2").view(np.uint8)
    q = np.arange(32) - 16
    blk[2:] = q.astype(np.int8).view(np.uint8)
    w = oracle.decode_block("q8_0", blk)
    assert np.array_equal(w, 0.5 * q.astype(np.float32))


def test_q8_0_bit_flips():
    blk = synth.q8_0_random(1, 32, seed=5)
    base = oracle.decode_block("q8_0", blk)
    for byte in range(2, 34):
        for bit in range(8):
            b2 = blk.copy()
            b2[byte] ^= 1 << bit
            changed = np.nonzero(oracle.decode_block("q8_0", b2) != base)[0]
            assert list(changed) == [byte - 2]


# ---------------------------------------------------------------- Q4_K

def pack_q4_k(d: float, dmin: float, sc, m, q) -> np.ndarray:
    """Build a Q4_K block from fields, by the layout rule (written in the
    packing direction, independently of the oracle's unpacking)."""
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([f16_bits(d)], dtype="<u2").view(np.uint8)
    blk[2:4] = np.array([f16_bits(dmin)], dtype="<u2").view(np.uint8)
    s = np.zeros(12, dtype=np.int64)
    for j in range(8):
        if j < 4:
            s[j] |= sc[j]
            s[j + 4] |= m[j]
        else:
            s[j + 4] |= (sc[j] & 15) | ((m[j] & 15) << 4)
            s[j - 4] |= (sc[j] >> 4) << 6
            s[j] |= (m[j] >> 4) << 6
    blk[4:16] = s.astype(np.uint8)
    for i in range(256):
        c, p = divmod(i, 64)
        if p < 32:
            blk[16 + 32 * c + p] |= q[i]
        else:
            blk[16 + 32 * c + p - 32] |= q[i] << 4
    return blk


SC = [1, 17, 33, 63, 40, 5, 22, 48]   # high 2 bits exercised for every j >= 4 but one
MN = [0, 31, 16, 2, 33, 63, 9, 50]


def test_q4_k_scale_min_unpack():
    blk = pack_q4_k(1.0, 1.0, SC, MN, [0] * 256)
    for j in range(8):
        assert oracle.q4_k_scale_min(blk[4:16], j) == (SC[j], MN[j])


def test_q4_k_closed_form():
    q = [i % 16 for i in range(256)]
    blk = pack_q4_k(1.0, 0.5, SC, MN, q)
    w = oracle.decode_block("q4_k", blk)
    # weight i belongs to sub-block i // 32; w = sc*q - 0.5*m
    want = np.array([SC[i // 32] * q[i] - 0.5 * MN[i // 32] for i in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q4_k_rounding_single_subtraction():
    # d*sc*q and dmin*m are exact; the one rounding is the final subtraction.
    d, dmin = 0.0999755859375, 0.0333251953125   # exact fp16 values
    q = [(7 * i + 3) % 16 for i in range(256)]
    blk = pack_q4_k(d, dmin, SC, MN, q)
    w = oracle.decode_block("q4_k", blk)
    want = np.array([np.float32(Fraction(d) * SC[i // 32] * q[i] - Fraction(dmin) * MN[i // 32])
                     for i in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q4_k_bit_flips():
    blk = synth.random_records("q4_k", 1, 256, seed=9)
    base = oracle.decode_block("q4_k", blk)
    for byte in range(16, 144):
        c, l = divmod(byte - 16, 32)
        for bit in range(8):
            b2 = blk.copy()
            b2[byte] ^= 1 << bit
            changed = set(np.nonzero(oracle.decode_block("q4_k", b2) != base)[0])
            expect = 64 * c + l + (32 if bit >= 4 else 0)
            assert changed == {expect}, (byte, bit)
    # scale bytes: a bit may only change the sub-block whose sc or m it holds
    for byte in range(4, 16):
        for bit in range(8):
            jj = byte - 4
            if jj < 4:
                sub = jj if bit < 6 else jj + 4
            elif jj < 8:
                sub = jj - 4 if bit < 6 else jj
            else:
                sub = jj - 4
            b2 = blk.copy()
            b2[byte] ^= 1 << bit
            changed = set(np.nonzero(oracle.decode_block("q4_k", b2) != base)[0])
            assert changed, (byte, bit)
            assert changed <= set(range(32 * sub, 32 * sub + 32)), (byte, bit)


# ---------------------------------------------------------------- Q6_K

def pack_q6_k(d: float, sc, codes) -> np.ndarray:
    blk = np.zeros(210, dtype=np.uint8)
    for n in range(256):
        h, r = divmod(n, 128)
        t, l = divmod(r, 32)
        lo4, hi2 = codes[n] & 15, codes[n] >> 4
        qlb = 64 * h + l + (32 if t in (1, 3) else 0)
        blk[qlb] |= lo4 << (4 if t >= 2 else 0)
        blk[128 + 32 * h + l] |= hi2 << (2 * t)
    blk[192:208] = np.array(sc, dtype=np.int8).view(np.uint8)
    blk[208:210] = np.array([f16_bits(d)], dtype="<u2").view(np.uint8)
    return blk


def test_q6_k_closed_form():
    sc = [s - 8 for s in range(16)]
    codes = [(7 * n + 3) % 64 for n in range(256)]   # every code 0..63 occurs
    assert len(set(codes)) == 64
    w = oracle.decode_block("q6_k", pack_q6_k(0.25, sc, codes))
    want = np.array([0.25 * sc[n // 16] * (codes[n] - 32) for n in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q6_k_bit_flips():
    blk = synth.random_records("q6_k", 1, 256, seed=11)
    base = oracle.decode_block("q6_k", blk)

    def flip(byte, bit):
        b2 = blk.copy()
        b2[byte] ^= 1 << bit
        return set(np.nonzero(oracle.decode_block("q6_k", b2) != base)[0])

    for byte in range(128):
        h, b = divmod(byte, 64)
        for bit in range(8):
            expect = 128 * h + b + (64 if bit >= 4 else 0)
            assert flip(byte, bit) == {expect}, (byte, bit)
    for byte in range(128, 192):
        h, l = divmod(byte - 128, 32)
        for bit in range(8):
            expect = 128 * h + l + 32 * (bit // 2)
            assert flip(byte, bit) == {expect}, (byte, bit)
    for s in range(16):
        for bit in range(8):
            ch = flip(192 + s, bit)
            assert ch and ch <= set(range(16 * s, 16 * s + 16))


# ---------------------------------------------------------------- per-row int8

def test_i8_row_closed_form_and_layout():
    n_out, k = 3, 5
    q = (np.arange(n_out * k) - 7).astype(np.int8)
    buf = np.zeros(oracle.weight_bytes("i8_row", n_out, k), dtype=np.uint8)
    assert buf.size == 16 + 12            # 15 codes -> next 16-byte boundary, then 3 scales
    buf[: n_out * k] = q.view(np.uint8)
    s = np.array([0.5, -2.0, 3.0], dtype=np.float32)
    buf[16:28] = s.view(np.uint8)
    w = oracle.dequant("i8_row", buf, n_out, k)
    assert np.array_equal(w, (q.reshape(n_out, k) * s[:, None]).astype(np.float32))


# ---------------------------------------------------------------- sizes

def test_weight_bytes_match_the_workload_sizes():
    wb = oracle.weight_bytes
    assert wb("q8_0", 896, 896) == 852_992
    assert wb("q4_k", 4096, 4096) == 9_437_184
    assert wb("q4_k", 6144, 4096) == 14_155_776
    assert wb("q4_k", 28672, 4096) == 66_060_288
    assert wb("q4_k", 4096, 14336) == 33_030_144 == wb("q4_k", 14336, 4096)
    assert wb("q6_k", 128256, 4096) == 430_940_160
    for fmt in ("q8_0", "q4_k", "q6_k", "i8_row"):
        assert wb(fmt, 7, 512) == synth.weight_bytes(fmt, 7, 512)
    with pytest.raises(ValueError):
        wb("q4_k", 3, 100)


# ---------------------------------------------------------------- matrix decode

@pytest.mark.parametrize("fmt,k", [("q8_0", 96), ("q4_k", 512), ("q6_k", 768)])
def test_dequant_is_blockwise_decode(fmt, k):
    n_out = 5
    w = synth.random_records(fmt, n_out, k, seed=3)
    full = oracle.dequant(fmt, w, n_out, k)
    qk, bb = synth.BLOCK[fmt]
    for r in range(n_out):
        for b in range(k // qk):
            off = (r * (k // qk) + b) * bb
            assert np.array_equal(full[r, b * qk:(b + 1) * qk],
                                  oracle.decode_block(fmt, w[off:off + bb]))


# ---------------------------------------------------------------- mat-vec

def test_gemv_integer_special_case_vs_numpy():
    # Q8_0 with d = 1 and per-row int8 with scale 1 are plain integer matrices.
    n_out, k, batch = 37, 320, 3
    g = np.random.default_rng(7)
    qi = g.integers(-127, 128, size=(n_out, k))
    rec = np.zeros((n_out * k // 32, 34), dtype=np.uint8)
    rec[:, 0:2] = np.array([f16_bits(1.0)], dtype="<u2").view(np.uint8)
    rec[:, 2:] = qi.reshape(-1, 32).astype(np.int8).view(np.uint8)
    x = synth.normal_x(batch, k, seed=8)
    want = (qi.astype(np.float64) @ x.astype(np.float64).T).T
    y = oracle.gemv("q8_0", rec.ravel(), n_out, k, x)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)

    buf = np.zeros(oracle.weight_bytes("i8_row", n_out, k), dtype=np.uint8)
    buf[: n_out * k] = qi.astype(np.int8).view(np.uint8).ravel()
    off = (n_out * k + 15) // 16 * 16
    buf[off: off + 4 * n_out] = np.ones(n_out, dtype=np.float32).view(np.uint8)
    y2 = oracle.gemv("i8_row", buf, n_out, k, x)
    np.testing.assert_allclose(y2, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k"])
def test_gemv_exact_rational_tiny(fmt):
    n_out, k, batch = 3, 256, 2
    w = synth.random_records(fmt, n_out, k, seed=21)
    x = synth.normal_x(batch, k, seed=22)
    y = oracle.gemv(fmt, w, n_out, k, x)
    W = oracle.dequant(fmt, w, n_out, k)
    for b in range(batch):
        for r in range(n_out):
            exact = sum(Fraction(float(W[r, i])) * Fraction(float(x[b, i])) for i in range(k))
            mag = sum(abs(float(W[r, i]) * float(x[b, i])) for i in range(k))
            assert abs(float(exact) - y[b, r]) <= 1e-13 * mag + 1e-300


def test_gemv_one_hot_column_and_rows_subset():
    fmt, n_out, k = "q4_k", 9, 512
    w = synth.random_records(fmt, n_out, k, seed=4)
    W = oracle.dequant(fmt, w, n_out, k)
    x = np.zeros((2, k), dtype=np.float32)
    x[0, 300] = 1.0
    x[1, 7] = -1.0
    y = oracle.gemv(fmt, w, n_out, k, x)
    assert np.array_equal(y[0], W[:, 300].astype(np.float64))
    assert np.array_equal(y[1], -W[:, 7].astype(np.float64))
    xr = synth.normal_x(3, k, seed=1)
    rows = np.array([8, 0, 5])
    assert np.array_equal(oracle.gemv_rows(fmt, w, n_out, k, xr, rows),
                          oracle.gemv(fmt, w, n_out, k, xr)[:, rows])


def test_gemv_threads_do_not_change_results():
    fmt, n_out, k = "q6_k", 64, 512
    w = synth.random_records(fmt, n_out, k, seed=2)
    x = synth.normal_x(2, k, seed=3)
    assert np.array_equal(oracle.gemv(fmt, w, n_out, k, x, nthreads=1),
                          oracle.gemv(fmt, w, n_out, k, x, nthreads=4))


# ---------------------------------------------------------------- quantizers

def _code_table(fmt, blk, setter):
    """Decoded value of every code at every position, by decoding blocks
    whose codes were all overwritten (brute force over the code set)."""
    return [oracle.decode_block(fmt, setter(blk.copy(), c)) for c in range(64 if fmt == "q6_k" else 16)]


def _set_q4(blk, c):
    blk[16:] = c | (c << 4)
    return blk


def _set_q6(blk, c):
    lo, hi = c & 15, c >> 4
    blk[0:128] = lo | (lo << 4)
    blk[128:192] = hi | (hi << 2) | (hi << 4) | (hi << 6)
    return blk


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k"])
def test_quantizer_picks_the_nearest_code(fmt):
    n_out, k = 4, 256
    v = synth.normal_weights(n_out, k, seed=31)
    w = oracle.quantize(fmt, v)
    bb = synth.BLOCK[fmt][1]
    for r in range(n_out):
        blk = w[r * bb:(r + 1) * bb]
        got = oracle.decode_block(fmt, blk)
        table = np.stack(_code_table(fmt, blk, _set_q4 if fmt == "q4_k" else _set_q6))
        best = np.abs(table - v[r][None, :]).min(axis=0)
        err = np.abs(got - v[r])
        # nearest up to one f32 rounding of the decoded values
        assert np.all(err <= best + 2 * np.spacing(np.abs(v[r]) + np.abs(got))), r


def test_quantizer_q8_0_nearest_and_round_trip():
    n_out, k = 4, 128
    v = synth.normal_weights(n_out, k, seed=41)
    w = oracle.quantize("q8_0", v)
    vh = oracle.dequant("q8_0", w, n_out, k)
    rec = w.reshape(-1, 34)
    d = rec[:, 0:2].copy().view("<f2").astype(np.float64).ravel()
    step = np.repeat(d, 32).reshape(n_out, k)
    assert np.all(np.abs(vh - v) <= 0.5 * step * (1 + 1e-6))
    # decoded values re-quantize to the same bytes (max |v| decodes to d*127)
    assert np.array_equal(oracle.quantize("q8_0", vh), w)


def test_quantizer_i8_row_nearest():
    n_out, k = 6, 100
    v = synth.normal_weights(n_out, k, seed=51)
    w = oracle.quantize("i8_row", v)
    vh = oracle.dequant("i8_row", w, n_out, k)
    off = (n_out * k + 15) // 16 * 16
    s = w[off: off + 4 * n_out].view(np.float32).astype(np.float64)
    assert np.all(np.abs(vh - v) <= 0.5 * s[:, None] * (1 + 1e-6) + 1e-9)
    q = w[: n_out * k].view(np.int8).reshape(n_out, k)
    assert np.abs(q).max() == 127


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k"])
def test_quantizer_covers_the_range(fmt):
    # the decoded block must reproduce N(0,0.02) weights to a small fraction
    # of their spread, and codes at both ends of the range must be used
    v = synth.normal_weights(64, 1024, seed=61)
    vh = oracle.dequant(fmt, oracle.quantize(fmt, v), 64, 1024)
    rel = np.sqrt(np.mean((vh - v) ** 2)) / np.sqrt(np.mean(v ** 2))
    assert rel < (0.12 if fmt == "q4_k" else 0.03)


# ---------------------------------------------------------------- inputs

def test_synth_is_deterministic():
    a = synth.random_records("q4_k", 3, 512, seed=5)
    b = synth.random_records("q4_k", 3, 512, seed=5)
    c = synth.random_records("q4_k", 3, 512, seed=6)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert np.array_equal(synth.normal_x(2, 64, 1), synth.normal_x(2, 64, 1))
    q = synth.q8_0_random(2, 64, seed=0)
    assert np.array_equal(q, synth.q8_0_random(2, 64, seed=0))
    codes = q.reshape(-1, 34)[:, 2:].view(np.int8)
    assert codes.min() >= -127 and codes.max() <= 127

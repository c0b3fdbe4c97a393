"""Pins for the oracle's Q5_K, Q3_K and Q2_K decoders.

The pages name these formats only as members of the K family that PESTI
decodes (PESTI README, "What This Is"); their byte layouts
are the public GGUF ones, read as a byte specification.  Each decoder is tied
here to things other than itself: hand-built blocks packed by an inverse map
written separately from the decoder (closed forms, exact rational rounding),
and single-bit flips of random blocks that must change exactly the weights
the layout predicts.  A swapped nibble, a wrong high-bit position, a scale
taken from the wrong group or a dropped min term fails one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f16_bytes(v: float) -> np.ndarray:
    return np.array([v], dtype="<f2").view(np.uint8)


def decode(fmt, blk):
    return oracle.decode_block(fmt, blk)


def changed(fmt, blk, byte, bit, base):
    b2 = blk.copy()
    b2[byte] ^= 1 << bit
    return set(np.nonzero(decode(fmt, b2) != base)[0].tolist())


# ---------------------------------------------------------------- Q5_K

def pack_scales_k4(sc, m) -> np.ndarray:
    """The 12 packed bytes of eight 6-bit (scale, min) pairs (Q4_K / Q5_K)."""
    s = np.zeros(12, dtype=np.int64)
    for j in range(8):
        if j < 4:
            s[j] |= sc[j]
            s[j + 4] |= m[j]
        else:
            s[j + 4] |= (sc[j] & 15) | ((m[j] & 15) << 4)
            s[j - 4] |= (sc[j] >> 4) << 6
            s[j] |= (m[j] >> 4) << 6
    return s.astype(np.uint8)


def pack_q5_k(d, dmin, sc, m, q) -> np.ndarray:
    blk = np.zeros(176, dtype=np.uint8)
    blk[0:2], blk[2:4] = f16_bytes(d), f16_bytes(dmin)
    blk[4:16] = pack_scales_k4(sc, m)
    for i in range(256):
        c, p = divmod(i, 64)
        h, l = divmod(p, 32)
        blk[48 + 32 * c + l] |= (q[i] & 15) << (4 * h)
        blk[16 + l] |= (q[i] >> 4) << (2 * c + h)
    return blk


SC = [1, 17, 33, 63, 40, 5, 22, 48]
MN = [0, 31, 16, 2, 33, 63, 9, 50]


def test_q5_k_closed_form():
    q = [(5 * i + 1) % 32 for i in range(256)]
    w = decode("q5_k", pack_q5_k(1.0, 0.5, SC, MN, q))
    want = np.array([SC[i // 32] * q[i] - 0.5 * MN[i // 32] for i in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q5_k_fifth_bit_alone():
    # q = 16 exactly where the high bit is set: every weight is 16*sc or 0
    q = [16 if (i * 7) % 3 == 0 else 0 for i in range(256)]
    w = decode("q5_k", pack_q5_k(1.0, 0.0, SC, MN, q))
    assert np.array_equal(w, np.array([SC[i // 32] * q[i] for i in range(256)], dtype=np.float32))


def test_q5_k_rounding_single_subtraction():
    d, dmin = 0.0999755859375, 0.0333251953125   # exact fp16 values
    q = [(11 * i + 3) % 32 for i in range(256)]
    w = decode("q5_k", pack_q5_k(d, dmin, SC, MN, q))
    want = np.array([np.float32(Fraction(d) * SC[i // 32] * q[i] - Fraction(dmin) * MN[i // 32])
                     for i in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q5_k_bit_flips():
    blk = synth.random_records("q5_k", 1, 256, seed=31)
    base = decode("q5_k", blk)

    def one(i):   # a code bit of weight i moves it unless its sub-block scale is 0
        return {i} if oracle.q4_k_scale_min(blk[4:16], i // 32)[0] else set()

    for byte in range(48, 176):               # qs: one weight per bit
        c, l = divmod(byte - 48, 32)
        for bit in range(8):
            assert changed("q5_k", blk, byte, bit, base) == one(64 * c + l + (32 if bit >= 4 else 0))
    for byte in range(16, 48):                # qh: bit b of byte l -> weight 32*b + l
        l = byte - 16
        for bit in range(8):
            assert changed("q5_k", blk, byte, bit, base) == one(32 * bit + l), (byte, bit)
    for byte in range(4, 16):                 # scale bytes: only the sub-block they serve
        jj = byte - 4
        for bit in range(8):
            if jj < 4:
                sub = jj if bit < 6 else jj + 4
            elif jj < 8:
                sub = jj - 4 if bit < 6 else jj
            else:
                sub = jj - 4
            ch = changed("q5_k", blk, byte, bit, base)
            assert ch and ch <= set(range(32 * sub, 32 * sub + 32)), (byte, bit)


# ---------------------------------------------------------------- Q3_K

def pack_q3_k(d, sc16, values) -> np.ndarray:
    """sc16: 16 signed scales in -32..31; values: 256 in -4..3."""
    blk = np.zeros(110, dtype=np.uint8)
    t = np.zeros(12, dtype=np.int64)
    for s, v in enumerate(sc16):
        u = v + 32
        if s < 8:
            t[s] |= u & 15
        else:
            t[s - 8] |= (u & 15) << 4
        t[8 + s % 4] |= (u >> 4) << (2 * (s // 4))
    blk[96:108] = t.astype(np.uint8)
    for i, v in enumerate(values):
        n, r = divmod(i, 128)
        j, l = divmod(r, 32)
        high = 1 if v >= 0 else 0
        code = v if high else v + 4
        blk[32 + 32 * n + l] |= code << (2 * j)
        blk[l] |= high << (4 * n + j)
    blk[108:110] = f16_bytes(d)
    return blk


SC3 = [-32, -17, -1, 0, 1, 5, 12, 31, 30, -8, 16, -16, 7, -25, 24, 2]


def test_q3_k_scale_unpack():
    blk = pack_q3_k(1.0, SC3, [0] * 256)
    assert [oracle.q3_k_scale(blk[96:108], s) for s in range(16)] == SC3


def test_q3_k_closed_form_and_exact():
    values = [((3 * i + 1) % 8) - 4 for i in range(256)]
    d = 0.0999755859375
    w = decode("q3_k", pack_q3_k(d, SC3, values))
    want = np.array([np.float32(Fraction(d) * SC3[i // 16] * values[i]) for i in range(256)],
                    dtype=np.float32)
    assert np.array_equal(w, want)
    # every product is exact: no rounding anywhere
    assert all(Fraction(float(w[i])) == Fraction(d) * SC3[i // 16] * values[i] for i in range(256))


def test_q3_k_bit_flips():
    blk = synth.random_records("q3_k", 1, 256, seed=32)
    base = decode("q3_k", blk)

    def one(i):   # a code bit of weight i moves it unless its group's scale is 0
        return {i} if oracle.q3_k_scale(blk[96:108], i // 16) else set()

    for byte in range(0, 32):                 # hmask: bit 4n+j of byte l -> weight 128n+32j+l
        for bit in range(8):
            n, j = divmod(bit, 4)
            assert changed("q3_k", blk, byte, bit, base) == one(128 * n + 32 * j + byte), (byte, bit)
    for byte in range(32, 96):                # qs: bits 2j, 2j+1 of byte 32n+l -> weight 128n+32j+l
        n, l = divmod(byte - 32, 32)
        for bit in range(8):
            assert changed("q3_k", blk, byte, bit, base) == one(128 * n + 32 * (bit // 2) + l)
    for byte in range(96, 108):               # scale bytes: only the group they serve
        t = byte - 96
        for bit in range(8):
            if t < 8:
                grp = t if bit < 4 else t + 8
            else:
                grp = 4 * (bit // 2) + (t - 8)
            ch = changed("q3_k", blk, byte, bit, base)
            assert ch <= set(range(16 * grp, 16 * grp + 16)), (byte, bit)
            # weights whose value is 0 keep w = 0 whatever the scale
            vals = np.nonzero(base[16 * grp:16 * grp + 16])[0]
            assert len(ch) == len(vals), (byte, bit)


# ---------------------------------------------------------------- Q2_K

def pack_q2_k(d, dmin, sc16, m16, codes) -> np.ndarray:
    blk = np.zeros(84, dtype=np.uint8)
    blk[0:16] = (np.array(sc16) | (np.array(m16) << 4)).astype(np.uint8)
    for i, c in enumerate(codes):
        n, r = divmod(i, 128)
        j, l = divmod(r, 32)
        blk[16 + 32 * n + l] |= c << (2 * j)
    blk[80:82], blk[82:84] = f16_bytes(d), f16_bytes(dmin)
    return blk


SC2 = [0, 1, 15, 7, 9, 3, 12, 5, 14, 2, 11, 6, 8, 13, 4, 10]
MN2 = [15, 0, 3, 8, 1, 14, 6, 9, 2, 13, 5, 12, 10, 4, 11, 7]


def test_q2_k_closed_form():
    codes = [(i * 5 + 2) % 4 for i in range(256)]
    w = decode("q2_k", pack_q2_k(1.0, 0.25, SC2, MN2, codes))
    want = np.array([SC2[i // 16] * codes[i] - 0.25 * MN2[i // 16] for i in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q2_k_rounding_single_subtraction():
    d, dmin = 0.0999755859375, 0.0333251953125
    codes = [(i * 7 + 1) % 4 for i in range(256)]
    w = decode("q2_k", pack_q2_k(d, dmin, SC2, MN2, codes))
    want = np.array([np.float32(Fraction(d) * SC2[i // 16] * codes[i] - Fraction(dmin) * MN2[i // 16])
                     for i in range(256)], dtype=np.float32)
    assert np.array_equal(w, want)


def test_q2_k_bit_flips():
    blk = synth.random_records("q2_k", 1, 256, seed=33)
    blk[0:16] |= 1                            # every group scale nonzero: code flips show
    base = decode("q2_k", blk)
    for byte in range(16, 80):                # qs
        n, l = divmod(byte - 16, 32)
        for bit in range(8):
            assert changed("q2_k", blk, byte, bit, base) == {128 * n + 32 * (bit // 2) + l}
    for byte in range(0, 16):                 # scale byte s serves weights 16s..16s+15
        for bit in range(8):
            ch = changed("q2_k", blk, byte, bit, base)
            grp = set(range(16 * byte, 16 * byte + 16))
            assert ch <= grp, (byte, bit)
            if bit >= 4:
                assert ch == grp, (byte, bit)   # the min term moves every weight of the group


# ---------------------------------------------------------------- whole matrices

def test_weight_bytes_new_formats():
    for fmt, bb in (("q5_k", 176), ("q3_k", 110), ("q2_k", 84)):
        assert oracle.weight_bytes(fmt, 7, 512) == 7 * 2 * bb == synth.weight_bytes(fmt, 7, 512)
        with pytest.raises(ValueError):
            oracle.weight_bytes(fmt, 3, 100)


@pytest.mark.parametrize("fmt", ["q5_k", "q3_k", "q2_k"])
def test_dequant_is_blockwise_decode(fmt):
    n_out, k = 5, 768
    w = synth.random_records(fmt, n_out, k, seed=34)
    full = oracle.dequant(fmt, w, n_out, k)
    qk, bb = synth.BLOCK[fmt]
    for r in range(n_out):
        for b in range(k // qk):
            off = (r * (k // qk) + b) * bb
            assert np.array_equal(full[r, b * qk:(b + 1) * qk], decode(fmt, w[off:off + bb]))


@pytest.mark.parametrize("fmt", ["q5_k", "q3_k", "q2_k"])
def test_gemv_exact_rational_tiny(fmt):
    n_out, k, batch = 3, 256, 2
    w = synth.random_records(fmt, n_out, k, seed=35)
    x = synth.normal_x(batch, k, seed=36)
    y = oracle.gemv(fmt, w, n_out, k, x)
    W = oracle.dequant(fmt, w, n_out, k)
    for b in range(batch):
        for r in range(n_out):
            exact = sum(Fraction(float(W[r, i])) * Fraction(float(x[b, i])) for i in range(k))
            mag = sum(abs(float(W[r, i]) * float(x[b, i])) for i in range(k))
            assert abs(float(exact) - y[b, r]) <= 1e-13 * mag + 1e-300


@pytest.mark.parametrize("fmt", ["q5_k", "q3_k", "q2_k"])
def test_no_quantizer(fmt):
    with pytest.raises(RuntimeError):
        oracle.quantize(fmt, np.zeros((2, 256), dtype=np.float32))


# ---------------------------------------------------------------- per-row int4

def pack_i4_row(q, scales) -> np.ndarray:
    """q: [n_out, k] ints in -8..7; scales: n_out f32."""
    n_out, k = q.shape
    nq = n_out * k // 2
    buf = np.zeros((nq + 15) // 16 * 16 + 4 * n_out, dtype=np.uint8)
    codes = (np.asarray(q, dtype=np.int64) & 15).reshape(-1)
    buf[:nq] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    off = (nq + 15) // 16 * 16
    buf[off:off + 4 * n_out] = np.asarray(scales, dtype="<f4").view(np.uint8)
    return buf


def test_i4_row_closed_form_sign_and_layout():
    n_out, k = 3, 10                       # 15 code bytes: the scales start at byte 16
    q = np.array([[(r * 7 + i * 3) % 16 - 8 for i in range(k)] for r in range(n_out)])
    scales = [0.5, -0.25, 3.0]
    w = pack_i4_row(q, scales)
    assert oracle.weight_bytes("i4_row", n_out, k) == len(w) == 16 + 12
    got = oracle.dequant("i4_row", w, n_out, k)
    want = np.array([[np.float32(scales[r]) * np.float32(q[r, i]) for i in range(k)]
                     for r in range(n_out)], dtype=np.float32)
    assert np.array_equal(got, want)
    assert got.min() == -8 * 3.0          # code 8 reads as -8
    with pytest.raises(ValueError):
        oracle.weight_bytes("i4_row", 2, 7)


def test_i4_row_bit_flips():
    n_out, k = 2, 16
    w = synth.random_records("i4_row", n_out, k, seed=41)
    base = oracle.dequant("i4_row", w, n_out, k).ravel()
    for byte in range(n_out * k // 2):
        for bit in range(8):
            w2 = w.copy()
            w2[byte] ^= 1 << bit
            ch = set(np.nonzero(oracle.dequant("i4_row", w2, n_out, k).ravel() != base)[0].tolist())
            assert ch == {2 * byte + (1 if bit >= 4 else 0)}, (byte, bit)


def test_i4_row_quantizer_nearest_code():
    g = np.random.default_rng(42)
    v = g.normal(0, 0.02, size=(4, 64)).astype(np.float32)
    w = oracle.quantize("i4_row", v)
    deq = oracle.dequant("i4_row", w, 4, 64).astype(np.float64)
    off = (4 * 32 + 15) // 16 * 16
    s = w[off:off + 16].view("<f4").astype(np.float64)
    assert np.allclose(s, np.abs(v).max(axis=1) / 7.0, rtol=1e-6)
    for r in range(4):
        cand = s[r] * np.arange(-7, 8)               # every code the quantizer may choose
        best = np.abs(v[r][:, None].astype(np.float64) - cand[None, :]).min(axis=1)
        err = np.abs(v[r].astype(np.float64) - deq[r])
        assert np.all(err <= best + 1e-6 * s[r])

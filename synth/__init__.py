"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and places them into byte records.  It
holds none of the mat-vec's arithmetic (no decoding, no dot products, no
quantization rounding): the oracle quantizes, the CUDA library decodes.

Generators (numpy PCG64 via ``default_rng``):

* ``normal_weights``  W ~ N(0, 0.02) drawn in f64, stored f32, row-chunked
  so that the 128256 x 4096 output-head shape never holds f64 for the whole
  matrix at once.
* ``normal_x``        x ~ N(0, 1) drawn in f64, stored f32, shape [batch, k].
* ``q8_0_random``     Q8_0 records drawn directly: q uniform in [-127, 127],
  d = float16(max of 32 |N(0, 0.02)| draws / 127), the d field first
  (bytes 0-1, little-endian) then the 32 codes.
* ``random_records``  records of any format with every byte uniform except
  the fp16 scale fields, which get finite positive values from a stated
  range: every bit pattern of the packed scales, mins and codes occurs, so
  decoders see all of them.
* ``special_scale_records``  the same, but the scale fields (fp16 d/dmin, or
  the f32 row scales of the per-row formats) take every IEEE class: positive
  and negative normals, subnormals, signed zeros and, at a stated rate,
  infinities and NaNs (quiet and signalling, random payloads).

Byte offsets of the fp16 fields (the only layout facts used here):
Q8_0 d @0; Q4_K d @0, dmin @2; Q6_K d @208; Q5_K d @0, dmin @2; Q3_K d @108;
Q2_K d @80, dmin @82.  Per-row int8: codes [n_out*k] then f32 scales at the
next 16-byte boundary; per-row int4 the same with two codes per byte.
"""
from __future__ import annotations

import numpy as np

BLOCK = {"q8_0": (32, 34), "q4_k": (256, 144), "q6_k": (256, 210), "i8_row": (1, 1),
         "q5_k": (256, 176), "q3_k": (256, 110), "q2_k": (256, 84)}


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal_weights(n_out: int, k: int, seed: int, std: float = 0.02,
                   chunk_rows: int = 4096) -> np.ndarray:
    g = rng(seed)
    out = np.empty((n_out, k), dtype=np.float32)
    for r0 in range(0, n_out, chunk_rows):
        r1 = min(n_out, r0 + chunk_rows)
        out[r0:r1] = g.normal(0.0, std, size=(r1 - r0, k))
    return out


def normal_x(batch: int, k: int, seed: int) -> np.ndarray:
    return rng(seed).normal(0.0, 1.0, size=(batch, k)).astype(np.float32)


def weight_bytes(fmt: str, n_out: int, k: int) -> int:
    if fmt == "i8_row":
        return (n_out * k + 15) // 16 * 16 + 4 * n_out
    if fmt == "i4_row":
        assert k % 2 == 0
        return (n_out * k // 2 + 15) // 16 * 16 + 4 * n_out
    qk, bb = BLOCK[fmt]
    assert k % qk == 0
    return n_out * (k // qk) * bb


def q8_0_random(n_out: int, k: int, seed: int) -> np.ndarray:
    """Q8_0 records with q ~ U{-127..127} and d = f16(max|N(0,0.02)|/127)."""
    assert k % 32 == 0
    g = rng(seed)
    nblk = n_out * (k // 32)
    q = g.integers(-127, 128, size=(nblk, 32), dtype=np.int64).astype(np.int8)
    n = g.normal(0.0, 0.02, size=(nblk, 32))
    d = (np.abs(n).max(axis=1) / 127.0).astype(np.float16)
    rec = np.empty((nblk, 34), dtype=np.uint8)
    rec[:, 0:2] = d.astype("<f2").view(np.uint8).reshape(nblk, 2)
    rec[:, 2:34] = q.view(np.uint8)
    return rec.reshape(-1)


def _f16_field(g: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    v = g.uniform(lo, hi, size=n).astype(np.float16)
    return v.astype("<f2").view(np.uint8).reshape(n, 2)


def random_records(fmt: str, n_out: int, k: int, seed: int,
                   d_range=(2e-5, 4e-4), dmin_range=(1e-4, 2e-3)) -> np.ndarray:
    """Uniform random bytes with finite positive fp16 scale fields."""
    g = rng(seed)
    if fmt in ("i8_row", "i4_row"):
        total = weight_bytes(fmt, n_out, k)
        nq = n_out * k if fmt == "i8_row" else n_out * k // 2
        buf = np.zeros(total, dtype=np.uint8)
        buf[:nq] = np.frombuffer(g.bytes(nq), dtype=np.uint8)
        soff = (nq + 15) // 16 * 16
        s = g.uniform(1e-4, 4e-4, size=n_out).astype(np.float32)
        buf[soff: soff + 4 * n_out] = s.astype("<f4").view(np.uint8)
        return buf
    qk, bb = BLOCK[fmt]
    assert k % qk == 0
    nblk = n_out * (k // qk)
    rec = np.frombuffer(g.bytes(nblk * bb), dtype=np.uint8).reshape(nblk, bb).copy()
    if fmt == "q8_0":
        rec[:, 0:2] = _f16_field(g, nblk, *d_range)
    elif fmt == "q4_k":
        rec[:, 0:2] = _f16_field(g, nblk, *d_range)
        rec[:, 2:4] = _f16_field(g, nblk, *dmin_range)
    elif fmt == "q6_k":
        rec[:, 208:210] = _f16_field(g, nblk, *d_range)
    elif fmt == "q5_k":
        rec[:, 0:2] = _f16_field(g, nblk, *d_range)
        rec[:, 2:4] = _f16_field(g, nblk, *dmin_range)
    elif fmt == "q3_k":
        rec[:, 108:110] = _f16_field(g, nblk, *d_range)
    elif fmt == "q2_k":
        rec[:, 80:82] = _f16_field(g, nblk, *d_range)
        rec[:, 82:84] = _f16_field(g, nblk, *dmin_range)
    return rec.reshape(-1)


# fp16 / f32 scale fields of each record format: (offset, kind) per block, or
# the per-row f32 scales of the per-row formats
_SCALE_FIELDS = {"q8_0": (0,), "q4_k": (0, 2), "q6_k": (208,), "q5_k": (0, 2),
                 "q3_k": (108,), "q2_k": (80, 82)}


def _f16_class_bits(g: np.random.Generator, n: int, nonfinite: float) -> np.ndarray:
    """n fp16 bit patterns: finite classes (normal with exponent field 1..11,
    i.e. |v| in [2^-14, 2^-3), subnormal, zero; either sign) and, with
    probability `nonfinite`, +-inf or a NaN."""
    sign = g.integers(0, 2, n).astype(np.uint16) << 15
    cls = g.choice(3, size=n, p=[0.7, 0.2, 0.1])                # normal, subnormal, zero
    exp = np.where(cls == 0, g.integers(1, 12, n), 0).astype(np.uint16)
    man = np.where(cls == 2, 0, g.integers(0, 1024, n)).astype(np.uint16)
    man = np.where((cls == 1) & (man == 0), 1, man).astype(np.uint16)
    bits = sign | (exp << 10) | man
    bad = g.random(n) < nonfinite
    nan = g.random(n) < 0.5
    payload = g.integers(1, 1024, n).astype(np.uint16)
    special = sign | np.uint16(0x7C00) | np.where(nan, payload, 0).astype(np.uint16)
    return np.where(bad, special, bits).astype(np.uint16)


def _f32_class_bits(g: np.random.Generator, n: int, nonfinite: float) -> np.ndarray:
    sign = g.integers(0, 2, n).astype(np.uint32) << 31
    cls = g.choice(3, size=n, p=[0.7, 0.2, 0.1])
    exp = np.where(cls == 0, g.integers(100, 121, n), 0).astype(np.uint32)
    man = np.where(cls == 2, 0, g.integers(0, 1 << 23, n)).astype(np.uint32)
    man = np.where((cls == 1) & (man == 0), 1, man).astype(np.uint32)
    bits = sign | (exp << 23) | man
    bad = g.random(n) < nonfinite
    nan = g.random(n) < 0.5
    payload = g.integers(1, 1 << 23, n).astype(np.uint32)
    special = sign | np.uint32(0x7F800000) | np.where(nan, payload, 0).astype(np.uint32)
    return np.where(bad, special, bits).astype(np.uint32)


def special_scale_records(fmt: str, n_out: int, k: int, seed: int, nonfinite: float = 0.05) -> np.ndarray:
    """Uniform random bytes whose scale fields take every IEEE class; each
    scale field is non-finite with probability `nonfinite`."""
    g = rng(seed)
    if fmt in ("i8_row", "i4_row"):
        buf = random_records(fmt, n_out, k, seed)
        nq = n_out * k if fmt == "i8_row" else n_out * k // 2
        soff = (nq + 15) // 16 * 16
        buf[soff: soff + 4 * n_out] = _f32_class_bits(g, n_out, nonfinite).astype("<u4").view(np.uint8)
        return buf
    qk, bb = BLOCK[fmt]
    nblk = n_out * (k // qk)
    rec = random_records(fmt, n_out, k, seed).reshape(nblk, bb).copy()
    for off in _SCALE_FIELDS[fmt]:
        rec[:, off:off + 2] = _f16_class_bits(g, nblk, nonfinite).astype("<u2").view(np.uint8).reshape(nblk, 2)
    return rec.reshape(-1)

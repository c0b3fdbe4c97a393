"""CPU oracle for the block-quantized mat-vec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it.

This is a ctypes shim over ``pq_oracle.c`` (plain C, f64 accumulation,
``-ffp-contract=off``).  What each function computes, and the passage it
follows, is documented in that file.  Every function here only marshals
numpy arrays.

Parity pins (checked by ``tests/test_oracle.py``):
  * fp16 decode: exhaustive against numpy's float16;
  * f64 -> fp16 encode: against numpy's float16 on random and edge values;
  * Q8_0 / Q4_K / Q6_K / per-row int8 decode: hand-built blocks with closed
    forms, and single-bit flips that must change exactly the predicted
    weights;
  * Q5_K / Q3_K / Q2_K decode: the same kinds of pins (closed forms on
    hand-built blocks, every single-bit flip of random blocks against the
    weights and amounts the layout predicts); no quantizer for them;
  * per-row int4: closed form incl. the scale offset and sign extension,
    single-bit flips, brute-force nearest code for the quantizer;
  * f64 mat-vec: integer-valued special cases against numpy's float64
    matmul, and exact rational sums on tiny shapes;
  * quantizers: brute-force best code on tiny matrices, re-quantization
    round trips, and the rounding error bound.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q8_0, Q4_K, Q6_K, I8_ROW, Q5_K, Q3_K, Q2_K, I4_ROW = 0, 1, 2, 3, 4, 5, 6, 7
FORMATS = {"q8_0": Q8_0, "q4_k": Q4_K, "q6_k": Q6_K, "i8_row": I8_ROW,
           "q5_k": Q5_K, "q3_k": Q3_K, "q2_k": Q2_K, "i4_row": I4_ROW}
# weights and bytes per block of the block formats
BLOCKS = {Q8_0: (32, 34), Q4_K: (256, 144), Q6_K: (256, 210), Q5_K: (256, 176),
          Q3_K: (256, 110), Q2_K: (256, 84)}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pq_oracle.c")
_SO = os.path.join(_HERE, "_pq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pq_oracle.c into an in-tree shared library (gcc, OpenMP)."""
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            L.pqo_half_to_float.argtypes = [ctypes.c_uint16]
            L.pqo_half_to_float.restype = ctypes.c_float
            L.pqo_double_to_half.argtypes = [ctypes.c_double]
            L.pqo_double_to_half.restype = ctypes.c_uint16
            L.pqo_weight_bytes.argtypes = [i32, i64, i64]
            L.pqo_weight_bytes.restype = i64
            for name in ("pqo_decode_q8_0", "pqo_decode_q4_k", "pqo_decode_q6_k",
                         "pqo_decode_q5_k", "pqo_decode_q3_k", "pqo_decode_q2_k"):
                getattr(L, name).argtypes = [vp, vp]
                getattr(L, name).restype = None
            L.pqo_q4_k_scale_min.argtypes = [vp, i32, vp, vp]
            L.pqo_q4_k_scale_min.restype = None
            L.pqo_q3_k_scale.argtypes = [vp, i32]
            L.pqo_q3_k_scale.restype = i32
            L.pqo_dequant.argtypes = [i32, vp, i64, i64, vp, i32]
            L.pqo_dequant.restype = i32
            L.pqo_gemv.argtypes = [i32, vp, i64, i64, vp, i64, vp, i32]
            L.pqo_gemv.restype = i32
            L.pqo_gemv_rows.argtypes = [i32, vp, i64, i64, vp, i64, vp, i64, vp, i32]
            L.pqo_gemv_rows.restype = i32
            L.pqo_quantize.argtypes = [i32, vp, i64, i64, vp, i32]
            L.pqo_quantize.restype = i32
            L.pqo_threads.argtypes = [i32]
            L.pqo_threads.restype = i32
            L.pqo_silu.argtypes = [ctypes.c_double]
            L.pqo_silu.restype = ctypes.c_double
            L.pqo_gemv_swiglu.argtypes = [i32, vp, i64, i64, vp, i64, vp, i32]
            L.pqo_gemv_swiglu.restype = i32
            L.pqo_gemv_bias.argtypes = [i32, vp, i64, i64, vp, i64, vp, vp, i32]
            L.pqo_gemv_bias.restype = i32
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def weight_bytes(fmt, n_out: int, k: int) -> int:
    n = lib().pqo_weight_bytes(_fmt(fmt), n_out, k)
    if n < 0:
        raise ValueError(f"k={k} is not a multiple of the block size of format {fmt}")
    return int(n)


def threads(nthreads: int = 0) -> int:
    """Threads an OpenMP region of the oracle gets for this request."""
    return int(lib().pqo_threads(nthreads))


def half_to_float(h: int) -> float:
    return float(lib().pqo_half_to_float(int(h)))


def half_to_float_array(h: np.ndarray) -> np.ndarray:
    L = lib()
    return np.array([L.pqo_half_to_float(int(v)) for v in np.asarray(h).ravel()],
                    dtype=np.float32).reshape(np.shape(h))


def double_to_half(v: float) -> int:
    return int(lib().pqo_double_to_half(float(v)))


def decode_block(fmt, blk: np.ndarray) -> np.ndarray:
    fmt = _fmt(fmt)
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    n, need = BLOCKS[fmt]
    if blk.size != need:
        raise ValueError(f"block of format {fmt} has {need} bytes, got {blk.size}")
    out = np.empty(n, dtype=np.float32)
    L = lib()
    fn = {Q8_0: L.pqo_decode_q8_0, Q4_K: L.pqo_decode_q4_k, Q6_K: L.pqo_decode_q6_k,
          Q5_K: L.pqo_decode_q5_k, Q3_K: L.pqo_decode_q3_k, Q2_K: L.pqo_decode_q2_k}[fmt]
    fn(_ptr(blk), _ptr(out))
    return out


def q4_k_scale_min(scales12: np.ndarray, j: int) -> tuple[int, int]:
    s = np.ascontiguousarray(scales12, dtype=np.uint8)
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().pqo_q4_k_scale_min(_ptr(s), j, ctypes.addressof(sc), ctypes.addressof(m))
    return sc.value, m.value


def q3_k_scale(scales12: np.ndarray, s: int) -> int:
    """Signed 6-bit scale of group s (0..15) of a Q3_K super-block."""
    t = np.ascontiguousarray(scales12, dtype=np.uint8)
    return int(lib().pqo_q3_k_scale(_ptr(t), s))


def _check_w(fmt, w: np.ndarray, n_out: int, k: int) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint8).ravel()
    need = weight_bytes(fmt, n_out, k)
    if w.size < need:
        raise ValueError(f"weights hold {w.size} bytes, {need} needed")
    return w


def dequant(fmt, w: np.ndarray, n_out: int, k: int, nthreads: int = 0) -> np.ndarray:
    w = _check_w(fmt, w, n_out, k)
    out = np.empty((n_out, k), dtype=np.float32)
    rc = lib().pqo_dequant(_fmt(fmt), _ptr(w), n_out, k, _ptr(out), nthreads)
    if rc:
        raise RuntimeError(f"pqo_dequant failed ({rc})")
    return out


def gemv(fmt, w: np.ndarray, n_out: int, k: int, x: np.ndarray,
         nthreads: int = 0) -> np.ndarray:
    """y[b][r] = sum_i w[r][i]*x[b][i] in f64; x is [batch, k] f32."""
    w = _check_w(fmt, w, n_out, k)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    assert x.shape[1] == k
    y = np.empty((x.shape[0], n_out), dtype=np.float64)
    rc = lib().pqo_gemv(_fmt(fmt), _ptr(w), n_out, k, _ptr(x), x.shape[0], _ptr(y), nthreads)
    if rc:
        raise RuntimeError(f"pqo_gemv failed ({rc})")
    return y


def gemv_rows(fmt, w: np.ndarray, n_out: int, k: int, x: np.ndarray,
              rows: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """The same sums for the listed rows only: returns [batch, len(rows)]."""
    w = _check_w(fmt, w, n_out, k)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < n_out)
    y = np.empty((x.shape[0], rows.size), dtype=np.float64)
    rc = lib().pqo_gemv_rows(_fmt(fmt), _ptr(w), n_out, k, _ptr(x), x.shape[0],
                             _ptr(rows), rows.size, _ptr(y), nthreads)
    if rc:
        raise RuntimeError(f"pqo_gemv_rows failed ({rc})")
    return y


def silu(z: float) -> float:
    return float(lib().pqo_silu(float(z)))


def gemv_swiglu(fmt, w: np.ndarray, n_ff: int, k: int, x: np.ndarray,
                nthreads: int = 0) -> np.ndarray:
    """h[b, j] = silu((W x_b)[j]) * (W x_b)[n_ff + j] for a fused gate+up W of
    2*n_ff rows, in f64; [batch, n_ff]."""
    w = _check_w(fmt, w, 2 * n_ff, k)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    h = np.empty((x.shape[0], n_ff), dtype=np.float64)
    rc = lib().pqo_gemv_swiglu(_fmt(fmt), _ptr(w), n_ff, k, _ptr(x), x.shape[0], _ptr(h), nthreads)
    if rc:
        raise RuntimeError(f"pqo_gemv_swiglu failed ({rc})")
    return h


def gemv_bias(fmt, w: np.ndarray, n_out: int, k: int, x: np.ndarray, bias: np.ndarray,
              nthreads: int = 0) -> np.ndarray:
    """y[b, r] = (W x_b)[r] + bias[r] in f64; [batch, n_out]."""
    w = _check_w(fmt, w, n_out, k)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    assert bias.shape == (n_out,)
    y = np.empty((x.shape[0], n_out), dtype=np.float64)
    rc = lib().pqo_gemv_bias(_fmt(fmt), _ptr(w), n_out, k, _ptr(x), x.shape[0], _ptr(bias), _ptr(y),
                             nthreads)
    if rc:
        raise RuntimeError(f"pqo_gemv_bias failed ({rc})")
    return y


def quantize(fmt, v: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """Quantize an f32 matrix [n_out, k] into the format's bytes."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    n_out, k = v.shape
    out = np.empty(weight_bytes(fmt, n_out, k), dtype=np.uint8)
    rc = lib().pqo_quantize(_fmt(fmt), _ptr(v), n_out, k, _ptr(out), nthreads)
    if rc:
        raise RuntimeError(f"pqo_quantize failed ({rc})")
    return out

"""Python binding of the block-quantized mat-vec library (``libpq.so``).

Argument marshalling only: every function forwards to the C ABI declared in
``include/pq.h`` under the same name.  Pointer arguments accept a torch
tensor (its ``data_ptr()``) or a plain integer address; ``stream`` accepts a
``torch.cuda.Stream``, a raw handle, or None for torch's current stream.
``fmt`` is a name from ``FORMATS`` ("q8_0", "q4_k", "q6_k", "q5_k", "q3_k",
"q2_k", "i8_row", "i4_row") or the ``pq_fmt`` value itself.
A missing or unloadable library raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

Q8_0, Q4_K, Q6_K, I8_ROW, Q5_K, Q3_K, Q2_K, I4_ROW = 0, 1, 2, 3, 4, 5, 6, 7
FORMATS = {"q8_0": Q8_0, "q4_k": Q4_K, "q6_k": Q6_K, "i8_row": I8_ROW,
           "q5_k": Q5_K, "q3_k": Q3_K, "q2_k": Q2_K, "i4_row": I4_ROW}
KERNEL_AUTO, KERNEL_GENERIC, KERNEL_STREAM, KERNEL_TC = -1, 0, 1, 2
KERNELS = {"auto": KERNEL_AUTO, "generic": KERNEL_GENERIC, "stream": KERNEL_STREAM, "tc": KERNEL_TC}

PQ_OK = 0
PQ_ERR_ARG, PQ_ERR_FMT, PQ_ERR_K, PQ_ERR_ALIGN = -1, -2, -3, -4
PQ_ERR_SIZE, PQ_ERR_DEVICE, PQ_ERR_LAUNCH, PQ_ERR_KERNEL = -5, -6, -7, -8

LIB_PATH = os.environ.get("PQ_LIB_PATH") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libpq.so")
EXPORTS = ("pq_gemv", "pq_dequant", "pq_weight_bytes", "pq_strerror",
           "pq_gemv_kernel", "pq_gemv_choice", "pq_gemv_launches", "pq_wait_timeouts",
           "pq_set_weight_prefetch", "pq_gemv_noalloc", "pq_selftest_wait_timeout",
           "pq_gemv_bias", "pq_gemv_swiglu")

_lock = threading.Lock()
_lib = None


class PQError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {pq_strerror(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libpq.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                                   "(run quantized_weight_mat_gb300.build.build())")
            L = ctypes.CDLL(LIB_PATH)
            i32, vp, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            L.pq_gemv.argtypes = [i32, vp, i32, i32, vp, i32, vp, vp]
            L.pq_gemv.restype = i32
            L.pq_gemv_kernel.argtypes = [i32, vp, i32, i32, vp, i32, vp, vp, i32]
            L.pq_gemv_kernel.restype = i32
            L.pq_dequant.argtypes = [i32, vp, i32, i32, vp, vp]
            L.pq_dequant.restype = i32
            L.pq_weight_bytes.argtypes = [i32, i32, i32]
            L.pq_weight_bytes.restype = sz
            L.pq_strerror.argtypes = [i32]
            L.pq_strerror.restype = ctypes.c_char_p
            L.pq_gemv_choice.argtypes = [i32, i32, i32, i32]
            L.pq_gemv_choice.restype = i32
            L.pq_gemv_launches.argtypes = [i32, i32, i32, i32]
            L.pq_gemv_launches.restype = i32
            L.pq_wait_timeouts.argtypes = [i32]
            L.pq_wait_timeouts.restype = i32
            L.pq_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
            L.pq_selftest_wait_timeout.restype = i32
            L.pq_gemv_noalloc.argtypes = [i32, vp, i32, i32, vp, i32, vp, vp]
            L.pq_gemv_noalloc.restype = i32
            L.pq_gemv_bias.argtypes = [i32, vp, i32, i32, vp, i32, vp, vp, vp]
            L.pq_gemv_bias.restype = i32
            L.pq_gemv_swiglu.argtypes = [i32, vp, i32, i32, vp, i32, vp, vp]
            L.pq_gemv_swiglu.restype = i32
            L.pq_set_weight_prefetch.argtypes = [i32]
            L.pq_set_weight_prefetch.restype = i32
            _lib = L
    return _lib


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _addr(p) -> int:
    if p is None:
        return 0
    if isinstance(p, int):
        return p
    return int(p.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def pq_strerror(status: int) -> str:
    return lib().pq_strerror(int(status)).decode()


def pq_weight_bytes(fmt, n_out: int, k: int) -> int:
    return int(lib().pq_weight_bytes(_fmt(fmt), int(n_out), int(k)))


def pq_gemv(fmt, w_blocks, n_out: int, k: int, x, batch: int, y, stream=None,
            check: bool = True) -> int:
    st = lib().pq_gemv(_fmt(fmt), _addr(w_blocks), int(n_out), int(k), _addr(x), int(batch),
                       _addr(y), _stream(stream))
    if check and st:
        raise PQError(st, "pq_gemv")
    return st


def pq_gemv_kernel(fmt, w_blocks, n_out: int, k: int, x, batch: int, y, stream=None,
                   kernel="auto", check: bool = True) -> int:
    kid = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    st = lib().pq_gemv_kernel(_fmt(fmt), _addr(w_blocks), int(n_out), int(k), _addr(x),
                              int(batch), _addr(y), _stream(stream), kid)
    if check and st:
        raise PQError(st, "pq_gemv_kernel")
    return st


def pq_gemv_bias(fmt, w_blocks, n_out: int, k: int, x, batch: int, bias, y, stream=None,
                 check: bool = True) -> int:
    """y = W x + bias (bias [n_out], fused into the store where the kernel allows)."""
    st = lib().pq_gemv_bias(_fmt(fmt), _addr(w_blocks), int(n_out), int(k), _addr(x), int(batch),
                            _addr(bias), _addr(y), _stream(stream))
    if check and st:
        raise PQError(st, "pq_gemv_bias")
    return st


def pq_gemv_swiglu(fmt, w_blocks, n_ff: int, k: int, x, batch: int, h, stream=None,
                   check: bool = True) -> int:
    """h = silu(W_gate x) * (W_up x) for a fused gate+up W of 2 * n_ff rows (gate rows first)."""
    st = lib().pq_gemv_swiglu(_fmt(fmt), _addr(w_blocks), int(n_ff), int(k), _addr(x), int(batch),
                              _addr(h), _stream(stream))
    if check and st:
        raise PQError(st, "pq_gemv_swiglu")
    return st


def pq_dequant(fmt, w_blocks, n_out: int, k: int, out, stream=None, check: bool = True) -> int:
    st = lib().pq_dequant(_fmt(fmt), _addr(w_blocks), int(n_out), int(k), _addr(out),
                          _stream(stream))
    if check and st:
        raise PQError(st, "pq_dequant")
    return st


def pq_gemv_choice(fmt, n_out: int, k: int, batch: int) -> int:
    return int(lib().pq_gemv_choice(_fmt(fmt), int(n_out), int(k), int(batch)))


def pq_gemv_launches(fmt, n_out: int, k: int, batch: int) -> int:
    return int(lib().pq_gemv_launches(_fmt(fmt), int(n_out), int(k), int(batch)))


def pq_wait_timeouts(reset: bool = False) -> int:
    return int(lib().pq_wait_timeouts(1 if reset else 0))


def pq_set_weight_prefetch(enable: bool) -> int:
    return int(lib().pq_set_weight_prefetch(1 if enable else 0))


def pq_gemv_noalloc(fmt, w_blocks, n_out: int, k: int, x, batch: int, y, stream=None,
                    check: bool = True) -> int:
    """Allocation-free mat-vec (fixed device scratch; see include/pq.h)."""
    st = lib().pq_gemv_noalloc(_fmt(fmt), _addr(w_blocks), int(n_out), int(k), _addr(x),
                               int(batch), _addr(y), _stream(stream))
    if check and st:
        raise PQError(st, "pq_gemv_noalloc")
    return st


def pq_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    """Bounded-wait self-test (see include/pq.h): 1 when the wait ran out as designed."""
    return int(lib().pq_selftest_wait_timeout(int(limit_us), _stream(stream)))

"""Device I/O helpers shared by the GPU tests (torch is used for device
memory only; every computation goes through the library's C ABI)."""
from __future__ import annotations

import numpy as np

import quantized_weight_mat_gb300 as pq

GUARD = 64
SENTINEL_BITS = 0x7fc0beef
SENTINEL = np.float32(np.frombuffer(np.uint32(SENTINEL_BITS).tobytes(), dtype=np.float32)[0])


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def out_buf(n):
    """A device f32 buffer of n values plus a guard band, all set to a NaN
    sentinel."""
    import torch
    t = torch.empty(n + GUARD, dtype=torch.float32, device="cuda")
    t.fill_(float(SENTINEL))
    return t


def guard_intact(t, n):
    g = t[n:].cpu().numpy().view(np.uint32)
    return bool(np.all(g == np.uint32(SENTINEL_BITS)))


def run_gemv(fmt, w, n_out, k, x, kernel="auto"):
    """y [batch, n_out] from pq_gemv_kernel, or None when that kernel does not
    take the case; asserts the guard band stayed untouched."""
    import torch
    batch = x.shape[0]
    wd, xd = dev(w), dev(x)
    y = out_buf(batch * n_out)
    st = pq.pq_gemv_kernel(fmt, wd, n_out, k, xd, batch, y, kernel=kernel, check=False)
    torch.cuda.synchronize()
    if st == pq.PQ_ERR_KERNEL:
        return None
    assert st == 0, pq.pq_strerror(st)
    assert guard_intact(y, batch * n_out)
    return y[: batch * n_out].cpu().numpy().reshape(batch, n_out)


def run_dequant(fmt, w, n_out, k):
    import torch
    out = out_buf(n_out * k)
    pq.pq_dequant(fmt, dev(w), n_out, k, out)
    torch.cuda.synchronize()
    assert guard_intact(out, n_out * k)
    return out[: n_out * k].cpu().numpy().reshape(n_out, k)

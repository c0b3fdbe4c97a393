"""The allocation-free mat-vec (pq_gemv_noalloc), through the C ABI.

Some callers cannot allocate device memory once they run: a serving process
whose memory was carved up ahead of time, a runtime with a fixed memory plan,
or code recorded into a legacy-stream capture.  pq_gemv_noalloc runs the
tensor-core kernel with its scratch in a fixed device array instead of pool
memory.  This file checks it on two calls in a row with different inputs:

* against the oracle, within the mat-vec bar of the parity tests,
  max|y - y_ref| <= 2e-3 * RMS(y_ref) + 1e-6;
* bit for bit against pq_gemv_kernel(..., "tc"), the same deterministic
  kernel with its scratch drawn from the pool, so only the scratch differs.

Collected last on purpose: it must pass after every other test of the suite
(the shared device array then holds whatever earlier calls left) as well as
alone in a fresh process (the first call does the per-device set-up).
"""
import numpy as np
import pytest

import oracle
import quantized_weight_mat_gb300 as pq
import synth
from pqcases import tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup(cuda_ok):
    from quantized_weight_mat_gb300 import build
    build.build()
    import torch
    torch.cuda.init()


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def both(w, n_out, k, x):
    """(y from pq_gemv_noalloc, y from the same tensor-core kernel with pool scratch)."""
    import torch
    batch = x.shape[0]
    wd, xd = dev(w), dev(x)
    y_na = torch.full((batch * n_out,), float("nan"), dtype=torch.float32, device="cuda")
    y_tc = torch.full((batch * n_out,), float("nan"), dtype=torch.float32, device="cuda")
    pq.pq_gemv_noalloc("q4_k", wd, n_out, k, xd, batch, y_na)
    for b0 in range(0, batch, 16):                 # pq_gemv_kernel takes up to 16 columns per call
        nb = min(16, batch - b0)
        pq.pq_gemv_kernel("q4_k", wd, n_out, k, xd.reshape(-1)[b0 * k:], nb, y_tc[b0 * n_out:], kernel="tc")
    torch.cuda.synchronize()
    return y_na.cpu().numpy().reshape(batch, n_out), y_tc.cpu().numpy().reshape(batch, n_out)


@pytest.mark.parametrize("n_out,k,batches", [
    (1000, 4096, (8, 13)),      # ragged last tile; 8 then 13 columns (two image widths)
    (4096, 14336, (16, 5)),     # down projection shape, near the scratch limit
    (384, 16384, (20, 3)),      # k at the limit; 20 columns run as chunks of 16 + 4
    (14336, 4096, (1, 2)),      # batch 1 and 2 run the tensor-core kernel too
])
def test_two_calls_in_a_row_match_the_oracle(n_out, k, batches):
    w = synth.random_records("q4_k", n_out, k, seed=70 + n_out % 7)
    for i, batch in enumerate(batches):
        x = synth.normal_x(batch, k, seed=80 + i)
        if i == 1:
            x[0] *= np.float32(1e6)                  # wide-range x on the second call
        y_na, y_tc = both(w, n_out, k, x)
        assert np.all(np.isfinite(y_na))
        ok, err, bound = tolerance_ok(y_na, oracle.gemv("q4_k", w, n_out, k, x))
        assert ok, f"call {i}: batch {batch}: max err {err} > {bound}"
        assert np.array_equal(y_na.view(np.uint32), y_tc.view(np.uint32)), f"call {i}: differs from pq_gemv_kernel tc"


def test_limits_are_reported_before_any_launch():
    import torch
    k_big = 16640
    w = torch.zeros(synth.weight_bytes("q4_k", 8, k_big), dtype=torch.uint8, device="cuda")
    x = torch.zeros(k_big, dtype=torch.float32, device="cuda")
    y = torch.zeros(8, dtype=torch.float32, device="cuda")
    assert pq.pq_gemv_noalloc("q4_k", w, 8, k_big, x, 1, y, check=False) == pq.PQ_ERR_SIZE
    w8 = torch.zeros(synth.weight_bytes("q8_0", 8, 256), dtype=torch.uint8, device="cuda")
    assert pq.pq_gemv_noalloc("q8_0", w8, 8, 256, x, 1, y, check=False) == pq.PQ_ERR_KERNEL
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0

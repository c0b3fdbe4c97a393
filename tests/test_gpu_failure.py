"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes runs out, is counted, and the kernel returns; the context stays
usable (a normal call afterwards matches the oracle)."""
import numpy as np
import pytest

import oracle
import quantized_weight_mat_gb300 as pq
from pqcases import tolerance_ok, weights, x_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup(cuda_ok):
    from quantized_weight_mat_gb300 import build
    build.build()
    import torch
    torch.cuda.init()


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    import torch
    before = pq.pq_wait_timeouts(reset=False)
    assert pq.pq_selftest_wait_timeout(2000) == 1        # a 2 ms wait on a barrier nothing completes
    assert pq.pq_wait_timeouts(reset=False) == before + 1
    # the same context still runs the library correctly
    n_out, k = 300, 2048
    w = weights("q4_k", n_out, k, "quantized", 3)
    x = x_for(2, k, 4)
    y = torch.empty(2 * n_out, dtype=torch.float32, device="cuda")
    pq.pq_gemv("q4_k", torch.from_numpy(w).cuda(), n_out, k, torch.from_numpy(x).cuda(), 2, y)
    torch.cuda.synchronize()
    ok, err, bound = tolerance_ok(y.cpu().numpy().reshape(2, n_out), oracle.gemv("q4_k", w, n_out, k, x))
    assert ok, (err, bound)
    pq.pq_wait_timeouts(reset=True)                      # leave the counter clean for later tests
    assert pq.pq_wait_timeouts(reset=False) == 0

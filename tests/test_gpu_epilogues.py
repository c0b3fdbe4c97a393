"""GPU parity of the fused epilogues, through the C ABI, against the oracle.

pq_gemv_swiglu: h[b][j] = silu(g) * u with g, u rows j and n_ff + j of a fused
gate+up matrix (gate rows first); pq_gemv_bias: y = W x + bias (PESTI README,
"Conformance").  Bar: max|out - ref| <= 2e-3 * RMS(ref) + 1e-6, the
mat-vec's bar applied to the epilogue's output: the kernels' per-output error
(about 2e-5 RMS on the batch-1 path) grows through silu(g) * u by a factor of
about 20 at the worst output, well inside it.  Batch 1 runs the whole-row
kernel with the epilogue in its stores; Q4_K and Q6_K at k = 4096 and
batch 2-8 the register-operand kernel, also with it in its stores; Q4_K at
other k, and batch 9 and above, the tensor-core kernels with it in the final
store or the finishing kernel; the rest a plain kernel followed by a small
epilogue kernel.
"""
import numpy as np
import pytest

import oracle
import quantized_weight_mat_gb300 as pq
from gpuio import dev, guard_intact, out_buf
from pqcases import tolerance_ok, weights, x_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup(cuda_ok):
    from quantized_weight_mat_gb300 import build
    build.build()
    import torch
    torch.cuda.init()


def run_swiglu(fmt, w, n_ff, k, x):
    import torch
    batch = x.shape[0]
    h = out_buf(batch * n_ff)
    pq.pq_gemv_swiglu(fmt, dev(w), n_ff, k, dev(x), batch, h)
    torch.cuda.synchronize()
    assert guard_intact(h, batch * n_ff)
    return h[: batch * n_ff].cpu().numpy().reshape(batch, n_ff)


def run_bias(fmt, w, n_out, k, x, bias):
    import torch
    batch = x.shape[0]
    y = out_buf(batch * n_out)
    pq.pq_gemv_bias(fmt, dev(w), n_out, k, dev(x), batch, dev(bias), y)
    torch.cuda.synchronize()
    assert guard_intact(y, batch * n_out)
    return y[: batch * n_out].cpu().numpy().reshape(batch, n_out)


def bias_for(n_out, seed):
    return np.random.default_rng(seed).normal(0.0, 0.5, n_out).astype(np.float32)


SW_SHAPES = [(300, 2048), (1000, 4096), (37, 14336), (129, 768)]
FMTS = ["q4_k", "q6_k", "q8_0", "i8_row"]


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8, 16, 17])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_ff,k", SW_SHAPES)
def test_swiglu_parity(n_ff, k, fmt, batch):
    kind = "quantized" if n_ff % 2 == 0 else "random"
    w = weights(fmt, 2 * n_ff, k, kind, 900 + n_ff)
    x = x_for(batch, k, 901 + batch)
    got = run_swiglu(fmt, w, n_ff, k, x)
    ok, err, bound = tolerance_ok(got, oracle.gemv_swiglu(fmt, w, n_ff, k, x))
    assert ok, f"max err {err:.3g} > {bound:.3g}"


@pytest.mark.parametrize("batch", [1, 2, 4, 5, 8, 16, 17])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_out,k", [(300, 2048), (129, 14336), (1000, 4096)])
def test_bias_parity(n_out, k, fmt, batch):
    kind = "quantized" if n_out % 2 == 0 else "random"
    w = weights(fmt, n_out, k, kind, 910 + n_out)
    x = x_for(batch, k, 911 + batch)
    b = bias_for(n_out, 912)
    got = run_bias(fmt, w, n_out, k, x, b)
    ok, err, bound = tolerance_ok(got, oracle.gemv_bias(fmt, w, n_out, k, x, b))
    assert ok, f"max err {err:.3g} > {bound:.3g}"


@pytest.mark.parametrize("batch", [2, 3, 5, 8])
@pytest.mark.parametrize("fmt", ["q4_k", "q6_k"])
def test_swiglu_stage_groups(fmt, batch):
    # 3500 pairs at k = 4096: 23 pairs per CTA, so three stages of 8, 8 and 7
    # pairs; the Q4_K kernel adds the partial sums of two stages after one
    # barrier, which leaves a group of one stage at the end
    n_ff, k = 3500, 4096
    w = weights(fmt, 2 * n_ff, k, "quantized", 36)
    x = x_for(batch, k, 37)
    got = run_swiglu(fmt, w, n_ff, k, x)
    ok, err, bound = tolerance_ok(got, oracle.gemv_swiglu(fmt, w, n_ff, k, x))
    assert ok, f"max err {err:.3g} > {bound:.3g}"


@pytest.mark.parametrize("batch", [1, 8])
def test_swiglu_gate_up_workload(batch):
    # the fused gate+up matrix of the 8B-shaped layer: 2 x 14336 rows, k = 4096
    n_ff, k = 14336, 4096
    w = weights("q4_k", 2 * n_ff, k, "quantized", 34)
    x = x_for(batch, k, 35)
    got = run_swiglu("q4_k", w, n_ff, k, x)
    ok, err, bound = tolerance_ok(got, oracle.gemv_swiglu("q4_k", w, n_ff, k, x))
    assert ok, f"max err {err:.3g} > {bound:.3g}"


@pytest.mark.parametrize("batch", [1, 8])
def test_bias_qkv_workload(batch):
    # the QKV projection of the same layer: 6144 x 4096 with a bias
    n_out, k = 6144, 4096
    w = weights("q4_k", n_out, k, "quantized", 30)
    x = x_for(batch, k, 31)
    b = bias_for(n_out, 32)
    got = run_bias("q4_k", w, n_out, k, x, b)
    ok, err, bound = tolerance_ok(got, oracle.gemv_bias("q4_k", w, n_out, k, x, b))
    assert ok, f"max err {err:.3g} > {bound:.3g}"


@pytest.mark.parametrize("prefetch", [False, True])
@pytest.mark.parametrize("batch", [1, 8])
def test_mlp_chain_respects_stream_order(batch, prefetch):
    # h = SwiGLU(W_gu x) feeds y = W_down h, and y feeds the next SwiGLU, three
    # times back to back on one stream: each call must read its predecessor's
    # finished output, also when it is scheduled while that one still runs
    import torch
    n_ff, k = 2048, 1024
    wgu = weights("q4_k", 2 * n_ff, k, "quantized", 80)
    wdn = weights("q4_k", k, n_ff, "quantized", 81)
    x = x_for(batch, k, 82)
    dgu, ddn = dev(wgu), dev(wdn)
    hs = [torch.empty(batch * n_ff, dtype=torch.float32, device="cuda") for _ in range(3)]
    ys = [torch.empty(batch * k, dtype=torch.float32, device="cuda") for _ in range(3)]
    old = pq.pq_set_weight_prefetch(prefetch)
    try:
        cur = dev(x)
        for i in range(3):
            pq.pq_gemv_swiglu("q4_k", dgu, n_ff, k, cur, batch, hs[i])
            pq.pq_gemv("q4_k", ddn, k, n_ff, hs[i], batch, ys[i])
            cur = ys[i]
        torch.cuda.synchronize()
    finally:
        pq.pq_set_weight_prefetch(bool(old))
    prev = x
    for i in range(3):
        h = hs[i].cpu().numpy().reshape(batch, n_ff)
        ok, err, bound = tolerance_ok(h, oracle.gemv_swiglu("q4_k", wgu, n_ff, k, prev))
        assert ok, (i, "swiglu", err, bound)
        y = ys[i].cpu().numpy().reshape(batch, k)
        ok, err, bound = tolerance_ok(y, oracle.gemv("q4_k", wdn, k, n_ff, h))
        assert ok, (i, "down", err, bound)
        prev = y


def test_epilogues_deterministic():
    import torch
    n_ff, k = 1000, 4096
    w = dev(weights("q4_k", 2 * n_ff, k, "random", 5))
    x = dev(x_for(8, k, 6))
    outs = []
    for batch in (1, 8):
        for _ in range(2):
            h = torch.empty(batch * n_ff, dtype=torch.float32, device="cuda")
            pq.pq_gemv_swiglu("q4_k", w, n_ff, k, x, batch, h)
            outs.append((batch, h.cpu().numpy()))
    torch.cuda.synchronize()
    for i in range(0, len(outs), 2):
        assert np.array_equal(outs[i][1].view(np.uint32), outs[i + 1][1].view(np.uint32))


def test_epilogue_argument_errors_launch_nothing():
    import torch
    n_ff, k = 64, 256
    w = dev(weights("q4_k", 2 * n_ff, k, "random", 1))
    x = torch.zeros(k, dtype=torch.float32, device="cuda")
    h = out_buf(n_ff)
    assert pq.pq_gemv_swiglu("q4_k", w, n_ff, k, x, 1, w.data_ptr() + 16, check=False) == pq.PQ_ERR_ARG
    assert pq.pq_gemv_swiglu("q4_k", w, 0, k, x, 1, h, check=False) == pq.PQ_ERR_ARG
    assert pq.pq_gemv_swiglu("q4_k", w, n_ff, 255, x, 1, h, check=False) == pq.PQ_ERR_K
    assert pq.pq_gemv_bias("q4_k", w, 2 * n_ff, k, x, 1, None, h, check=False) == pq.PQ_ERR_ARG
    bias = torch.zeros(2 * n_ff + 1, dtype=torch.float32, device="cuda")
    assert pq.pq_gemv_bias("q4_k", w, 2 * n_ff, k, x, 1, bias.data_ptr() + 2, h, check=False) == pq.PQ_ERR_ALIGN
    torch.cuda.synchronize()
    assert guard_intact(h, 0)

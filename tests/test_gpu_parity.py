"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Dequant must be bit-exact; the mat-vec must satisfy
max|y_gpu - y_ref| <= 2e-3 * RMS(y_ref) + 1e-6 (RMS over all outputs of the call).
Every output buffer carries a guard band that must stay untouched.
"""
import numpy as np
import pytest

import oracle
import quantized_weight_mat_gb300 as pq
from gpuio import dev, guard_intact, out_buf, run_gemv
from pqcases import tolerance_ok, weights, x_for

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def setup(cuda_ok):
    from quantized_weight_mat_gb300 import build
    build.build()
    import torch
    torch.cuda.init()


# ------------------------------------------------------------------ dequant

DQ_CASES = [
    ("q8_0", 1, 32), ("q8_0", 7, 96), ("q8_0", 129, 896), ("q8_0", 300, 4096),
    ("q4_k", 1, 256), ("q4_k", 7, 768), ("q4_k", 129, 4096), ("q4_k", 37, 14336),
    ("q6_k", 1, 256), ("q6_k", 7, 768), ("q6_k", 129, 4096), ("q6_k", 9, 14336),
    ("i8_row", 1, 1), ("i8_row", 7, 13), ("i8_row", 129, 100), ("i8_row", 33, 4096),
    ("q5_k", 1, 256), ("q5_k", 7, 768), ("q5_k", 129, 4096), ("q5_k", 9, 14336),
    ("q3_k", 1, 256), ("q3_k", 7, 768), ("q3_k", 129, 4096), ("q3_k", 9, 14336),
    ("q2_k", 1, 256), ("q2_k", 7, 768), ("q2_k", 129, 4096), ("q2_k", 9, 14336),
    ("i4_row", 1, 2), ("i4_row", 7, 14), ("i4_row", 129, 100), ("i4_row", 33, 4096),
]
# formats the oracle can quantize; the others (Q5_K, Q3_K, Q2_K) are tested on
# random records, which hold every bit pattern of every field
QUANTIZABLE = {"q8_0", "q4_k", "q6_k", "i8_row", "i4_row"}
DQ_PARAMS = [(f, n, k, kind) for (f, n, k) in DQ_CASES
             for kind in (("quantized", "random") if f in QUANTIZABLE else ("random",))]


@pytest.mark.parametrize("fmt,n_out,k,kind", DQ_PARAMS)
def test_dequant_bit_exact(fmt, n_out, k, kind):
    import torch
    w = weights(fmt, n_out, k, kind, 100 + n_out)
    ref = oracle.dequant(fmt, w, n_out, k)
    out = out_buf(n_out * k)
    pq.pq_dequant(fmt, dev(w), n_out, k, out)
    torch.cuda.synchronize()
    got = out[: n_out * k].cpu().numpy().reshape(n_out, k)
    assert guard_intact(out, n_out * k)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ mat-vec, small shapes

GEMV_SHAPES = {
    "q8_0": [(1, 32), (7, 96), (129, 896), (300, 4096), (1000, 768)],
    "q4_k": [(1, 256), (7, 768), (129, 4096), (300, 2048), (37, 14336), (1000, 8192), (333, 6144)],
    "q6_k": [(1, 256), (7, 768), (129, 4096), (300, 2048), (9, 14336), (1000, 4096), (2001, 2048)],
    "i8_row": [(1, 1), (7, 13), (129, 100), (300, 4096), (33, 2048), (1000, 768)],
    "q5_k": [(1, 256), (7, 768), (129, 4096), (9, 14336), (1000, 4096)],
    "q3_k": [(1, 256), (7, 768), (129, 4096), (9, 14336), (1000, 2048)],
    "q2_k": [(1, 256), (7, 768), (129, 4096), (9, 14336), (1000, 1024)],
    "i4_row": [(1, 2), (7, 14), (129, 100), (300, 4096), (33, 2048), (1000, 768)],
}
CASES = [(f, n, k) for f, shapes in GEMV_SHAPES.items() for (n, k) in shapes]


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8, 16, 17, 24, 32, 33, 40])
@pytest.mark.parametrize("kernel", ["auto", "generic", "stream", "tc"])
@pytest.mark.parametrize("fmt,n_out,k", CASES)
def test_gemv_parity(fmt, n_out, k, kernel, batch):
    kind = "random" if n_out % 2 or fmt not in QUANTIZABLE else "quantized"
    w = weights(fmt, n_out, k, kind, 200 + n_out)
    x = x_for(batch, k, 300 + batch)
    y = run_gemv(fmt, w, n_out, k, x, kernel)
    if y is None:
        assert kernel in ("stream", "tc"), "generic and auto take every case"
        pytest.skip(f"{kernel} kernel does not take this case")
    ref = oracle.gemv(fmt, w, n_out, k, x)
    ok, err, bound = tolerance_ok(y, ref)
    assert ok, f"max err {err:.3g} > {bound:.3g}"


@pytest.mark.parametrize("fmt,n_out,k,batch", [("q4_k", 4096, 4096, 1), ("q6_k", 1000, 4096, 2),
                                               ("q4_k", 4096, 4096, 16), ("q8_0", 896, 896, 1),
                                               ("q5_k", 1000, 4096, 3), ("q2_k", 700, 2048, 5)])
def test_gemv_deterministic(fmt, n_out, k, batch):
    import torch
    w = weights(fmt, n_out, k, "random", 7)
    x = x_for(batch, k, 8)
    wd, xd = dev(w), dev(x)
    ys = []
    for _ in range(3):
        y = torch.empty(batch * n_out, dtype=torch.float32, device="cuda")
        pq.pq_gemv(fmt, wd, n_out, k, xd, batch, y)
        ys.append(y.cpu().numpy())
    torch.cuda.synchronize()
    assert all(np.array_equal(ys[0].view(np.uint32), v.view(np.uint32)) for v in ys[1:])


def test_gemv_one_hot_x_gives_the_column():
    # one-hot x: the exact result is one decoded column; the dot product has a
    # single nonzero term, so every kernel must return it exactly
    fmt, n_out, k = "q4_k", 513, 4096
    w = weights(fmt, n_out, k, "quantized", 11)
    W = oracle.dequant(fmt, w, n_out, k)
    x = np.zeros((4, k), dtype=np.float32)
    for b, col in enumerate((0, 255, 2049, 4095)):
        x[b, col] = 1.0
    for kernel in ("generic", "stream", "auto"):
        y = run_gemv(fmt, w, n_out, k, x, kernel)
        if y is None:
            continue
        for b, col in enumerate((0, 255, 2049, 4095)):
            np.testing.assert_allclose(y[b], W[:, col], rtol=0, atol=1e-7 * np.abs(W).max())


def test_errors_on_device_launch_nothing():
    import torch
    w = dev(weights("q4_k", 8, 256, "random", 1))
    x = torch.zeros(256 + 4, dtype=torch.float32, device="cuda")
    y = out_buf(8)
    assert pq.pq_gemv("q4_k", w, 8, 256, x[1:].data_ptr(), 1, y, check=False) == pq.PQ_ERR_ALIGN
    assert pq.pq_gemv("q4_k", w, 8, 255, x, 1, y, check=False) == pq.PQ_ERR_K
    assert pq.pq_gemv("q4_k", w, 8, 256, x, 1, w.data_ptr() + 16, check=False) == pq.PQ_ERR_ARG
    torch.cuda.synchronize()
    assert guard_intact(y, 0)     # nothing written anywhere in y


# ------------------------------------------------------------------ workload-sized cases

def full_case(fmt, n_out, k, batch, wseed, xseed, kind="quantized"):
    w = weights(fmt, n_out, k, kind, wseed)
    x = x_for(batch, k, xseed)
    y = run_gemv(fmt, w, n_out, k, x, "auto")
    ref = oracle.gemv(fmt, w, n_out, k, x)
    ok, err, bound = tolerance_ok(y, ref)
    assert ok, f"{fmt} {n_out}x{k} b{batch}: max err {err:.3g} > {bound:.3g}"
    return err / bound


def test_workload_q8_0_896():
    full_case("q8_0", 896, 896, 1, 0, 1)


def test_workload_q4_k_4096():
    full_case("q4_k", 4096, 4096, 1, 20, 21)


@pytest.mark.parametrize("n_out,batch", [(7000, 5), (7000, 8), (6144, 8), (20000, 6), (2500, 7), (20000, 8),
                                         (7000, 3), (20000, 4), (2500, 2), (6144, 2)])
def test_register_operand_stage_groups(n_out, batch):
    # Q4_K at k = 4096 with 2-8 columns: the register-operand kernel adds the
    # partial sums of two 16-row stages after one barrier.  Rows per CTA give
    # odd stage counts with a partial last stage (7000: 46-47 rows, stages of
    # 16, 16 and 14-15; 20000: 131-132 rows, nine stages) and CTAs of one or
    # two stages (2500: 16-17 rows)
    full_case("q4_k", n_out, 4096, batch, 60, 61)


@pytest.mark.parametrize("batch", [2, 3])
def test_workload_gate_up_small_batch(batch):
    # 28672 x 4096: at batch 2 the two-column dp4a kernel (tall matrices), at
    # batch 3 the register-operand kernel
    full_case("q4_k", 28672, 4096, batch, 24, 25)


@pytest.mark.parametrize("j,n_out,k", [(0, 6144, 4096), (1, 4096, 4096), (2, 28672, 4096),
                                       (3, 4096, 14336)])
def test_workload_decode_layer_set(j, n_out, k):
    full_case("q4_k", n_out, k, 1, 30 + 2 * j, 31 + 2 * j)


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 8])
def test_workload_q6_k_output_head(batch):
    # batch 2-4: one pass over the 431 MB head for all columns; 8: two passes
    full_case("q6_k", 128256, 4096, batch, 40, 41)


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 6, 7, 8, 16])
@pytest.mark.parametrize("n_out,k,j", [(14336, 4096, 0), (4096, 14336, 1)])
def test_workload_small_batch(n_out, k, j, batch):
    full_case("q4_k", n_out, k, batch, 50 + 2 * j, 51 + 2 * j)


@pytest.mark.parametrize("batch", [32, 64])
@pytest.mark.parametrize("n_out,k,j", [(14336, 4096, 0), (4096, 14336, 1)])
def test_workload_prompt_width(n_out, k, j, batch):
    # 32-row prompt-width mat-vec (one tensor-core pass over W per 32 columns)
    full_case("q4_k", n_out, k, batch, 50 + 2 * j, 51 + 2 * j)


def test_workload_dequant_output_head_sampled():
    # the 2.1 GB f32 output of the 128256 x 4096 head, compared bit for bit on
    # a sample of rows (first, last, tails of every power-of-two tile size)
    import torch
    fmt, n_out, k = "q6_k", 128256, 4096
    w = weights(fmt, n_out, k, "quantized", 40)
    out = out_buf(n_out * k)
    pq.pq_dequant(fmt, dev(w), n_out, k, out)
    torch.cuda.synchronize()
    assert guard_intact(out, n_out * k)
    rows = sorted({0, 1, 127, 128, n_out - 257, n_out - 256, n_out - 2, n_out - 1,
                   *np.random.default_rng(0).integers(0, n_out, 64).tolist()})
    bb = 210 * (k // 256)
    o = out[: n_out * k].view(n_out, k)
    for r in rows:
        ref = oracle.dequant(fmt, w[r * bb:(r + 1) * bb], 1, k)[0]
        assert np.array_equal(o[r].cpu().numpy().view(np.uint32), ref.view(np.uint32)), r


@pytest.mark.parametrize("batch", [1, 2, 8])
@pytest.mark.parametrize("prefetch", [False, True])
def test_chained_calls_respect_stream_order(prefetch, batch):
    # y1 = W1 x, y2 = W2 y1, y3 = W3 y2 issued back to back on one stream: each
    # call must read its predecessor's finished output, also when its kernel is
    # scheduled while the predecessor is still running.  At batch 2 the long
    # rows (4096 x 14336) run the two-column kernel that converts x itself; at
    # batch 8 the three shapes run the register-operand kernel (k = 4096) and
    # the tensor-core item kernel with its finishing kernel (4096 x 14336).
    import torch
    shapes = [(14336, 4096), (4096, 14336), (4096, 4096)]
    ws = [weights("q4_k", n, k, "quantized", 60 + j) for j, (n, k) in enumerate(shapes)]
    wd = [dev(w) for w in ws]
    x = x_for(batch, shapes[0][1], 63)
    ys = [torch.empty(batch * n, dtype=torch.float32, device="cuda") for n, _ in shapes]
    old = pq.pq_set_weight_prefetch(prefetch)
    try:
        for rep in range(3):
            cur = dev(x)
            for j, (n, k) in enumerate(shapes):
                pq.pq_gemv("q4_k", wd[j], n, k, cur, batch, ys[j])
                cur = ys[j]
            torch.cuda.synchronize()
            prev = x
            for j, (n, k) in enumerate(shapes):
                got = ys[j].cpu().numpy().reshape(batch, n)
                ref = oracle.gemv("q4_k", ws[j], n, k, prev)
                ok, err, bound = tolerance_ok(got, ref)
                assert ok, (rep, j, err, bound)
                prev = got.astype(np.float32)
    finally:
        pq.pq_set_weight_prefetch(bool(old))


@pytest.mark.parametrize("prefetch", [False, True])
def test_chained_q6_k_calls_at_batch_2(prefetch):
    # the Q6_K two-column kernel converts x itself after the dependency wait
    # (and streams weights before it when they are declared static): a chain
    # whose every x is the previous call's y must still read finished outputs
    import torch
    shapes = [(4096, 2048), (2048, 4096), (1000, 2048)]
    ws = [weights("q6_k", n, k, "quantized", 80 + j) for j, (n, k) in enumerate(shapes)]
    wd = [dev(w) for w in ws]
    x = x_for(2, shapes[0][1], 83)
    ys = [torch.empty(2 * n, dtype=torch.float32, device="cuda") for n, _ in shapes]
    old = pq.pq_set_weight_prefetch(prefetch)
    try:
        for rep in range(3):
            cur = dev(x)
            for j, (n, k) in enumerate(shapes):
                pq.pq_gemv("q6_k", wd[j], n, k, cur, 2, ys[j])
                cur = ys[j]
            torch.cuda.synchronize()
            prev = x
            for j, (n, k) in enumerate(shapes):
                got = ys[j].cpu().numpy().reshape(2, n)
                ref = oracle.gemv("q6_k", ws[j], n, k, prev)
                ok, err, bound = tolerance_ok(got, ref)
                assert ok, (rep, j, err, bound)
                prev = got.astype(np.float32)
    finally:
        pq.pq_set_weight_prefetch(bool(old))


@pytest.mark.parametrize("batch", [1, 3, 6])
@pytest.mark.parametrize("n_out,k", [(896, 896), (129, 896), (7, 128), (1000, 1024), (33, 512)])
def test_q8_0_short_rows_with_static_weights(n_out, k, batch):
    # with the weights declared static, Q8_0 rows of at most 1024 run the
    # short-row kernel (weights read before the dependency wait)
    import torch
    w = weights("q8_0", n_out, k, "quantized", 90 + n_out)
    x = x_for(batch, k, 91 + batch)
    old = pq.pq_set_weight_prefetch(True)
    try:
        y = torch.empty(batch * n_out, dtype=torch.float32, device="cuda")
        pq.pq_gemv("q8_0", dev(w), n_out, k, dev(x), batch, y)
        torch.cuda.synchronize()
    finally:
        pq.pq_set_weight_prefetch(bool(old))
    ok, err, bound = tolerance_ok(y.cpu().numpy().reshape(batch, n_out), oracle.gemv("q8_0", w, n_out, k, x))
    assert ok, (err, bound)


def test_chained_q8_0_short_rows():
    # each call's x is the previous call's y; the short-row kernel may be
    # resident before its predecessor ends and must wait before reading x
    import torch
    n = k = 896
    ws = [weights("q8_0", n, k, "quantized", 95 + j) for j in range(4)]
    wd = [dev(w) for w in ws]
    x = x_for(1, k, 99)
    ys = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in ws]
    old = pq.pq_set_weight_prefetch(True)
    try:
        for rep in range(3):
            cur = dev(x)
            for j in range(len(ws)):
                pq.pq_gemv("q8_0", wd[j], n, k, cur, 1, ys[j])
                cur = ys[j]
            torch.cuda.synchronize()
            prev = x
            for j in range(len(ws)):
                got = ys[j].cpu().numpy().reshape(1, n)
                ok, err, bound = tolerance_ok(got, oracle.gemv("q8_0", ws[j], n, k, prev))
                assert ok, (rep, j, err, bound)
                prev = got.astype(np.float32)
    finally:
        pq.pq_set_weight_prefetch(bool(old))


@pytest.mark.parametrize("batch,k", [(1, 4096), (8, 4096), (2, 8192)])
def test_weights_written_by_the_preceding_kernel(batch, k):
    # with prefetch off (the default), a kernel that writes the weight buffer
    # right before pq_gemv must be fully visible to it (batch 8: the
    # register-operand kernel; batch 2 at k = 8192: the two-column kernel)
    import torch
    n = 2048
    wa, wb = weights("q4_k", n, k, "random", 70), weights("q4_k", n, k, "random", 71)
    da, db = dev(wa), dev(wb)
    mask = torch.bitwise_xor(da, db)
    wbuf = da.clone()
    x = x_for(batch, k, 72)
    xd = dev(x)
    y = torch.empty(batch * n, dtype=torch.float32, device="cuda")
    assert pq.pq_set_weight_prefetch(False) in (0, 1)
    for _ in range(3):
        torch.bitwise_xor(da, mask, out=wbuf)          # a kernel writes W = wb
        pq.pq_gemv("q4_k", wbuf, n, k, xd, batch, y)
        torch.bitwise_xor(db, mask, out=wbuf)          # and back to wa
        torch.cuda.synchronize()
        ok, err, bound = tolerance_ok(y.cpu().numpy().reshape(batch, n), oracle.gemv("q4_k", wb, n, k, x))
        assert ok, (err, bound)


def test_zz_no_bounded_wait_ran_out():
    # every barrier wait in the kernels is bounded; none may have expired
    assert pq.pq_wait_timeouts(reset=False) == 0

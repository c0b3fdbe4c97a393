"""GPU parity over the whole input domain, through the C ABI, against the oracle.

1. x of any finite magnitude: |x| up to 1e6 and 1e30, a column at 1e-30
   beside N(0, 1) columns, a single spike per column, and values near 3000
   on whole sub-blocks (sums of 32 values that an unscaled fp16 pair could
   not hold).  Every kernel that takes the case, and the automatic choice, at
   batch 1-16; checked column by column, each column against its own RMS.
2. Scale fields of every IEEE class (positive and negative normals,
   subnormals, signed zeros, infinities, NaNs): pq_dequant bit-exact with
   NaN compared as NaN; the mat-vec within the tolerance on every output
   whose reference is finite, and non-finite wherever the reference is.
"""
import numpy as np
import pytest

import oracle
import synth
from gpuio import run_dequant, run_gemv
from pqcases import tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup(cuda_ok):
    from quantized_weight_mat_gb300 import build
    build.build()
    import torch
    torch.cuda.init()


# ------------------------------------------------------------------ x range

def x_case(case: str, batch: int, k: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    x = g.normal(0.0, 1.0, (batch, k))
    if case == "large":                       # |x| up to 1e6
        x = g.uniform(-1e6, 1e6, (batch, k))
    elif case == "huge":
        x = x * 1e30
    elif case == "mixed":                     # 1e-30 column, a +-1e6 column, N(0,1) columns
        x[0] *= 1e-30
        if batch > 1:
            x[1] = g.uniform(-1e6, 1e6, k)
    elif case == "spike":                     # one large value per column on a small background
        x *= 1e-3
        for b in range(batch):
            x[b, g.integers(0, k)] = 5e4 * (b + 1)
    elif case == "subblock3000":              # whole 32-value runs near 3000
        for b in range(batch):
            for j in g.choice(k // 32, size=max(1, k // 256), replace=False):
                x[b, 32 * j:32 * j + 32] = g.uniform(2900.0, 3100.0, 32) * g.choice([-1, 1])
    else:
        raise ValueError(case)
    return x.astype(np.float32)


def columns_ok(y, ref):
    """Each column within 2e-3 * RMS(column) + 1e-6, and finite."""
    assert np.all(np.isfinite(y))
    for b in range(ref.shape[0]):
        ok, err, bound = tolerance_ok(y[b], ref[b])
        assert ok, f"column {b}: max err {err:.3g} > {bound:.3g}"


X_CASES = ["large", "huge", "mixed", "spike", "subblock3000"]


@pytest.mark.parametrize("case", X_CASES)
@pytest.mark.parametrize("batch", [1, 2, 4, 5, 8, 16])
@pytest.mark.parametrize("kernel", ["auto", "tc", "stream", "generic"])
@pytest.mark.parametrize("n_out,k", [(300, 2048), (1000, 4096)])
def test_gemv_x_range_q4_k(n_out, k, kernel, batch, case):
    w = synth.random_records("q4_k", n_out, k, seed=400 + n_out)
    x = x_case(case, batch, k, seed=500 + batch)
    y = run_gemv("q4_k", w, n_out, k, x, kernel)
    if y is None:
        pytest.skip(f"{kernel} kernel does not take this case")
    columns_ok(y, oracle.gemv("q4_k", w, n_out, k, x))


@pytest.mark.parametrize("case", X_CASES)
@pytest.mark.parametrize("fmt,batch", [("q8_0", 1), ("q6_k", 1), ("q6_k", 3), ("i8_row", 2), ("q5_k", 1),
                                       ("q3_k", 2), ("q2_k", 1), ("i4_row", 1)])
def test_gemv_x_range_other_formats(fmt, batch, case):
    n_out, k = 257, 4096
    w = synth.random_records(fmt, n_out, k, seed=410)
    x = x_case(case, batch, k, seed=510 + batch)
    y = run_gemv(fmt, w, n_out, k, x, "auto")
    columns_ok(y, oracle.gemv(fmt, w, n_out, k, x))


def test_gemv_x_range_full_size_tc():
    # the 14336 x 4096 shape at batch 8 (whole tiles) and 4096 x 14336 at
    # batch 16 (split-K with the finishing kernel), wide-range x
    for (n_out, k, batch) in ((14336, 4096, 8), (4096, 14336, 16)):
        w = synth.random_records("q4_k", n_out, k, seed=420)
        x = x_case("mixed", batch, k, seed=520)
        x[2:] *= (10.0 ** np.linspace(-20, 20, batch - 2))[:, None].astype(np.float32)
        y = run_gemv("q4_k", w, n_out, k, x, "auto")
        columns_ok(y, oracle.gemv("q4_k", w, n_out, k, x))


# ------------------------------------------------------------------ scale fields of every IEEE class

FMTS = ["q8_0", "q4_k", "q6_k", "i8_row", "q5_k", "q3_k", "q2_k", "i4_row"]


def same_or_both_nan(a: np.ndarray, b: np.ndarray) -> bool:
    both_nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(both_nan | (a.view(np.uint32) == b.view(np.uint32))))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_out,k", [(7, 768), (129, 4096)])
def test_dequant_ieee_scale_classes(fmt, n_out, k):
    per_row = fmt in ("i8_row", "i4_row")          # one scale per row: more of them non-finite
    w = synth.special_scale_records(fmt, n_out, k, seed=600 + n_out, nonfinite=0.6 if per_row else 0.15)
    ref = oracle.dequant(fmt, w, n_out, k)
    got = run_dequant(fmt, w, n_out, k)
    assert np.isnan(ref).any() and np.isinf(ref).any()          # the classes really occur
    assert same_or_both_nan(got, ref)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch,kernel", [(1, "auto"), (2, "auto"), (4, "auto"), (8, "auto"), (16, "auto"),
                                          (1, "generic"), (1, "stream"), (3, "stream"), (8, "tc")])
def test_gemv_ieee_scale_classes(fmt, batch, kernel):
    n_out, k = 517, 4096
    blocks = k // (32 if fmt == "q8_0" else 256 if fmt not in ("i8_row", "i4_row") else k)
    # about one row in ten reaches a non-finite scale field
    w = synth.special_scale_records(fmt, n_out, k, seed=610, nonfinite=0.05 / blocks)
    x = x_case("large", batch, k, seed=611) * np.float32(1e-6)   # N(0,1)-sized, uniform
    y = run_gemv(fmt, w, n_out, k, x, kernel)
    if y is None:
        pytest.skip(f"{kernel} kernel does not take this case")
    ref = oracle.gemv(fmt, w, n_out, k, x)
    fin = np.isfinite(ref)
    assert 0 < (~fin).sum() < fin.sum()
    assert not np.any(np.isfinite(y[~fin])), "non-finite reference, finite result"
    ok, err, bound = tolerance_ok(y[fin], ref[fin])
    assert ok, f"max err {err:.3g} > {bound:.3g} over the finite outputs"

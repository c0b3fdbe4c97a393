"""Pins for the oracle's decode-layer epilogues: silu, SwiGLU on a fused
gate+up matrix, and the bias add (the PESTI README, "Conformance": the MLP
multiplies the sigmoid-based silu of the gate projection by the up
projection, and the QKV projections carry a bias).

silu is tied to closed forms (silu(0) = 0; sigmoid(+-ln 3) = 3/4, 1/4), to the
identity silu(z) - silu(-z) = z, and to its two tails; the epilogues to
integer-valued matrices where every term is known exactly, so that a swapped
gate/up order, a wrong row pairing or a dropped bias fails.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def q8_0_integer_matrix(codes: np.ndarray) -> np.ndarray:
    """Q8_0 records with d = 1: the decoded matrix is `codes` exactly."""
    n, k = codes.shape
    rec = np.zeros((n * k // 32, 34), dtype=np.uint8)
    rec[:, 0:2] = np.array([1.0], dtype="<f2").view(np.uint8)
    rec[:, 2:] = codes.reshape(-1, 32).astype(np.int8).view(np.uint8)
    return rec.ravel()


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    l3 = math.log(3.0)
    assert oracle.silu(l3) == pytest.approx(0.75 * l3, rel=1e-15)
    assert oracle.silu(-l3) == pytest.approx(-0.25 * l3, rel=1e-15)


def test_silu_odd_part_identity_and_tails():
    for z in np.linspace(-40, 40, 801):
        assert oracle.silu(z) - oracle.silu(-z) == pytest.approx(z, rel=1e-14, abs=1e-14)
    assert oracle.silu(60.0) == 60.0                       # e^-60 is below the last bit
    assert -1e-23 < oracle.silu(-60.0) < 0.0               # -60 e^-60 ~ -5e-25
    assert oracle.silu(-800.0) == 0.0 or abs(oracle.silu(-800.0)) < 1e-300   # no overflow
    assert oracle.silu(1e-9) / 1e-9 == pytest.approx(0.5, rel=1e-8)          # slope 1/2 at 0


def test_swiglu_pairs_gate_row_j_with_up_row_n_ff_plus_j():
    n_ff, k = 3, 64
    g = np.random.default_rng(70)
    codes = g.integers(-5, 6, size=(2 * n_ff, k))
    w = q8_0_integer_matrix(codes)
    for i in (0, 17, 63):
        x = np.zeros((1, k), dtype=np.float32)
        x[0, i] = 1.0
        h = oracle.gemv_swiglu("q8_0", w, n_ff, k, x)[0]
        for j in range(n_ff):
            gate, up = float(codes[j, i]), float(codes[n_ff + j, i])
            assert h[j] == oracle.silu(gate) * up, (i, j)


def test_swiglu_general_x_against_its_parts():
    n_ff, k, batch = 5, 256, 3
    w = synth.random_records("q4_k", 2 * n_ff, k, seed=71)
    x = synth.normal_x(batch, k, seed=72)
    y = oracle.gemv("q4_k", w, 2 * n_ff, k, x)
    h = oracle.gemv_swiglu("q4_k", w, n_ff, k, x)
    for b in range(batch):
        for j in range(n_ff):
            assert h[b, j] == oracle.silu(y[b, j]) * y[b, n_ff + j]


def test_bias_is_added_once_per_output():
    n_out, k, batch = 4, 64, 2
    codes = np.zeros((n_out, k), dtype=np.int64)
    w = q8_0_integer_matrix(codes)
    bias = np.array([0.5, -1.25, 3.0, 0.0], dtype=np.float32)
    x = synth.normal_x(batch, k, seed=73)
    y = oracle.gemv_bias("q8_0", w, n_out, k, x, bias)
    assert np.array_equal(y, np.tile(bias.astype(np.float64), (batch, 1)))   # zero weights: y = bias
    codes = np.random.default_rng(74).integers(-3, 4, size=(n_out, k))
    w = q8_0_integer_matrix(codes)
    xi = np.random.default_rng(75).integers(-4, 5, size=(batch, k)).astype(np.float32)
    y = oracle.gemv_bias("q8_0", w, n_out, k, xi, bias)
    want = (xi.astype(np.float64) @ codes.T.astype(np.float64)) + bias.astype(np.float64)
    assert np.array_equal(y, want)                          # integer sums: exact

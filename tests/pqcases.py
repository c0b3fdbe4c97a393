"""Seeded parity cases shared by the GPU tests.

Weights come from the oracle's quantizers (N(0, 0.02) weights, as the
workloads specify) or from ``synth.random_records`` (every bit pattern of the
packed fields); x ~ N(0, 1).  Expected values come from the oracle only.
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
import synth

TOL_REL = 2e-3      # max|y_gpu - y_ref| <= TOL_REL * RMS(y_ref) + TOL_ABS
TOL_ABS = 1e-6


@functools.lru_cache(maxsize=16)
def weights(fmt: str, n_out: int, k: int, kind: str, seed: int) -> np.ndarray:
    if kind == "quantized":
        if fmt == "q8_0" and seed == 0 and (n_out, k) == (896, 896):
            return synth.q8_0_random(n_out, k, seed=0)
        return oracle.quantize(fmt, synth.normal_weights(n_out, k, seed))
    if kind == "random":
        return synth.random_records(fmt, n_out, k, seed)
    raise ValueError(kind)


def x_for(batch: int, k: int, seed: int) -> np.ndarray:
    return synth.normal_x(batch, k, seed)


def tolerance_ok(y_gpu: np.ndarray, y_ref: np.ndarray, rms: float | None = None):
    """The parity bar for the mat-vec: returns (ok, max_err, bound)."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    err = float(np.max(np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref))) if y_ref.size else 0.0
    bound = TOL_REL * rms + TOL_ABS
    return err <= bound, err, bound

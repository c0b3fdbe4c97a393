"""The library's Q5_K / Q3_K / Q2_K lane decoders, built for the host, against the oracle.

The decoders in ``csrc/pq_kfamily.cuh`` are ``__host__ __device__`` templates
over a byte loader; the kernels run them on the GPU.  Here the same source is
compiled with g++ (``tests/kfamily_host.cpp``) and every one of the 256
weights of each block must match the oracle's decode bit for bit: random
records, blocks of fully random bytes (every fp16 class, incl. subnormals,
inf and NaN in the scale fields) and all-zero / all-one blocks.  The GPU
parity tests check the device build of the same functions.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "quantized_weight_mat_gb300", "csrc")


@pytest.fixture(scope="module")
def host_lib(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    out = str(tmp_path_factory.mktemp("kfhost") / "kfamily_host.so")
    subprocess.run(["g++", "-O2", "-ffp-contract=off", "-std=c++17", "-fPIC", "-shared",
                    "-Wno-unknown-pragmas", "-I", CSRC, "-o", out,
                    os.path.join(HERE, "kfamily_host.cpp")], check=True)
    L = ctypes.CDLL(out)
    L.kf_host_decode.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    L.kf_host_decode.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("fmt", ["q5_k", "q3_k", "q2_k"])
def test_lane_decoders_match_the_oracle(host_lib, fmt):
    code = oracle.FORMATS[fmt]
    bb = synth.BLOCK[fmt][1]
    n = 1500
    blocks = np.concatenate([
        synth.random_records(fmt, n, 256, seed=51).reshape(n, bb),
        np.random.default_rng(52).integers(0, 256, (500, bb), dtype=np.uint8),
        np.zeros((1, bb), np.uint8), np.full((1, bb), 255, np.uint8)])
    out = np.empty(256, np.float32)
    for i, blk in enumerate(blocks):
        blk = np.ascontiguousarray(blk)
        assert host_lib.kf_host_decode(code, blk.ctypes.data, out.ctypes.data) == 0
        ref = oracle.decode_block(fmt, blk)
        same = (ref.view(np.uint32) == out.view(np.uint32)) | (np.isnan(ref) & np.isnan(out))
        assert same.all(), (fmt, i, np.nonzero(~same)[0][:8])

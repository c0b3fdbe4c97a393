"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a GPU."""
import os
import re

import pytest

import oracle
import quantized_weight_mat_gb300 as pq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_weight_mat_gb300 import build
    build.build()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"pq_gemv", "pq_dequant", "pq_weight_bytes", "pq_strerror"} <= set(names)
    lib = pq.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pq.EXPORTS)


def test_weight_bytes_agree_with_oracle():
    for fmt in ("q8_0", "q4_k", "q6_k", "i8_row", "q5_k", "q3_k", "q2_k", "i4_row"):
        for n_out, k in [(1, 256), (7, 512), (896, 896 if fmt in ("q8_0", "i8_row") else 1024),
                         (128256, 4096)]:
            assert pq.pq_weight_bytes(fmt, n_out, k) == oracle.weight_bytes(fmt, n_out, k)
    assert pq.pq_weight_bytes("q4_k", 4, 100) == 0
    assert pq.pq_weight_bytes(8, 4, 256) == 0
    assert pq.pq_weight_bytes("i4_row", 4, 7) == 0                # odd k
    assert pq.pq_weight_bytes("q4_k", 0, 256) == 0
    assert pq.pq_weight_bytes("q4_k", 1 << 30, 1 << 30) == 0     # overflow guard


def test_strerror_covers_every_code():
    for st in range(0, -9, -1):
        s = pq.pq_strerror(st)
        assert s and s != "unknown status"
    assert pq.pq_strerror(-99) == "unknown status"


A16 = 1 << 20        # a 16-byte aligned fake address (never dereferenced)


@pytest.mark.parametrize("args,status", [
    (("q4_k", A16, 4, 256, A16 * 2, 1, A16 * 3), pq.PQ_OK),
    ((9, A16, 4, 256, A16 * 2, 1, A16 * 3), pq.PQ_ERR_FMT),
    (("q4_k", 0, 4, 256, A16 * 2, 1, A16 * 3), pq.PQ_ERR_ARG),
    (("q4_k", A16, 4, 256, 0, 1, A16 * 3), pq.PQ_ERR_ARG),
    (("q4_k", A16, 4, 256, A16 * 2, 1, 0), pq.PQ_ERR_ARG),
    (("q4_k", A16, 0, 256, A16 * 2, 1, A16 * 3), pq.PQ_ERR_ARG),
    (("q4_k", A16, 4, 0, A16 * 2, 1, A16 * 3), pq.PQ_ERR_ARG),
    (("q4_k", A16, 4, 256, A16 * 2, 0, A16 * 3), pq.PQ_ERR_ARG),
    (("q4_k", A16, 4, 100, A16 * 2, 1, A16 * 3), pq.PQ_ERR_K),
    (("q8_0", A16, 4, 48, A16 * 2, 1, A16 * 3), pq.PQ_ERR_K),
    (("q5_k", A16, 4, 128, A16 * 2, 1, A16 * 3), pq.PQ_ERR_K),
    (("q2_k", A16, 4, 256, A16 * 2, 1, A16 * 3), pq.PQ_OK),
    (("q4_k", A16 + 8, 4, 256, A16 * 2, 1, A16 * 3), pq.PQ_ERR_ALIGN),
    (("q4_k", A16, 4, 256, A16 * 2 + 4, 1, A16 * 3), pq.PQ_ERR_ALIGN),
    (("q4_k", A16, 4, 256, A16 * 2, 1, A16 * 3 + 2), pq.PQ_ERR_ALIGN),
    (("q4_k", A16, 4, 256, A16 * 2, 1, A16 + 16), pq.PQ_ERR_ARG),       # y overlaps w
    (("q4_k", A16, 4, 256, A16 * 2, 1, A16 * 2 + 512), pq.PQ_ERR_ARG),  # y overlaps x
    (("q4_k", A16, 1 << 30, 1 << 20, A16 * 2, 1, A16 * 3), pq.PQ_ERR_SIZE),
])
def test_gemv_argument_checks(args, status):
    import torch
    st = pq.lib().pq_gemv(pq._fmt(args[0]), *args[1:], 0)
    if status == pq.PQ_OK:
        # valid arguments reach the device check; without a GPU that fails
        if torch.cuda.is_available():
            pytest.skip("would launch on a real GPU with fake pointers")
        assert st == pq.PQ_ERR_DEVICE
    else:
        assert st == status


def test_dequant_argument_checks():
    L = pq.lib()
    assert L.pq_dequant(1, A16, 4, 256, 0, 0) == pq.PQ_ERR_ARG
    assert L.pq_dequant(1, A16, 4, 256, A16 * 2 + 4, 0) == pq.PQ_ERR_ALIGN
    assert L.pq_dequant(1, A16, 4, 255, A16 * 2, 0) == pq.PQ_ERR_K
    assert L.pq_dequant(9, A16, 4, 256, A16 * 2, 0) == pq.PQ_ERR_FMT
    assert L.pq_dequant(pq.Q3_K, A16, 4, 200, A16 * 2, 0) == pq.PQ_ERR_K
    assert L.pq_dequant(1, A16, 4, 256, A16 + 32, 0) == pq.PQ_ERR_ARG   # out overlaps w


def test_kernel_choice_table():
    # pure host logic: which kernel and how many launches a call makes
    assert pq.pq_gemv_choice("q4_k", 4096, 4096, 0) == pq.PQ_ERR_ARG
    assert pq.pq_gemv_choice("q4_k", 4096, 100, 1) == pq.PQ_ERR_K
    for fmt, k in (("q4_k", 4096), ("q6_k", 4096), ("q8_0", 896), ("i8_row", 100)):
        for b in (1, 2, 3, 4, 8, 16, 17, 40):
            c = pq.pq_gemv_choice(fmt, 4096, k, b)
            assert c in (pq.KERNEL_GENERIC, pq.KERNEL_STREAM, pq.KERNEL_TC)
            n = pq.pq_gemv_launches(fmt, 4096, k, b)
            # slices of up to 32 (tensor core) or 4 columns, or one column at a
            # time for a one-column streaming kernel (Q8_0, per-row int8)
            assert (b + 31) // 32 <= n <= (b if fmt != "q4_k" else (b + 3) // 4)


def test_k_family_and_int4_rows_stream_one_column_at_a_time():
    # Q5_K, Q3_K, Q2_K and per-row int4 take the whole-row kernel, one launch
    # per column, when a row is a whole number of 16-byte units (Q3_K: k a
    # multiple of 2048, Q2_K of 1024); other k take the generic kernel, 4
    # columns a launch
    S, G = pq.KERNEL_STREAM, pq.KERNEL_GENERIC
    for fmt in ("q5_k", "q3_k", "q2_k", "i4_row"):
        for b in (1, 2, 4, 5, 16, 17):
            assert pq.pq_gemv_choice(fmt, 4096, 4096, b) == S
            assert pq.pq_gemv_launches(fmt, 4096, 4096, b) == b
    for fmt, k in (("q3_k", 1024), ("q2_k", 768), ("i4_row", 100)):
        for b in (1, 5):
            assert pq.pq_gemv_choice(fmt, 4096, k, b) == G
            assert pq.pq_gemv_launches(fmt, 4096, k, b) == (b + 3) // 4
    assert pq.pq_gemv_choice("q2_k", 4096, 100, 1) == pq.PQ_ERR_K
    assert pq.pq_gemv_choice("i4_row", 4096, 101, 1) == pq.PQ_ERR_K


def test_bad_kernel_id_rejected():
    assert pq.lib().pq_gemv_kernel(1, A16, 4, 256, A16 * 2, 1, A16 * 3, 0, 7) == pq.PQ_ERR_KERNEL


def test_noalloc_argument_checks():
    # the allocation-free entry checks as pq_gemv does, then its own limits
    L = pq.lib()
    assert L.pq_gemv_noalloc(1, 0, 4, 256, A16 * 2, 1, A16 * 3, 0) == pq.PQ_ERR_ARG
    assert L.pq_gemv_noalloc(1, A16 + 8, 4, 256, A16 * 2, 1, A16 * 3, 0) == pq.PQ_ERR_ALIGN
    assert L.pq_gemv_noalloc(0, A16, 4, 256, A16 * 2, 1, A16 * 3, 0) == pq.PQ_ERR_KERNEL   # Q8_0
    assert L.pq_gemv_noalloc(1, A16, 4, 16640, A16 * 2, 1, A16 * 3, 0) == pq.PQ_ERR_SIZE
    import torch
    if not torch.cuda.is_available():
        assert L.pq_gemv_noalloc(1, A16, 4, 16384, A16 * 2, 1, A16 * 3, 0) == pq.PQ_ERR_DEVICE


def test_selftest_limit_is_checked_before_any_launch():
    L = pq.lib()
    assert L.pq_selftest_wait_timeout(0, 0) == pq.PQ_ERR_ARG
    assert L.pq_selftest_wait_timeout(1000001, 0) == pq.PQ_ERR_ARG


def test_q4_k_dispatch_matches_the_measured_winners():
    # batch 1-4 winners measured on the decode-layer shapes (CUDA graph, GB300):
    # the streaming kernels up to the batch where the tensor-core kernel wins,
    # the tensor-core kernel from batch 5 on
    S, T = pq.KERNEL_STREAM, pq.KERNEL_TC
    # (at k = 4096 batch 3-8 is the register-operand whole-row kernel, a
    # streaming kernel: one pass over W for up to 8 columns)
    table = {
        (14336, 4096): [S, S, S, S, S, S, T],
        (4096, 14336): [S, S, T, T, T, T, T],
        (28672, 4096): [S, S, S, S, S, S, T],
        (6144, 4096): [S, S, S, S, S, S, T],
        (4096, 4096): [S, S, S, S, S, S, T],
    }
    for (n, k), want in table.items():
        got = [pq.pq_gemv_choice("q4_k", n, k, b) for b in (1, 2, 3, 4, 5, 8, 16)]
        assert got == want, (n, k, got)
    # prompt width: up to 32 columns in one tensor-core pass over W
    for b, launches in ((17, 1), (32, 1), (33, 2), (64, 2), (65, 3)):
        assert pq.pq_gemv_choice("q4_k", 14336, 4096, b) == T
        assert pq.pq_gemv_launches("q4_k", 14336, 4096, b) == launches
    # the Q6_K head streams W once per call for up to 8 columns, in passes of 8
    assert [pq.pq_gemv_choice("q6_k", 128256, 4096, b) for b in (1, 2, 3, 4, 8)] == [S] * 5
    for b, launches in ((1, 1), (2, 1), (3, 1), (4, 1), (5, 1), (8, 1), (16, 2), (17, 3)):
        assert pq.pq_gemv_launches("q6_k", 128256, 4096, b) == launches
    # Q4_K at k = 4096: batches 5-8 in one streaming pass too, 9-16 on the tensor-core kernel
    for b, launches in ((5, 1), (8, 1), (9, 1), (16, 1)):
        assert pq.pq_gemv_launches("q4_k", 14336, 4096, b) == launches
    # rows that are not whole 16-byte units (k not a multiple of 2048) take
    # the generic kernel
    assert pq.pq_gemv_choice("q6_k", 4096, 768, 2) == pq.KERNEL_GENERIC
    # so do Q8_0 and per-row int8 when k is a multiple of 256 (whole-row
    # kernel); other k take the generic kernel
    for fmt in ("q8_0", "i8_row"):
        assert [pq.pq_gemv_choice(fmt, 14336, 4096, b) for b in (1, 2, 4, 16)] == [S, S, S, S]
        assert pq.pq_gemv_launches(fmt, 14336, 4096, 4) == 4
        assert pq.pq_gemv_launches(fmt, 14336, 4096, 17) == 17
    assert pq.pq_gemv_choice("q8_0", 896, 896, 1) == pq.KERNEL_GENERIC
    assert pq.pq_gemv_choice("i8_row", 4096, 100, 1) == pq.KERNEL_GENERIC

"""The oracle against its stored golden decodes (tests/golden/decode_golden.txt).

The fixture is written by tests/golden/make_golden.py, which calls only the
oracle; the pages print no worked example to take values from.  A mismatch
means the oracle's decode arithmetic changed: such a change must be justified
by the layout it follows and the fixture rewritten by the script.
"""
import hashlib
import os

import numpy as np
import pytest

import oracle

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "decode_golden.txt")


def entries():
    with open(PATH) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            fmt, hexblk, digest, *head = ln.split()
            yield fmt, hexblk, digest, [float(v) for v in head]


@pytest.mark.parametrize("fmt,hexblk,digest,head", list(entries()))
def test_oracle_reproduces_the_golden_decode(fmt, hexblk, digest, head):
    blk = np.frombuffer(bytes.fromhex(hexblk), dtype=np.uint8).copy()
    w = oracle.decode_block(fmt, blk)
    assert hashlib.sha256(w.astype("<f4").tobytes()).hexdigest() == digest
    np.testing.assert_array_equal(w[:4], np.array(head, dtype=np.float32))


def test_every_block_format_is_covered():
    assert {e[0] for e in entries()} == {"q8_0", "q4_k", "q6_k", "q5_k", "q3_k", "q2_k"}

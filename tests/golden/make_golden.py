"""Write decode_golden.txt: decoded blocks of every format, from the oracle only.

The pages print no worked decode example, so these stored values are the
oracle's (oracle/pq_oracle.c), written by this script and nothing else: per
format, two seeded random records plus an all-zero and an all-0xFF block;
for each, the block bytes (hex), the sha256 of the decoded f32 values
(little-endian bits) and the first four values.  tests/test_golden.py checks
that the oracle still reproduces them, so a change to the oracle's arithmetic
cannot pass unnoticed.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402

BLOCK_FORMATS = ["q8_0", "q4_k", "q6_k", "q5_k", "q3_k", "q2_k"]


def blocks_for(fmt):
    qk, bb = synth.BLOCK[fmt]
    rec = synth.random_records(fmt, 2, qk, seed=900).reshape(2, bb)
    return [rec[0], rec[1], np.zeros(bb, np.uint8), np.full(bb, 255, np.uint8)]


def line(fmt, blk):
    w = oracle.decode_block(fmt, blk)
    digest = hashlib.sha256(w.astype("<f4").tobytes()).hexdigest()
    head = " ".join(f"{v:.9g}" for v in w[:4])
    return f"{fmt} {blk.tobytes().hex()} {digest} {head}"


def main():
    lines = ["# format block-hex sha256(decoded f32 LE) first-four-values; written by make_golden.py from the oracle"]
    for fmt in BLOCK_FORMATS:
        for blk in blocks_for(fmt):
            lines.append(line(fmt, np.ascontiguousarray(blk)))
    with open(os.path.join(HERE, "decode_golden.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()

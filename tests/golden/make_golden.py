"""Write tests/golden/tiny256_seed0.txt from the oracle alone.

The pages print no worked numeric example, so this fixture is a regression lock on the
oracle for the 256x256 workload (B=1, H=1, Nq=Nk=256, d=128, N(0,1) BF16 inputs from
seed 0, scale = 1/sqrt(128) in float32): every LSE value plus five full output rows,
together with a hash of the inputs that detects any drift in the input generator.
Run from the repository root: ``python tests/golden/make_golden.py``.
"""
import hashlib
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dense_attention_forward_fwd_gb300.inputs import make_qkv  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny256_seed0.txt")
ROWS = (0, 1, 127, 128, 255)


def input_digest(q, k, v) -> str:
    h = hashlib.sha256()
    for a in (q, k, v):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def main():
    q, k, v = make_qkv(1, 1, 256, 256, d=128, seed=0)
    scale = float(np.float32(1 / math.sqrt(128)))
    o, lse = oracle.attention(q, k, v, scale)
    with open(OUT, "w") as f:
        f.write("# oracle regression fixture: B=1 H=1 Nq=Nk=256 d=128 seed=0 N(0,1) BF16\n")
        f.write("# written by tests/golden/make_golden.py (calls only oracle/)\n")
        f.write(f"inputs_sha256 {input_digest(q, k, v)}\n")
        f.write(f"scale {scale!r}\n")
        f.write("lse " + " ".join(repr(float(x)) for x in lse[0, 0]) + "\n")
        for r in ROWS:
            f.write(f"o_row {r} " + " ".join(repr(float(x)) for x in o[0, 0, r]) + "\n")


if __name__ == "__main__":
    main()

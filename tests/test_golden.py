"""Regression fixture for the oracle on the 256x256 workload (see tests/golden/make_golden.py)."""
import math
import os

import numpy as np

import oracle
from dense_attention_forward_fwd_gb300.inputs import make_qkv

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny256_seed0.txt")


def load_golden():
    out = {"o_rows": {}}
    for line in open(GOLDEN):
        if line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "inputs_sha256":
            out["sha"] = vals[0]
        elif key == "scale":
            out["scale"] = float(vals[0])
        elif key == "lse":
            out["lse"] = np.array([float(x) for x in vals])
        elif key == "o_row":
            out["o_rows"][int(vals[0])] = np.array([float(x) for x in vals[1:]])
    return out


def test_inputs_are_unchanged():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(os.path.dirname(GOLDEN), "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    g = load_golden()
    q, k, v = make_qkv(1, 1, 256, 256, d=128, seed=0)
    assert mg.input_digest(q, k, v) == g["sha"]
    assert g["scale"] == float(np.float32(1 / math.sqrt(128)))


def test_oracle_matches_fixture():
    g = load_golden()
    q, k, v = make_qkv(1, 1, 256, 256, d=128, seed=0)
    o, lse = oracle.attention(q, k, v, g["scale"])
    assert np.max(np.abs(lse[0, 0] - g["lse"])) < 1e-12
    for r, row in g["o_rows"].items():
        assert np.max(np.abs(o[0, 0, r] - row)) < 1e-12

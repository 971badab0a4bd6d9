"""bench.py's output contract on a host without a GPU: the reference arm (the FP64 oracle on
the host cores) prints one JSON line with every key of the contract for each variant, the
flags that have no entry point together are refused, and the roofline arithmetic and
traffic keys are the documented ones."""
import dataclasses
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*flags):
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny-256", "--steps", "1", "--warmup", "1", *flags],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    return r


@pytest.mark.parametrize("flags", [(), ("--causal",), ("--bias", "shared"), ("--backward",), ("--fp8-qk",),
                                   ("--fp8",), ("--head-dim", "256", "--bias", "full"),
                                   ("--head-dim", "256", "--fp8-qk", "--causal")])
def test_reference_arm_prints_the_contract_line(flags):
    r = run_bench(*flags)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1 and d["gpu_launches"] == 0
    assert d["config"]["workload"] == "tiny-256"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    if "--fp8" in flags:
        assert d["config"]["qk"] == "e4m3" and d["config"]["pv"] == "e4m3"
    if "--backward" in flags:
        assert d["config"]["pass"] == "backward"


@pytest.mark.parametrize("flags", [("--mxfp8", "--bias", "full"), ("--fp8-qk", "--bias", "shared", "--causal"),
                                   ("--fp8", "--fp8-qk"),
                                   ("--bias", "full", "--causal"), ("--head-dim", "256", "--backward"),
                                   ("--head-dim", "256", "--mxfp8"),
                                   ("--fp8", "--backward")])
def test_flags_without_an_entry_point_are_refused(flags):
    r = run_bench(*flags)
    assert r.returncode == 2 and "error" in r.stderr


def test_roofline_peaks():
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"bf16_tflops": 1800.0}
    base = dict(fp8_qk=False, fp8=False, mxfp8=False)
    assert bench.roofline_peak(SimpleNamespace(**base), peaks, "measured")[0] == 1800.0
    assert bench.roofline_peak(SimpleNamespace(**dict(base, fp8_qk=True)), peaks, "measured")[0] == \
        pytest.approx(2400.0)   # 4P/3: Q K^T at 2P, P V at P
    assert bench.roofline_peak(SimpleNamespace(**dict(base, fp8=True)), peaks, "measured")[0] == 3600.0
    assert bench.roofline_peak(SimpleNamespace(**dict(base, mxfp8=True)), peaks, "measured")[0] == 3600.0


def test_traffic_keys_match_the_recorded_ones():
    sys.path.insert(0, ROOT)
    import bench
    from dense_attention_forward_fwd_gb300.configs import by_name
    base = dict(causal=False, bias="none", backward=False, fp8_qk=False, fp8=False, mxfp8=False)
    cases = {"rect-4k-8k": ("rect-4k-8k", {}), "long-16k": ("long-16k", {}), "peaked-8k": ("peaked-8k", {}),
             "square-4k": ("square-4k", {}), "long-16k-mxfp8": ("long-16k", {"mxfp8": True}),
             "rect-4k-8k-mxfp8": ("rect-4k-8k", {"mxfp8": True}), "rect-4k-8k-fp8qk": ("rect-4k-8k", {"fp8_qk": True}),
             "rect-4k-8k-fp8": ("rect-4k-8k", {"fp8": True}), "square-4k-causal": ("square-4k", {"causal": True}),
             "rect-4k-8k-bias-shared": ("rect-4k-8k", {"bias": "shared"}),
             "square-4k-backward": ("square-4k", {"backward": True}),
             "square-4k-bias-shared-backward": ("square-4k", {"bias": "shared", "backward": True}),
             "rect-4k-8k-bias-shared-fp8qk": ("rect-4k-8k", {"bias": "shared", "fp8_qk": True}),
             "square-4k-d256": ("square-4k", {"d": 256}),
             "square-4k-bias-shared-d256": ("square-4k", {"bias": "shared", "d": 256}),
             "square-4k-fp8qk-d256": ("square-4k", {"fp8_qk": True, "d": 256}),
             "square-4k-fp8-d256": ("square-4k", {"fp8": True, "d": 256})}
    recorded = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert set(recorded) <= set(cases)
    for key, (name, over) in cases.items():
        w = by_name(name)
        if "d" in over:
            w = dataclasses.replace(w, d=over.pop("d"))
        assert bench.traffic_key(w, SimpleNamespace(**dict(base, **over))) == key

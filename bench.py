#!/usr/bin/env python3
"""Benchmark of the dense BF16 attention forward (d=128; non-causal by default) on GB300.

One step = one attn_fwd call over the whole workload (every (b, h) and every query
tile). Default workload: long-16k, B=1, H=16, Nq=Nk=16384 (the largest of the 4K/8K/16K
sequence lengths that "Sıfırdan yazılan CUDA attention kerneli..." measures at, and the
largest of the five that fits one GPU); --workload picks another of the five (rect-4k-8k
is the shape of the RTX 5090 table in "Flash Attention на 5090 в CUDA C++").

Kernel time: CUDA events around each launch on the launching stream, inputs resident
in HBM, L2 flushed (a 512 MiB write) before every timed launch. value = total
4*B*H*Nq*Nk*d FLOPs of all ranks / max-over-ranks time. e2e: the same metric through
the same C-ABI call, with the host->device copy of Q, K, V from pinned memory and the
device->host copy of O and LSE inside each timed step; steps are pipelined over three
streams (copy in, compute, copy out) with two device buffer sets, so one step's copies
overlap its neighbours' kernels.

--causal times attn_fwd_causal instead (query i sees keys 0 .. i + Nk - Nq); its FLOPs
count the visible (query, key) pairs only, 4*d each, and vs_baseline is null.

--bias shared|full times attn_fwd_bias with a BF16 N(0,1) bias, one [Nq, Nk] matrix for
every head or one per head; the FLOP count is unchanged (the bias adds one addend per
score).

--backward times attn_bwd (dQ, dK, dV for an N(0,1) upstream gradient, given the forward's
O and LSE) and counts 2.5x the forward's FLOPs (the five products of the method's
backward); with --impl reference it times the FP64 backward oracle.

--fp8-qk times attn_fwd_fp8qk: Q and K quantized per tensor to FP8 E4M3 codes (descale =
amax / 448), V in BF16; the FLOP count is unchanged and the roofline peak is that of a
contraction done half at the FP8 rate (twice the measured BF16 rate, the nominal ratio) and
half at the BF16 rate.

--fp8 times attn_fwd_fp8: Q, K and V quantized per tensor to E4M3 (V passed transposed), P
rounded to E4M3 for the P V product; the roofline peak is the FP8 rate for all FLOPs.

--mxfp8 times attn_fwd_mxfp8: Q, K and V quantized to MXFP8 (E4M3 codes, one E8M0 scale per 32
elements along d for Q and K, per 32 keys for V), both products block-scaled on the tensor
cores; the roofline peak is the FP8 rate for all FLOPs.

--impl reference times the FP64 CPU oracle (the plain definition) on host cores, on a
bounded sample of query rows per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dense_attention_forward_fwd_gb300.configs import WORKLOADS, by_name  # noqa: E402

METRIC = "attention fwd TFLOPS (4·B·H·N²·d) and % of GB300 dense-BF16 tensor peak"
DEFAULT_WORKLOAD = "long-16k"
# The pages' own figure for this shape: the from-scratch v5 kernel on an RTX 5090
# ("Flash Attention на 5090 в CUDA C++", benchmark table). Another GPU: context only.
PAGES_TFLOPS = {"rect-4k-8k": 197.74}
L2_FLUSH_BYTES = 512 << 20
KERNEL_SRC = os.path.join(ROOT, "dense_attention_forward_fwd_gb300", "csrc", "attn_fwd.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=[w.name for w in WORKLOADS])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    ap.add_argument("--causal", action="store_true",
                    help="causal mask (query i sees keys 0 .. i + Nk - Nq); FLOPs count visible pairs only")
    ap.add_argument("--bias", choices=["none", "shared", "full"], default="none",
                    help="additive BF16 bias N(0,1): one [Nq, Nk] matrix for all heads, or one per head")
    ap.add_argument("--backward", action="store_true",
                    help="time attn_bwd (dQ, dK, dV for an N(0,1) upstream gradient); FLOPs = 2.5x the forward's")
    ap.add_argument("--fp8-qk", action="store_true",
                    help="time attn_fwd_fp8qk (Q and K as FP8 E4M3 codes with per-tensor descale factors)")
    ap.add_argument("--fp8", action="store_true",
                    help="time attn_fwd_fp8 (Q, K and V as FP8 E4M3 codes, P rounded to E4M3 for P V)")
    ap.add_argument("--mxfp8", action="store_true",
                    help="time attn_fwd_mxfp8 (Q, K and V in MXFP8, both products block-scaled)")
    ap.add_argument("--head-dim", type=int, choices=[128, 192, 256], default=128,
                    help="head dimension d of the workload's tensors (192 and 256: the one-Q-tile kernel "
                         "of attn_fwd and attn_fwd_causal; scale 1/sqrt(d))")
    args = ap.parse_args()
    if args.head_dim != 128 and (args.backward or args.mxfp8):
        ap.error("--head-dim 192 / 256 has the forward entry points without block scales only (attn_fwd, "
                 "attn_fwd_causal, attn_fwd_bias and the attn_fwd_fp8qk and attn_fwd_fp8 families)")
    if (args.fp8_qk or args.fp8 or args.mxfp8) and args.backward:
        ap.error("--fp8-qk, --fp8 and --mxfp8 have no backward entry point")
    if args.mxfp8 and args.bias != "none":
        ap.error("--mxfp8 has no bias entry point (--fp8-qk and --fp8 have)")
    if args.fp8_qk + args.fp8 + args.mxfp8 > 1:
        ap.error("--fp8-qk, --fp8 and --mxfp8 are different entry points; pick one")
    if args.bias != "none" and args.causal:
        ap.error("--bias has no causal entry point (a causal bias carries the mask)")
    return args


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def run_config(w, args) -> dict:
    """The workload description both arms print (the reference arm times the same one)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": args.causal,
            "bias": args.bias, "pass": "backward" if args.backward else "forward", "qk_mult": w.qk_mult,
            "qk": "mxfp8" if args.mxfp8 else "e4m3" if (args.fp8_qk or args.fp8) else "bf16",
            "pv": "mxfp8" if args.mxfp8 else "e4m3" if args.fp8 else "bf16",
            "inputs": ("iid N(0,1) (Q,K x qk_mult); Q, K, V in MXFP8 (E4M3, E8M0 scale per 32 along d for Q, K "
                       "and per 32 keys for V)" if args.mxfp8 else
                       "iid N(0,1) (Q,K x qk_mult); Q, K, V quantized per tensor to E4M3 (descale = amax/448)"
                       if args.fp8 else
                       "iid N(0,1) (Q,K x qk_mult); Q, K quantized per tensor to E4M3 (descale = amax/448), V BF16"
                       if args.fp8_qk else "iid N(0,1) BF16 (Q,K x qk_mult)"),
            "l2": "flushed (512 MiB write) before every timed launch",
            "vs_baseline_ref": "RTX 5090 v5 kernel, same shape (other hardware: context only)"}


def max_over_ranks(values, pg, device):
    """Each value's maximum over all ranks (a job takes as long as its slowest rank)."""
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs its own copy of the workload (weak scaling, no
    collective on the data path), so the job does world x the work in the slowest rank's time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def kernel_hash(backward: bool = False, wide: bool = False) -> str:
    h = hashlib.sha256()
    csrc = os.path.dirname(KERNEL_SRC)
    shared = os.path.join(csrc, "tc_sm103.cuh")   # the PTX wrappers every kernel file includes
    files = ((os.path.join(csrc, "attn_bwd.cu"), shared, os.path.join(ROOT, "include", "attn_bwd.h")) if backward else
             (os.path.join(csrc, "attn_fwd_wide.cu"), os.path.join(csrc, "attn_wide.h"), shared,
              os.path.join(ROOT, "include", "attn_fwd.h")) if wide else
             (KERNEL_SRC, shared, os.path.join(ROOT, "include", "attn_fwd.h")))
    for f in files:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def roofline_peak(args, peaks: dict, peak_src: str):
    """(peak TFLOP/s, description) of the timed kernel's tensor work. Every FLOP of the BF16
    kernels runs at the measured BF16 burst rate (each launch is timed alone). FP8 MMAs run
    at twice that, the nominal 4.5 / 2.25 PFLOP/s ratio: with FP8 scores only, half the FLOPs
    (Q K^T) do, which gives the harmonic mean 2 / (1/(2P) + 1/P) = 4P/3; with FP8 scores and
    values, all of them (2P)."""
    peak = float(peaks["bf16_tflops"])
    if args.fp8_qk:
        return (2.0 / (1.0 / (2.0 * peak) + 1.0 / peak),
                f"half the FLOPs at 2 x {peak_src} bf16_tflops (FP8 E4M3, nominal ratio 4.5/2.25), "
                "half at bf16_tflops (burst)")
    if args.fp8 or args.mxfp8:
        return 2.0 * peak, f"2 x {peak_src} bf16_tflops (FP8 E4M3, nominal ratio 4.5/2.25; burst)"
    return peak, f"{peak_src} bf16_tflops (burst: each launch is timed alone)"


def traffic_key(w, args) -> str:
    """The profiles/traffic.json key of this run's kernel and workload."""
    return (w.name + ("-causal" if args.causal else "") + ("" if args.bias == "none" else "-bias-" + args.bias)
            + ("-backward" if args.backward else "") + ("-fp8qk" if args.fp8_qk else "")
            + ("-fp8" if args.fp8 else "") + ("-mxfp8" if args.mxfp8 else "")
            + ("" if w.d == 128 else f"-d{w.d}"))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks (nvidia-smi) ----

SMI_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits", "-i", str(gpu_index),
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if len(inside) < 2:
            inside, window = rows, "warmup+timed+after"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


def workload_flops(w, causal: bool) -> float:
    """4*d FLOPs per visible (query, key) pair: all Nq*Nk pairs, or under the causal mask
    Nq*(Nk - Nq) + Nq*(Nq + 1)/2 of them."""
    if not causal:
        return float(w.flops)
    pairs = w.Nq * (w.Nk - w.Nq) + w.Nq * (w.Nq + 1) / 2
    return 4.0 * w.B * w.H * w.d * pairs


# ------------------------------------------------------------------ reference arm (oracle) ---

def oracle_rows_fn(oracle, w, causal: bool, bias_kind: str, H1: int, nq: int, fp8_qk: bool = False,
                   fp8: bool = False, mxfp8: bool = False):
    """The oracle entry point for this run's variant, as fn(q, k, v, scale, rows)."""
    if mxfp8:   # Q, K and V of the same draw in MXFP8
        from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8
        q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, H1, nq, w.Nk, d=w.d, seed=w.seed, qk_mult=w.qk_mult)
        return lambda q, k, v, scale, rows: oracle.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, scale, rows,
                                                                        causal=causal)
    bias = None
    if bias_kind != "none":
        from dense_attention_forward_fwd_gb300.inputs import make_bias
        bias = make_bias((1, 1, nq, w.Nk) if bias_kind == "shared" else (1, H1, nq, w.Nk), seed=w.seed + 1)
    if fp8:   # Q, K and V of the same draw as E4M3 codes
        from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
        q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, H1, nq, w.Nk, d=w.d, seed=w.seed, qk_mult=w.qk_mult)
        return lambda q, k, v, scale, rows: oracle.attention_rows_e4m3(q8, k8, v8, scale, dq, dk, dv, rows,
                                                                       causal=causal, bias=bias)
    if fp8_qk:   # Q and K of the same draw (seed, shape) as E4M3 codes; V is make_qkv's V
        from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3
        q8, k8, _, dq, dk = make_qk_e4m3(1, H1, nq, w.Nk, d=w.d, seed=w.seed, qk_mult=w.qk_mult)
        return lambda q, k, v, scale, rows: oracle.attention_rows_e4m3qk(q8, k8, v, scale, dq, dk, rows,
                                                                         causal=causal, bias=bias)
    if bias is not None:
        return lambda q, k, v, scale, rows: oracle.attention_rows_bias(q, k, v, bias, scale, rows)
    return oracle.attention_rows_causal if causal else oracle.attention_rows


def cpu_oracle_backward_sample(w, target_seconds: float, causal: bool = False, bias_kind: str = "none"):
    """Time the FP64 backward oracle on one head with nq of the workload's query rows (all Nk
    keys, as dK and dV need every row); returns (TFLOPS at 2.5x forward FLOPs, rows, seconds,
    threads)."""
    import numpy as np

    import oracle
    from dense_attention_forward_fwd_gb300.inputs import make_qkv

    def run(nq):
        q, k, v = make_qkv(1, 1, nq, w.Nk, d=w.d, seed=w.seed, qk_mult=w.qk_mult)
        do = np.random.Generator(np.random.PCG64(w.seed + 7)).standard_normal((1, 1, nq, w.d))
        bias = None
        if bias_kind != "none":   # one head's bias (shared or per head: the same work)
            from dense_attention_forward_fwd_gb300.inputs import make_bias
            bias = make_bias((1, 1, nq, w.Nk), seed=w.seed + 1)
        t = time.perf_counter()
        oracle.attention_bwd(q, k, v, do, w.scale, causal=causal, bias=bias)
        return time.perf_counter() - t

    nq = min(w.Nq, 32)
    dt = run(nq)
    nq = int(min(w.Nq, max(nq, nq * target_seconds / max(dt, 1e-6))))
    dt = run(nq)
    pairs = nq * (w.Nk - nq) + nq * (nq + 1) / 2 if causal else nq * w.Nk   # the sample's last nq rows
    return 2.5 * 4.0 * pairs * w.d / dt / 1e12, nq, dt, oracle.max_threads()


def cpu_oracle_sample(w, target_seconds: float, rank_seed: int = 0, causal: bool = False, bias_kind: str = "none",
                      fp8_qk: bool = False, fp8: bool = False, mxfp8: bool = False):
    """Time the FP64 oracle on a sample of query rows; returns (TFLOPS, rows, seconds, threads)."""
    import numpy as np

    import oracle
    from dense_attention_forward_fwd_gb300.inputs import make_qkv

    # K and V of one head are all a row needs; draw the workload's own tensors at full
    # size only when they are small, else draw one head (same distribution).
    H1 = w.H if w.B * w.H * w.Nk * w.d <= (1 << 26) else 1
    nq = min(w.Nq, 4096)
    q, k, v = make_qkv(1, H1, nq, w.Nk, d=w.d, seed=w.seed + rank_seed, qk_mult=w.qk_mult)
    threads = oracle.max_threads()
    fn = oracle_rows_fn(oracle, w, causal, bias_kind, H1, nq, fp8_qk, fp8, mxfp8)

    def flop_rows(rows):   # 4*d FLOPs per visible key of each sampled row
        if not causal:
            return 4.0 * w.Nk * w.d * len(rows)
        # the sample's nq queries are aligned to the end of the key range, like the last nq
        # rows of the workload: row r sees keys 0 .. r + Nk - nq
        i = rows % nq + (w.Nq - nq)
        return float(np.sum(4.0 * w.d * (i + (w.Nk - w.Nq) + 1)))

    n_rows_total = q.shape[1] * q.shape[2]
    probe = min(max(threads, 8), n_rows_total)
    rows = np.linspace(0, n_rows_total - 1, probe).astype(np.int64)   # spread: causal rows differ in length
    t = time.perf_counter()
    fn(q, k, v, w.scale, rows)
    dt = time.perf_counter() - t
    n = int(min(n_rows_total, max(probe, target_seconds / max(dt / probe, 1e-9))))
    rows = np.linspace(0, n_rows_total - 1, n).astype(np.int64)
    t = time.perf_counter()
    fn(q, k, v, w.scale, rows)
    dt = time.perf_counter() - t
    return flop_rows(rows) / dt / 1e12, n, dt, threads


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from dense_attention_forward_fwd_gb300.inputs import make_qkv

    steps, warm = args.steps, args.warmup
    if args.backward:   # each step: the backward oracle on one head, sized to share ~2 minutes
        total, flops_sum = 0.0, 0.0
        for i in range(warm + steps):
            tfl, n, dt, threads = cpu_oracle_backward_sample(w, 120.0 / (steps + warm), args.causal, args.bias)
            if i >= warm:
                total += dt
                flops_sum += tfl * 1e12 * dt
        ms = total / steps * 1e3
        tflops = flops_sum / total / 1e12
        sample = f"backward of one head with {n} query rows x {w.Nk} keys of {w.describe()} per step, FP64"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": run_config(w, args),
            "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }), flush=True)
        return 0
    H1 = w.H if w.B * w.H * w.Nk * w.d <= (1 << 26) else 1
    nq = min(w.Nq, 4096)
    q, k, v = make_qkv(1, H1, nq, w.Nk, d=w.d, seed=w.seed, qk_mult=w.qk_mult)
    threads = oracle.max_threads()
    n_rows_total = q.shape[1] * q.shape[2]
    fn = oracle_rows_fn(oracle, w, args.causal, args.bias, H1, nq, args.fp8_qk, args.fp8, args.mxfp8)

    def flop_rows(rows):   # 4*d FLOPs per visible key; causal sample rows sit at the end of the sequence
        if not args.causal:
            return 4.0 * w.Nk * w.d * len(rows)
        return float(np.sum(4.0 * w.d * (rows % nq + (w.Nk - nq) + 1)))
    # size each step so that warmup + steps take about two minutes in all
    t = time.perf_counter()
    fn(q, k, v, w.scale, np.linspace(0, n_rows_total - 1, threads).astype(np.int64))
    per_row = (time.perf_counter() - t) / threads
    rows_per_step = int(max(1, min(n_rows_total, 120.0 / (steps + warm) / per_row)))
    rng = np.random.Generator(np.random.PCG64(1234))
    for _ in range(warm):
        fn(q, k, v, w.scale, rng.choice(n_rows_total, rows_per_step, replace=False))
    total, flops = 0.0, 0.0
    for _ in range(steps):
        rows = rng.choice(n_rows_total, rows_per_step, replace=False)
        t = time.perf_counter()
        fn(q, k, v, w.scale, rows)
        total += time.perf_counter() - t
        flops += flop_rows(rows)
    ms = total / steps * 1e3
    tflops = flops / total / 1e12
    keys = "visible keys of each row, causal" if args.causal else "full Nk per row"
    sample = f"{rows_per_step} query rows per step of {w.describe()} ({keys}), FP64"
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(w, args),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm ---------------

def run_ours(args, w):
    import numpy as np
    import torch

    import dense_attention_forward_fwd_gb300 as attn

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    attn.load_library()

    def barrier():
        if pg is not None:
            pg.barrier()

    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + rank)
    mult = w.qk_mult
    q = (torch.randn(w.B, w.H, w.Nq, w.d, device=dev, generator=g) * mult).to(torch.bfloat16)
    k = (torch.randn(w.B, w.H, w.Nk, w.d, device=dev, generator=g) * mult).to(torch.bfloat16)
    v = torch.randn(w.B, w.H, w.Nk, w.d, device=dev, generator=g).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.Nq, device=dev, dtype=torch.float32)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.int32)
    stream = torch.cuda.current_stream(dev)

    ins = [q, k, v]
    descale = (1.0, 1.0, 1.0)
    if args.fp8_qk or args.fp8:   # per-tensor quantization to E4M3 codes
        x8, descale = [], []
        for x in ((q, k, v) if args.fp8 else (q, k)):
            ds = float(torch.tensor(x.float().abs().max().item() / 448.0, dtype=torch.float32))
            x8.append((x.float() / ds).to(torch.float8_e4m3fn))
            descale.append(ds)
        if args.fp8:   # V^T, keys innermost (Nk of every workload is a multiple of 16)
            x8[2] = x8[2].transpose(2, 3).contiguous()
        ins = [x8[0], x8[1], x8[2] if args.fp8 else v]
    if args.mxfp8:   # E4M3 codes with an E8M0 scale per 32 elements: along d for Q and K, keys for V
        def mx(x, dim):
            xb = x.float().movedim(dim, -1)
            blocks = xb.reshape(*xb.shape[:-1], -1, 32)
            amax = blocks.abs().amax(dim=-1).clamp_min(torch.finfo(torch.float32).tiny)
            e = (torch.floor(torch.log2(amax)) - 8).clamp(-127, 127)
            codes = (blocks / torch.exp2(e)[..., None]).clamp(-448, 448).to(torch.float8_e4m3fn)
            return codes.reshape(xb.shape), (e + 127).to(torch.uint8)
        q8, sq = mx(q, 3)
        k8, sk = mx(k, 3)
        vt8, svt = mx(v.transpose(2, 3), 3)   # V^T [B,H,d,Nk]: blocks of 32 keys (Nk a multiple of 128)
        ins = [q8.contiguous(), sq.contiguous(), k8.contiguous(), sk.contiguous(), vt8.contiguous(), svt.contiguous()]
    outs = [o, lse]
    if args.bias != "none":
        bshape = (1, 1, w.Nq, w.Nk) if args.bias == "shared" else (w.B, w.H, w.Nq, w.Nk)
        ins.append(torch.randn(bshape, device=dev, generator=g).to(torch.bfloat16))
    if args.backward:   # the forward's O and LSE and an upstream gradient (and the bias) are the inputs
        dout = torch.randn(w.B, w.H, w.Nq, w.d, device=dev, generator=g).to(torch.bfloat16)
        if args.bias != "none":
            attn.attn_fwd_bias(q, k, v, ins[3], o, lse, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, stream)
            ins = [q, k, v, o, dout, lse, ins[3]]
        else:
            (attn.attn_fwd_causal if args.causal else attn.attn_fwd)(q, k, v, o, lse, w.B, w.H, w.Nq, w.Nk, w.d,
                                                                     w.scale, stream)
            ins = [q, k, v, o, dout, lse]
        outs = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]

    def call(ins_, outs_, st):
        if args.backward:
            attn.attn_bwd(*ins_[:6], *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, st, causal=args.causal,
                          bias=ins_[6] if len(ins_) > 6 else None)
        elif args.fp8_qk:
            attn.attn_fwd_fp8qk(*ins_[:3], *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, descale[0], descale[1], st,
                                causal=args.causal, bias=ins_[3] if args.bias != "none" else None)
        elif args.fp8:
            attn.attn_fwd_fp8(*ins_[:3], *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, descale[0], descale[1],
                              descale[2], st, causal=args.causal, bias=ins_[3] if args.bias != "none" else None)
        elif args.bias != "none":
            attn.attn_fwd_bias(ins_[0], ins_[1], ins_[2], ins_[3], *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, st)
        elif args.mxfp8:
            attn.attn_fwd_mxfp8(*ins_, *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, st, causal=args.causal)
        elif args.causal:
            attn.attn_fwd_causal(*ins_, *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, st)
        else:
            attn.attn_fwd(*ins_, *outs_, w.B, w.H, w.Nq, w.Nk, w.d, w.scale, st)

    def kernel_count():
        return attn.attn_fwd_kernel_count() + attn.attn_bwd_kernel_count()

    def status_ok(st):
        return attn.attn_fwd_status(st) == attn.ATTN_OK and attn.attn_bwd_status(st) == attn.ATTN_OK

    flops = (2.5 if args.backward else 1.0) * workload_flops(w, args.causal)

    def step():
        call(ins, outs, stream)

    sampler = ClockSampler(local_rank)   # started early: nvidia-smi needs a moment to come up
    time.sleep(1.0)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    if not status_ok(stream):
        raise RuntimeError("kernel reported a timeout during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    launches0 = kernel_count()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    launches = kernel_count() - launches0
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    durs = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(durs) / len(durs)
    if not status_ok(stream):
        raise RuntimeError("kernel reported a timeout")

    # e2e through host buffers: every step copies its inputs (Q, K, V, and the bias, or for
    # the backward also O, dO and LSE) from pinned host memory, calls the entry point and
    # copies its outputs (O and LSE, or dQ, dK, dV) back, all inside the timed region.
    # Steps are pipelined over three streams with two device buffer sets, as a serving loop
    # would run them: the H2D of step i+1 and the D2H of step i-1 overlap the kernel of step i.
    h_ins = [t.cpu().pin_memory() for t in ins]
    h_outs = [torch.empty_like(t, device="cpu").pin_memory() for t in outs]
    bufs = [([torch.empty_like(t) for t in ins], [torch.empty_like(t) for t in outs]) for _ in range(2)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            d_ins, d_outs = bufs[b]
            s_in.wait_event(ev_done[b])                  # the kernel that read buffer set b is done
            with torch.cuda.stream(s_in):
                for dst, src in zip(d_ins, h_ins):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(s_in)
            s_run.wait_event(ev_in[b])
            s_run.wait_event(ev_out[b])                  # this output set has been copied out
            call(d_ins, d_outs, s_run)
            ev_done[b].record(s_run)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                for dst, src in zip(h_outs, d_outs):
                    dst.copy_(src, non_blocking=True)
                ev_out[b].record(s_out)

    for st in (s_in, s_run, s_out):
        st.wait_stream(stream)
    e2e_steps(3)
    torch.cuda.synchronize()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    es.record(stream)
    for st in (s_in, s_run, s_out):
        st.wait_stream(stream)
    e2e_steps(args.e2e_steps)
    for st in (s_in, s_run, s_out):
        stream.wait_stream(st)
    ee.record(stream)
    torch.cuda.synchronize()
    e2e_ms = es.elapsed_time(ee) / args.e2e_steps
    # the last step's result, read back to the host, must be the device-timed leg's result
    if not all(torch.equal(h, t.cpu()) for h, t in zip(h_outs, outs)):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    h2d = sum(t.numel() * t.element_size() for t in h_ins)
    d2h = sum(t.numel() * t.element_size() for t in h_outs)

    # max over ranks
    if pg is not None:
        ms, e2e_ms = max_over_ranks([ms, e2e_ms], pg, dev)
    value = job_tflops(flops, world, ms)
    e2e_value = job_tflops(flops, world, e2e_ms)

    peak, peak_note = roofline_peak(args, *measured_peaks())
    achieved = flops / (ms * 1e-3) / 1e12   # one launch on one GPU
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        key = traffic_key(w, args)
        rec = json.load(open(TRAFFIC_FILE)).get(key)
        if rec and rec.get("kernel_hash") == kernel_hash(args.backward, w.d != 128):
            traffic = rec.get("bytes_per_launch")

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": ((value / PAGES_TFLOPS[w.name])
                        if w.name in PAGES_TFLOPS and not args.causal and args.bias == "none" and not args.backward
                        and not args.fp8_qk and not args.fp8 and not args.mxfp8 else None),
        "dtype": "mxfp8" if args.mxfp8 else "e4m3" if args.fp8 else "e4m3+bf16" if args.fp8_qk else "bf16",
        "data": "synthetic",
        "config": run_config(w, args),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_note},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
        "kernel_ms_min": min(durs), "kernel_ms_median": statistics.median(durs),
        "gpu": {"name": torch.cuda.get_device_properties(dev).name,
                "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
    }
    if rank == 0 and not args.no_cpu_baseline:
        if args.backward:
            tfl, n, dt, thr = cpu_oracle_backward_sample(w, args.cpu_seconds, args.causal, args.bias)
            sample = f"backward of one head with {n} query rows x {w.Nk} keys of {w.describe()}, FP64, {dt:.1f} s"
        else:
            tfl, n, dt, thr = cpu_oracle_sample(w, args.cpu_seconds, causal=args.causal, bias_kind=args.bias,
                                                fp8_qk=args.fp8_qk, fp8=args.fp8, mxfp8=args.mxfp8)
            keys = "visible keys of each row, causal" if args.causal else "full Nk each"
            sample = f"{n} query rows of {w.describe()} ({keys}), FP64, {dt:.1f} s"
        line["cpu_baseline"] = {"value": tfl, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": sample}
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    w = by_name(args.workload)
    if args.head_dim != w.d:
        import dataclasses
        w = dataclasses.replace(w, d=args.head_dim)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

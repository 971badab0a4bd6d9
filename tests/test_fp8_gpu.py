"""GPU parity of attn_fwd_fp8qk (Q and K as FP8 E4M3 codes with per-tensor descale factors)
and attn_fwd_fp8 (V too) against the FP64 oracle on the same codes.

attn_fwd_fp8qk: the tensor cores form each product of two E4M3 values exactly and sum them
in FP32, as they do for BF16 inputs, so the tolerance is the forward's own: max|dO| <= 1e-2,
mean|dO| <= 1e-3, LSE relative error <= 1e-4 (tests/parity.py). attn_fwd_fp8 also rounds P
to E4M3; its tolerance is derived below.
"""
import math

import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.configs import by_name
from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3, sample_rows
from parity import bf16_to_np, compare, run_gpu, to_device

pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1 / math.sqrt(128)))


def run_fp8(attn, q8, k8, v, scale, dq, dk, causal=False, bias=None):
    import torch
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    q8d = torch.from_numpy(np.ascontiguousarray(q8)).cuda().view(torch.float8_e4m3fn)
    k8d = torch.from_numpy(np.ascontiguousarray(k8)).cuda()          # raw bytes are accepted too
    attn.attn_fwd_fp8qk(q8d, k8d, to_device(v), o, lse, B, H, Nq, Nk, d, scale, dq, dk, causal=causal,
                        bias=None if bias is None else to_device(bias))
    assert attn.attn_fwd_status() == attn.ATTN_OK
    return bf16_to_np(o), lse.cpu().numpy()


def check_fp8(attn, B, H, Nq, Nk, seed, qk_mult=1.0, scale=SCALE, rows=None, causal=False, bias=None):
    q8, k8, v, dq, dk = make_qk_e4m3(B, H, Nq, Nk, seed=seed, qk_mult=qk_mult)
    o, lse = run_fp8(attn, q8, k8, v, scale, dq, dk, causal, bias)
    o_ref, lse_ref = oracle.attention_rows_e4m3qk(q8, k8, v, scale, dq, dk, rows, causal=causal, bias=bias)
    o, lse = o.reshape(-1, 128), lse.reshape(-1)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    # a sharp bias (std 8) concentrates rows on few keys, so |O| reaches the binade where
    # half a BF16 ulp exceeds 1e-2, as with peaked scores
    return compare(o, lse, o_ref, lse_ref, ulp_aware=qk_mult != 1.0 or bias is not None)


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),
    (1, 2, 256, 384),
    (2, 3, 300, 1000),     # ragged query and key tails
    (1, 1, 1, 200),        # a single query row
    (1, 2, 129, 129),
    (1, 2, 256, 5120),     # few groups with long rows: key steps split across blocks
    (4, 2, 768, 768),
])
def test_fp8qk_full_parity(gpu_lib, B, H, Nq, Nk):
    check_fp8(gpu_lib, B, H, Nq, Nk, seed=13000 + Nq + Nk)


def test_fp8qk_peaked_scores(gpu_lib):
    check_fp8(gpu_lib, 1, 2, 512, 2048, seed=13100, qk_mult=3.0)


@pytest.mark.parametrize("scale", [0.0, -0.0883883461356163, 0.5])
def test_fp8qk_other_scales(gpu_lib, scale):
    check_fp8(gpu_lib, 1, 2, 256, 640, seed=13200, scale=scale)


@pytest.mark.parametrize("name", ["rect-4k-8k", "square-4k", "long-16k"])
def test_fp8qk_workload_sampled_rows(gpu_lib, name):
    # the measured shapes at full size, in the launch configuration the benchmark times
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    check_fp8(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows)


def test_fp8qk_agrees_with_the_bf16_entry_point_on_the_same_values(gpu_lib):
    # descale factors of 1: the codes' values are BF16 values, so attn_fwd sees the same inputs
    q8, k8, v, dq, dk = make_qk_e4m3(1, 2, 384, 640, seed=13300)
    torch = pytest.importorskip("torch")
    widen = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    scale = float(np.float32(SCALE * dq * dk))   # the scores of the unquantized N(0,1) inputs
    o8, l8 = run_fp8(gpu_lib, q8, k8, v, scale, 1.0, 1.0)
    ob, lb = run_gpu(gpu_lib, widen(q8), widen(k8), v, scale)
    assert np.max(np.abs(o8 - ob)) <= 1e-2 and np.max(np.abs(l8 - lb)) <= 1e-4 * max(1.0, np.max(np.abs(lb)))


def test_fp8qk_is_deterministic(gpu_lib):
    q8, k8, v, dq, dk = make_qk_e4m3(1, 2, 256, 5120, seed=13400)
    a = run_fp8(gpu_lib, q8, k8, v, SCALE, dq, dk)
    b = run_fp8(gpu_lib, q8, k8, v, SCALE, dq, dk)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- attn_fwd_fp8: V as E4M3 codes too, P rounded to E4M3 for the P V product ----------------
#
# Tolerance. P rounded to E4M3 keeps 3 mantissa bits: each weight moves by up to 2^-4 of
# itself, weights below 2^-6 of the running maximum keep fewer bits and those below 2^-10
# vanish. A CPU emulation of the kernel's rounding points (FP32 scores and weights, the
# running maximum moved in steps of more than 8 in log2 units, P rounded to E4M3, l the
# FP32 sum of the unrounded weights plus the rounding error of each tile's largest, BF16
# output) against the FP64 definition on exactly the inputs below gives at most 1.85e-2
# (max) and 2.5e-3 (mean) on N(0,1) inputs, and 9.2e-2 / 4.3e-3 on the peaked (x3) ones.
# The bounds are about twice that. A P byte in the wrong key position, V's descale dropped
# or V read from the wrong rows moves O by 1e-1 or more on average. The LSE does not depend
# on P's rounding and keeps the forward's 1e-4.

def fp8pv_tolerance(qk_mult, causal=False, bias=False):
    # under the causal mask rows near the diagonal average over few keys, and a bias sharpens
    # the rows too (tests/test_fp8_tolerance.py derives both)
    if bias:
        return (1.2e-1, 8e-3)
    if causal:
        return (7e-2, 7e-3) if qk_mult == 1.0 else (2e-1, 1e-2)
    return (4e-2, 5e-3) if qk_mult == 1.0 else (2e-1, 1e-2)


def run_fp8pv(attn, q8, k8, v8, scale, dq, dk, dv, ldv=None, pad_code=0x7F, causal=False, bias=None):
    """v8 is key-major [B,H,Nk,d]; the kernel gets V^T [B,H,d,ldv] with the bytes past Nk of
    each row set to pad_code (NaN by default: a read of them would show in O)."""
    import torch
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    ldv = ldv or (Nk + 15) // 16 * 16
    vt = np.full((B, H, d, ldv), pad_code, dtype=np.uint8)
    vt[..., :Nk] = np.swapaxes(v8, 2, 3)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_fp8(torch.from_numpy(np.ascontiguousarray(q8)).cuda(), torch.from_numpy(np.ascontiguousarray(k8)).cuda(),
                      torch.from_numpy(vt).cuda().view(torch.float8_e4m3fn), o, lse, B, H, Nq, Nk, d, scale, dq, dk, dv,
                      causal=causal, bias=None if bias is None else to_device(bias))
    assert attn.attn_fwd_status() == attn.ATTN_OK
    return bf16_to_np(o), lse.cpu().numpy()


def check_fp8pv(attn, B, H, Nq, Nk, seed, qk_mult=1.0, scale=SCALE, rows=None, ldv=None, causal=False, bias=None):
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(B, H, Nq, Nk, seed=seed, qk_mult=qk_mult)
    o, lse = run_fp8pv(attn, q8, k8, v8, scale, dq, dk, dv, ldv, causal=causal, bias=bias)
    o_ref, lse_ref = oracle.attention_rows_e4m3(q8, k8, v8, scale, dq, dk, dv, rows, causal=causal, bias=bias)
    o, lse = o.reshape(-1, 128), lse.reshape(-1)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), "non-finite output"
    err = np.abs(o.astype(np.float64) - o_ref)
    lse_err = np.abs(lse.astype(np.float64) - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    t_max, t_mean = fp8pv_tolerance(qk_mult, causal, bias is not None)
    assert err.max() <= t_max and err.mean() <= t_mean and lse_err.max() <= 1e-4, \
        f"max {err.max():.3e} mean {err.mean():.3e} lse {lse_err.max():.3e}"
    return err.max(), err.mean()


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),
    (1, 2, 256, 384),
    (2, 3, 300, 1000),     # ragged tails; V^T rows padded to 1008 bytes
    (1, 1, 1, 200),
    (1, 2, 129, 129),
    (1, 2, 256, 5120),     # key steps split across blocks
    (4, 2, 768, 768),
])
def test_fp8_full_parity(gpu_lib, B, H, Nq, Nk):
    check_fp8pv(gpu_lib, B, H, Nq, Nk, seed=14000 + Nq + Nk)


def test_fp8_peaked_scores(gpu_lib):
    check_fp8pv(gpu_lib, 1, 2, 512, 2048, seed=14100, qk_mult=3.0)


@pytest.mark.parametrize("scale", [0.0, -0.0883883461356163])
def test_fp8_other_scales(gpu_lib, scale):
    check_fp8pv(gpu_lib, 1, 2, 256, 640, seed=14200, scale=scale)


def test_fp8_wide_value_rows(gpu_lib):
    # ldv well past Nk: the rows' tails (NaN codes) are never read
    check_fp8pv(gpu_lib, 1, 2, 256, 300, seed=14300, ldv=512)


@pytest.mark.parametrize("name", ["rect-4k-8k", "square-4k", "long-16k"])
def test_fp8_workload_sampled_rows(gpu_lib, name):
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    check_fp8pv(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows)


def test_fp8_lse_matches_the_fp8_score_entry_point(gpu_lib):
    # same scores, same row sums: only the rounding order of l differs between the two
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 2, 384, 1000, seed=14400)
    _, l8 = run_fp8pv(gpu_lib, q8, k8, v8, SCALE, dq, dk, dv)
    vb = (oracle.e4m3_to_f64(v8) * dv).astype(np.float32)
    from dense_attention_forward_fwd_gb300.inputs import f32_to_bf16_bits
    _, lq = run_fp8(gpu_lib, q8, k8, f32_to_bf16_bits(vb), SCALE, dq, dk)
    assert np.max(np.abs(l8 - lq) / np.maximum(1.0, np.abs(lq))) <= 1e-5


def test_fp8_is_deterministic(gpu_lib):
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 2, 256, 5120, seed=14500)
    a = run_fp8pv(gpu_lib, q8, k8, v8, SCALE, dq, dk, dv)
    b = run_fp8pv(gpu_lib, q8, k8, v8, SCALE, dq, dk, dv)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- under the causal mask: attn_fwd_fp8qk_causal and attn_fwd_fp8_causal ----------------------

@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),
    (1, 2, 256, 384),      # Nq < Nk: the mask's corner at key Nk - Nq
    (2, 3, 300, 1000),     # ragged
    (1, 1, 1, 200),
    (1, 2, 129, 129),
    (1, 2, 1000, 1000),
])
def test_fp8qk_causal_parity(gpu_lib, B, H, Nq, Nk):
    check_fp8(gpu_lib, B, H, Nq, Nk, seed=15000 + Nq + Nk, causal=True)


def test_fp8qk_causal_peaked(gpu_lib):
    check_fp8(gpu_lib, 1, 2, 512, 1024, seed=15100, qk_mult=3.0, causal=True)


@pytest.mark.parametrize("B,H,Nq,Nk,seed", [
    (1, 1, 128, 128, 16256),
    (1, 2, 256, 384, 16640),
    (1, 2, 129, 129, 16258),
    (1, 2, 1000, 1000, 18000),
])
def test_fp8_causal_parity(gpu_lib, B, H, Nq, Nk, seed):
    # the inputs tests/test_fp8_tolerance.py derives the causal bounds on
    check_fp8pv(gpu_lib, B, H, Nq, Nk, seed=seed, causal=True)


def test_fp8_causal_peaked(gpu_lib):
    check_fp8pv(gpu_lib, 1, 2, 512, 1024, seed=16100, qk_mult=3.0, causal=True)


@pytest.mark.parametrize("name", ["square-4k"])
def test_fp8_causal_workload_sampled_rows(gpu_lib, name):
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    check_fp8(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows, causal=True)
    check_fp8pv(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows, causal=True)


# ---- with the additive bias: attn_fwd_fp8qk_bias and attn_fwd_fp8_bias -------------------------

def bias_shape(kind, B, H, Nq, Nk):
    return {"full": (B, H, Nq, Nk), "shared": (1, 1, Nq, Nk), "key": (1, 1, 1, Nk)}[kind]


@pytest.mark.parametrize("B,H,Nq,Nk,seed,kind,std", [
    (1, 2, 256, 384, 22640, "full", 2.0),
    (2, 3, 300, 1000, 23300, "shared", 2.0),   # ragged; one [Nq, Nk] bias for every head
    (1, 2, 129, 136, 22265, "key", 2.0),       # one bias per key (a padding mask's shape)
    (1, 2, 256, 5120, 27376, "full", 2.0),     # key steps split across blocks
    (1, 2, 512, 1024, 22100, "full", 8.0),     # a sharp bias: late maxima and O rescales
])
def test_fp8_bias_parity(gpu_lib, B, H, Nq, Nk, seed, kind, std):
    # the inputs tests/test_fp8_tolerance.py derives the biased bounds on; the FP8-score entry
    # point (P in BF16) takes the forward's own bounds on the same shapes
    from dense_attention_forward_fwd_gb300.inputs import make_bias
    bias = make_bias(bias_shape(kind, B, H, Nq, Nk), seed=seed + 1, std=std)
    check_fp8pv(gpu_lib, B, H, Nq, Nk, seed=seed, bias=bias)
    check_fp8(gpu_lib, B, H, Nq, Nk, seed=seed, bias=bias)


def test_fp8_bias_masks_keys(gpu_lib):
    # -inf entries remove keys, whole key tiles of them included
    from dense_attention_forward_fwd_gb300.inputs import BF16_NEG_INF, make_bias
    bias = make_bias((1, 1, 1, 1024), seed=22700)
    bias[..., :300] = BF16_NEG_INF
    bias[..., 900:] = BF16_NEG_INF
    check_fp8pv(gpu_lib, 1, 2, 384, 1024, seed=22701, bias=bias)
    check_fp8(gpu_lib, 1, 2, 384, 1024, seed=22701, bias=bias)


@pytest.mark.parametrize("kind", ["shared", "full"])
def test_fp8_bias_workload_sampled_rows(gpu_lib, kind):
    # rect-4k-8k with one bias for every head, or one per head, as `bench.py --bias` times them
    from dense_attention_forward_fwd_gb300.inputs import make_bias
    w = by_name("rect-4k-8k")
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    bias = make_bias(bias_shape(kind, w.B, w.H, w.Nq, w.Nk), seed=88, std=1.0)
    check_fp8pv(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows, bias=bias)
    check_fp8(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows, bias=bias)


def test_fp8_bias_and_causal_together_are_refused(gpu_lib):
    import torch
    from dense_attention_forward_fwd_gb300.inputs import make_bias
    q8, k8, v, dq, dk = make_qk_e4m3(1, 1, 128, 128, seed=22800)
    o = torch.empty(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, 128, device="cuda")
    with pytest.raises(ValueError):
        gpu_lib.attn_fwd_fp8qk(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), to_device(v), o, lse, 1, 1, 128,
                               128, 128, SCALE, dq, dk, causal=True, bias=to_device(make_bias((1, 1, 128, 128), seed=1)))

"""Parity of the forward at head dimensions above 128 (d = 192 and 256, attn_fwd's one-Q-tile
kernel) against the FP64 oracle, through the C ABI, on seeded inputs.

The tolerance is the d = 128 one (max|dO| <= 1e-2, mean|dO| <= 1e-3, LSE relative error <=
1e-4): the kernel rounds at the same points (S in FP32, P to BF16 for the tensor cores, FP32
accumulation, BF16 O), and a longer dot product per score adds only FP32 rounding, far below
those bounds.
"""
import numpy as np
import pytest

from dense_attention_forward_fwd_gb300.inputs import (BF16_NEG_INF, bf16_bits_to_f32, f32_to_bf16_bits, make_bias,
                                                  make_qkv, sample_rows)
from parity import check_case, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),     # one query tile, one key step
    (1, 2, 256, 384),     # three key steps: the K ring's boxes wrap
    (1, 2, 300, 200),     # ragged Nq and Nk
    (1, 1, 1, 1),         # a single query and key
    (1, 1, 129, 1),
    (1, 1, 1, 129),
    (2, 3, 1000, 777),
    (1, 2, 128, 2176),    # 17 key steps
])
def test_wide_parity_small(gpu_lib, d, B, H, Nq, Nk):
    check_case(gpu_lib, B, H, Nq, Nk, seed=B * 1000 + Nq + Nk + d, d=d)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_more_tiles_than_blocks(gpu_lib, d):
    # 2 * 8 * 16 = 256 query tiles on at most 152 blocks: blocks run several tiles in turn,
    # so Q, the K ring, the S buffers and O pass from one tile to the next
    check_case(gpu_lib, 2, 8, 2048, 1024, seed=7 + d, d=d)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("seed", [1, 2])
def test_wide_peaked(gpu_lib, d, seed):
    # scores with std ~9: the running max moves late and O is rescaled
    check_case(gpu_lib, 1, 2, 512, 2048, seed=seed, qk_mult=3.0, ulp_aware=True, d=d)


def test_wide_hot_key_in_last_tile_forces_late_rescale(gpu_lib):
    d = 256
    q, k, v = make_qkv(1, 1, 256, 1024, d=d, seed=11)
    qf, kf = bf16_bits_to_f32(q), bf16_bits_to_f32(k)
    kf[0, 0, 1000] = qf[0, 0, 0].copy() * 4   # row 0 sees a score far above all others, late
    kf[0, 0, 1001] = qf[0, 0, 200].copy() * 2
    check_case(gpu_lib, 1, 1, 256, 1024, qkv=(q, f32_to_bf16_bits(kf), v), ulp_aware=True, d=d)


@pytest.mark.parametrize("scale", [-0.0625, 0.0, 0.25])
def test_wide_other_scales(gpu_lib, scale):
    # negative and zero scales take the kernel's other instantiation (scores scaled at load)
    check_case(gpu_lib, 1, 2, 200, 300, seed=5, scale=scale, ulp_aware=True, d=256)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_sampled_rows_long(gpu_lib, d):
    # 8K keys, 16 query tiles per head, 64 seeded rows per head checked
    B, H, Nq, Nk = 1, 4, 2048, 8192
    rows = sample_rows(B, H, Nq, per_head=64)
    check_case(gpu_lib, B, H, Nq, Nk, seed=3, rows=rows, d=d)


def test_wide_deterministic(gpu_lib):
    q, k, v = make_qkv(1, 4, 1024, 2048, d=256, seed=9)
    o1, l1 = run_gpu(gpu_lib, q, k, v, 0.0625)
    o2, l2 = run_gpu(gpu_lib, q, k, v, 0.0625)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_wide_unsupported_head_dims_rejected(gpu_lib):
    import torch
    for d in (64, 160, 320):
        q = torch.zeros(1, 1, 128, d, dtype=torch.bfloat16, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty(1, 1, 128, device="cuda")
        with pytest.raises(gpu_lib.AttnError) as e:
            gpu_lib.attn_fwd(q, q, q, o, lse, 1, 1, 128, 128, d, 0.1)
        assert e.value.status == gpu_lib.ATTN_ERR_UNSUPPORTED


# ---- under the causal mask (attn_fwd_causal at d > 128): query i sees keys 0 .. i + Nk - Nq ----

@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),     # one tile on the diagonal
    (1, 2, 256, 384),     # Nq < Nk: the mask starts at key Nk - Nq
    (2, 3, 300, 1000),    # ragged, several tile lengths
    (1, 1, 1, 129),
    (1, 1, 129, 129),
    (1, 2, 1000, 1000),
])
def test_wide_causal_parity(gpu_lib, d, B, H, Nq, Nk):
    check_case(gpu_lib, B, H, Nq, Nk, seed=B * 100 + Nq + Nk + d, causal=True, d=d)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_causal_many_tiles(gpu_lib, d):
    # 2 * 8 * 16 = 256 tiles of 1 .. 16 key steps on at most 152 blocks (snake order)
    check_case(gpu_lib, 2, 8, 2048, 2048, seed=21 + d, causal=True, d=d)


def test_wide_causal_peaked(gpu_lib):
    check_case(gpu_lib, 1, 2, 512, 1024, seed=4, qk_mult=3.0, ulp_aware=True, causal=True, d=256)


# ---- with an additive bias (attn_fwd_bias at d > 128): S = scale * Q K^T + B ----

def _bias_shape(kind, B, H, Nq, Nk):
    return {"full": (B, H, Nq, Nk), "shared": (1, 1, Nq, Nk), "per_head": (1, H, Nq, Nk),
            "per_key": (1, 1, 1, Nk)}[kind]


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk,kind", [
    (1, 1, 128, 128, "full"),       # one tile, one key step
    (2, 3, 300, 1000, "full"),      # ragged query and key tails
    (1, 2, 384, 640, "shared"),
    (1, 3, 1000, 1776, "per_key"),
    (1, 1, 1, 200, "full"),
    (1, 1, 129, 136, "per_head"),
    (2, 8, 2048, 1024, "shared"),   # more query tiles than blocks
])
def test_wide_bias_parity(gpu_lib, d, B, H, Nq, Nk, kind):
    bias = make_bias(_bias_shape(kind, B, H, Nq, Nk), seed=9500 + Nq + Nk + d, std=2.0)
    check_case(gpu_lib, B, H, Nq, Nk, seed=8500 + Nq + Nk + d, bias=bias, d=d)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_bias_padding_mask_hides_whole_key_tiles(gpu_lib, d):
    # keys 0..299 and 900..999 removed for every row: the running maximum is still -inf when
    # the first visible key arrives, two key steps in
    Nk = 1000
    bias = make_bias((1, 1, 1, Nk), seed=95, std=1.0)
    bias[..., :300] = BF16_NEG_INF
    bias[..., 900:] = BF16_NEG_INF
    check_case(gpu_lib, 1, 2, 384, Nk, seed=96, bias=bias, d=d)


def test_wide_bias_causal_pattern_agrees_with_the_causal_entry_point(gpu_lib):
    d, Nq, Nk = 256, 384, 640
    bias = np.zeros((1, 1, Nq, Nk), dtype=np.uint16)
    for i in range(Nq):
        bias[0, 0, i, i + Nk - Nq + 1:] = BF16_NEG_INF
    q, k, v = make_qkv(1, 2, Nq, Nk, d=d, seed=97)
    check_case(gpu_lib, 1, 2, Nq, Nk, qkv=(q, k, v), bias=bias, d=d)
    ob, lb = run_gpu(gpu_lib, q, k, v, d ** -0.5, bias=bias)
    oc, lc = run_gpu(gpu_lib, q, k, v, d ** -0.5, causal=True)
    assert np.max(np.abs(ob - oc)) <= 2e-2 and np.max(np.abs(lb - lc)) <= 1e-4 * max(1.0, np.max(np.abs(lc)))


@pytest.mark.parametrize("scale", [-0.0625, 0.0])
def test_wide_bias_peaked_and_other_scales(gpu_lib, scale):
    # a bias of standard deviation 8 on peaked scores (late maxima, O rescales; nearly one-hot
    # rows, so |O| reaches 3 and O's own BF16 rounding is judged ulp-aware), and scales of the
    # other sign and zero, where S is the bias alone
    check_case(gpu_lib, 1, 2, 512, 2048, seed=98, qk_mult=3.0, ulp_aware=True, d=256,
               bias=make_bias((1, 2, 512, 2048), seed=99, std=8.0))
    check_case(gpu_lib, 1, 2, 200, 304, seed=100, scale=scale, d=256,
               bias=make_bias((1, 1, 200, 304), seed=101, std=2.0))


def test_wide_bias_of_zeros_matches_the_plain_entry_point(gpu_lib):
    q, k, v = make_qkv(1, 2, 256, 512, d=256, seed=102)
    ob, lb = run_gpu(gpu_lib, q, k, v, 0.0625, bias=np.zeros((1, 1, 1, 512), dtype=np.uint16))
    o0, l0 = run_gpu(gpu_lib, q, k, v, 0.0625)
    assert np.max(np.abs(ob - o0)) <= 1e-2 and np.max(np.abs(lb - l0)) <= 1e-5 * np.max(np.abs(l0))


@pytest.mark.parametrize("kind", ["shared", "full"])
def test_wide_bias_sampled_rows_square(gpu_lib, kind):
    # the 4K x 4K shape at d = 256 as `bench.py --head-dim 256 --bias` times it
    from dense_attention_forward_fwd_gb300.configs import by_name
    w = by_name("square-4k")
    d = 256
    rows = sample_rows(w.B, w.H, w.Nq, per_head=8)
    bias = make_bias(_bias_shape(kind, w.B, w.H, w.Nq, w.Nk), seed=103, std=1.0)
    check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, rows=rows, bias=bias, d=d)


def test_wide_bias_deterministic(gpu_lib):
    q, k, v = make_qkv(1, 4, 1024, 2048, d=192, seed=104)
    bias = make_bias((1, 4, 1024, 2048), seed=105, std=2.0)
    o1, l1 = run_gpu(gpu_lib, q, k, v, 0.07, bias=bias)
    o2, l2 = run_gpu(gpu_lib, q, k, v, 0.07, bias=bias)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("name", ["rect-4k-8k", "square-4k", "peaked-8k", "long-16k"])
def test_wide_workload_sampled_rows(gpu_lib, d, name):
    # the four workloads at d = 192 and 256 as `bench.py --head-dim` launches them
    from dense_attention_forward_fwd_gb300.configs import by_name
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=8)
    check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed + d, qk_mult=w.qk_mult, rows=rows, d=d,
               ulp_aware=w.qk_mult != 1.0)


@pytest.mark.parametrize("name", ["rect-4k-8k", "long-16k"])
def test_wide_causal_workload_sampled_rows(gpu_lib, name):
    from dense_attention_forward_fwd_gb300.configs import by_name
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=8)
    check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed + 256, rows=rows, d=256, causal=True)


# ---- Q and K as FP8 E4M3 codes (the attn_fwd_fp8qk family at d > 128): Q K^T on kind::f8f6f4 ----

def run_fp8_wide(attn, q8, k8, v, scale, dq, dk, causal=False, bias=None):
    import torch
    from parity import bf16_to_np, to_device
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_fp8qk(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), to_device(v), o, lse, B, H, Nq,
                        Nk, d, scale, dq, dk, causal=causal, bias=None if bias is None else to_device(bias))
    assert attn.attn_fwd_status() == attn.ATTN_OK
    return bf16_to_np(o), lse.cpu().numpy()


def check_fp8_wide(attn, B, H, Nq, Nk, d, seed, qk_mult=1.0, rows=None, causal=False, bias=None):
    from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3
    from parity import compare
    import oracle
    scale = d ** -0.5
    q8, k8, v, dq, dk = make_qk_e4m3(B, H, Nq, Nk, d=d, seed=seed, qk_mult=qk_mult)
    o, lse = run_fp8_wide(attn, q8, k8, v, scale, dq, dk, causal, bias)
    o_ref, lse_ref = oracle.attention_rows_e4m3qk(q8, k8, v, scale, dq, dk, rows, causal=causal, bias=bias)
    o, lse = o.reshape(-1, d), lse.reshape(-1)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    return compare(o, lse, o_ref, lse_ref, ulp_aware=qk_mult != 1.0 or bias is not None)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),
    (1, 2, 300, 200),     # ragged Nq and Nk
    (2, 3, 1000, 777),
    (1, 1, 1, 129),
    (1, 2, 128, 2176),    # 17 key steps
    (2, 8, 2048, 1024),   # more query tiles than blocks
])
def test_wide_fp8qk_parity(gpu_lib, d, B, H, Nq, Nk):
    check_fp8_wide(gpu_lib, B, H, Nq, Nk, d, seed=18000 + Nq + Nk + d)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk", [(1, 2, 256, 384), (2, 3, 300, 1000)])
def test_wide_fp8qk_causal_parity(gpu_lib, d, B, H, Nq, Nk):
    check_fp8_wide(gpu_lib, B, H, Nq, Nk, d, seed=18100 + Nq + Nk + d, causal=True)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk,kind", [(2, 3, 300, 1000, "full"), (1, 2, 384, 640, "shared")])
def test_wide_fp8qk_bias_parity(gpu_lib, d, B, H, Nq, Nk, kind):
    bias = make_bias(_bias_shape(kind, B, H, Nq, Nk), seed=18200 + Nq + Nk + d, std=2.0)
    check_fp8_wide(gpu_lib, B, H, Nq, Nk, d, seed=18300 + Nq + Nk + d, bias=bias)


def test_wide_fp8qk_peaked(gpu_lib):
    check_fp8_wide(gpu_lib, 1, 2, 512, 2048, 256, seed=18400, qk_mult=3.0)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_fp8qk_agrees_with_the_bf16_entry_point(gpu_lib, d):
    # descale factors of 1: the codes' values are BF16 values, so attn_fwd sees the same inputs
    torch = pytest.importorskip("torch")
    from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3
    q8, k8, v, _, _ = make_qk_e4m3(1, 2, 384, 640, d=d, seed=18500 + d)
    widen = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    scale = 0.01
    o8, l8 = run_fp8_wide(gpu_lib, q8, k8, v, scale, 1.0, 1.0)
    ob, lb = run_gpu(gpu_lib, widen(q8), widen(k8), v, scale)
    assert np.max(np.abs(o8 - ob)) <= 1e-2 and np.max(np.abs(l8 - lb)) <= 1e-4 * max(1.0, np.max(np.abs(lb)))


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("name", ["square-4k", "long-16k"])
def test_wide_fp8qk_workload_sampled_rows(gpu_lib, d, name):
    # as `bench.py --head-dim d --fp8-qk` launches it
    from dense_attention_forward_fwd_gb300.configs import by_name
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=8)
    check_fp8_wide(gpu_lib, w.B, w.H, w.Nq, w.Nk, d, seed=w.seed + 8 * d, rows=rows)


# ---- V as FP8 too (the attn_fwd_fp8 family at d > 128): P rounded to E4M3, P V on kind::f8f6f4 ----
# The tolerance is the d = 128 one (derived in tests/test_fp8_tolerance.py by emulating the
# kernel's rounding of P): it bounds each element of O, an average over keys, whatever d is.

def check_fp8pv_wide(attn, B, H, Nq, Nk, d, seed, qk_mult=1.0, rows=None, causal=False, bias=None, ldv=None):
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    from test_fp8_gpu import fp8pv_tolerance, run_fp8pv
    import oracle
    scale = d ** -0.5
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(B, H, Nq, Nk, d=d, seed=seed, qk_mult=qk_mult)
    o, lse = run_fp8pv(attn, q8, k8, v8, scale, dq, dk, dv, ldv, causal=causal, bias=bias)
    o_ref, lse_ref = oracle.attention_rows_e4m3(q8, k8, v8, scale, dq, dk, dv, rows, causal=causal, bias=bias)
    o, lse = o.reshape(-1, d), lse.reshape(-1)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), "non-finite output"
    err = np.abs(o.astype(np.float64) - o_ref)
    lse_err = np.abs(lse.astype(np.float64) - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    t_max, t_mean = fp8pv_tolerance(qk_mult, causal, bias is not None)
    print(f"d={d} max {err.max():.3e} mean {err.mean():.3e} lse {lse_err.max():.3e}")
    assert err.max() <= t_max and err.mean() <= t_mean and lse_err.max() <= 1e-4, \
        f"max {err.max():.3e} mean {err.mean():.3e} lse {lse_err.max():.3e}"


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),
    (2, 3, 300, 1000),    # ragged tails; V^T rows padded to 1008 bytes (NaN codes past Nk)
    (1, 1, 1, 200),
    (1, 2, 129, 129),
    (1, 2, 128, 2176),    # 17 key steps: the V^T ring wraps
    (2, 8, 2048, 1024),   # more query tiles than blocks
])
def test_wide_fp8_parity(gpu_lib, d, B, H, Nq, Nk):
    check_fp8pv_wide(gpu_lib, B, H, Nq, Nk, d, seed=19000 + Nq + Nk + d)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_fp8_wide_row_stride(gpu_lib, d):
    # V^T rows of 1,024 bytes for 640 keys
    check_fp8pv_wide(gpu_lib, 1, 2, 384, 640, d, seed=19100 + d, ldv=1024)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_fp8_causal_and_bias(gpu_lib, d):
    check_fp8pv_wide(gpu_lib, 2, 3, 300, 1000, d, seed=19200 + d, causal=True)
    bias = make_bias((1, 1, 384, 640), seed=19300 + d, std=2.0)
    check_fp8pv_wide(gpu_lib, 1, 2, 384, 640, d, seed=19400 + d, bias=bias)


def test_wide_fp8_peaked(gpu_lib):
    # the running maximum moves late: with P in E4M3 the rescale threshold is 8 (P <= 256)
    check_fp8pv_wide(gpu_lib, 1, 2, 512, 2048, 256, seed=19500, qk_mult=3.0)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("name", ["square-4k", "long-16k"])
def test_wide_fp8_workload_sampled_rows(gpu_lib, d, name):
    # as `bench.py --head-dim d --fp8` launches it
    from dense_attention_forward_fwd_gb300.configs import by_name
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=8)
    check_fp8pv_wide(gpu_lib, w.B, w.H, w.Nq, w.Nk, d, seed=w.seed + 16 * d, rows=rows)

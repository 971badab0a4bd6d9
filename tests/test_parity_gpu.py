"""Parity of the CUDA path (through the C-ABI) against the FP64 oracle on seeded inputs."""
import math

import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.configs import WORKLOADS, by_name
from dense_attention_forward_fwd_gb300.inputs import (BF16_NEG_INF, bf16_bits_to_f32, f32_to_bf16_bits, make_bias,
                                                      make_qkv, sample_rows)
from parity import check_case, compare, run_gpu

pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1 / math.sqrt(128)))


# ---- every element, at sizes spanning several tiles and ragged tails --------------------------

@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 256, 256),     # one block, both Q tiles, two K/V tiles
    (1, 2, 512, 1024),    # several blocks and K/V steps, ring wrap-around
    (2, 3, 384, 640),     # an odd number of Q tiles: second tile of the last block is empty
    (1, 2, 300, 200),     # ragged Nq and Nk
    (1, 1, 1, 1),         # a single query and key
    (1, 1, 129, 1),
    (1, 1, 1, 129),
    (1, 3, 1000, 777),
    (2, 2, 128, 2176),    # 17 K/V steps
    (1, 1, 256, 5120),    # one group of 40 key steps split over 5 blocks
    (1, 2, 300, 3000),    # 4 groups of 24 steps split three ways, ragged tails
    (2, 3, 520, 1290),    # 18 groups of 11 steps: shares cut groups at uneven points
])
def test_full_parity_small(gpu_lib, B, H, Nq, Nk):
    check_case(gpu_lib, B, H, Nq, Nk, seed=B * 1000 + Nq + Nk)


def test_full_parity_tiny_256_workload(gpu_lib):
    w = by_name("tiny-256")
    rep = check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale)
    assert rep.max_abs < 5e-3


@pytest.mark.parametrize("seed", [1, 2])
def test_full_parity_peaked_small(gpu_lib, seed):
    # scores with std ~9: the running max moves late and the O rescale path runs
    check_case(gpu_lib, 1, 2, 512, 2048, seed=seed, qk_mult=3.0, ulp_aware=True)


# ---- the five workloads at full size: every element of O and every LSE on the first four,
# ---- 64 seeded query rows per head on the 16K one ----------------------------------------------

@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_workload_full_size(gpu_lib, name):
    w = by_name(name)
    rows = None
    if w.oracle_rows_per_head is not None:
        rows = sample_rows(w.B, w.H, w.Nq, per_head=w.oracle_rows_per_head)
    check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, qk_mult=w.qk_mult, scale=w.scale, rows=rows,
               ulp_aware=w.qk_mult != 1.0)


# ---- the oracle's closed forms, replayed on the GPU -------------------------------------------

def test_zero_query_gives_mean_of_v(gpu_lib):
    _, k, v = make_qkv(1, 2, 256, 1000, seed=3)
    q = np.zeros((1, 2, 256, 128), dtype=np.uint16)
    o, lse = run_gpu(gpu_lib, q, k, v, SCALE)
    mean_v = bf16_bits_to_f32(v).astype(np.float64).mean(axis=2)
    compare(o.reshape(-1, 128), lse.reshape(-1), np.repeat(mean_v[0], 256, axis=0),
            np.full(512, math.log(1000)))


def test_constant_v_returns_it(gpu_lib):
    q, k, _ = make_qkv(1, 1, 256, 384, seed=4, qk_mult=3.0)
    c = np.array([((i % 9) - 4) * 0.5 for i in range(128)], dtype=np.float32)
    v = np.broadcast_to(f32_to_bf16_bits(c), (1, 1, 384, 128)).copy()
    o, _ = run_gpu(gpu_lib, q, k, v, SCALE)
    assert np.max(np.abs(o - c)) <= 1e-2


def test_identical_keys_behave_like_one_key(gpu_lib):
    q, k1, v1 = make_qkv(1, 1, 256, 1, seed=5)
    k = np.repeat(k1, 128, axis=2)
    v = np.repeat(v1, 128, axis=2)
    o, lse = run_gpu(gpu_lib, q, k, v, SCALE)
    s = SCALE * (bf16_bits_to_f32(q)[0, 0].astype(np.float64) @ bf16_bits_to_f32(k1)[0, 0, 0].astype(np.float64))
    compare(o.reshape(-1, 128), lse.reshape(-1),
            np.repeat(bf16_bits_to_f32(v1)[0, 0].astype(np.float64), 256, axis=0), s + math.log(128))


def test_hot_key_in_last_tile_forces_late_rescale(gpu_lib):
    q, k, v = make_qkv(1, 1, 256, 1024, seed=6)
    qf = bf16_bits_to_f32(q)
    kf = bf16_bits_to_f32(k)
    kf[0, 0, 1000] = qf[0, 0, 0].copy() * 4  # row 0 sees a score far above all others, late
    kf[0, 0, 1001] = qf[0, 0, 200].copy() * 2
    k = f32_to_bf16_bits(kf)
    check_case(gpu_lib, 1, 1, 256, 1024, qkv=(q, k, v), ulp_aware=True)


@pytest.mark.parametrize("scale", [0.0, -0.0883883461356163, 0.5, 1e-3, 2.0])
def test_other_scales(gpu_lib, scale):
    # scale 2: scores with a standard deviation of ~33 in log2 units, so the running max
    # of most rows moves by more than the rescale threshold after the first tile
    check_case(gpu_lib, 1, 2, 256, 384, seed=8, scale=scale, ulp_aware=True)


def test_rescale_on_many_rows_long_sequence(gpu_lib):
    # scale 2 over 16 key tiles: rescales of O in TMEM at different steps in different rows
    check_case(gpu_lib, 1, 2, 512, 2048, seed=12, scale=2.0, ulp_aware=True)


def test_results_are_deterministic(gpu_lib):
    # a split group: the merge order must not depend on which share finishes last
    q, k, v = make_qkv(1, 1, 256, 5120, seed=9)
    o1, l1 = run_gpu(gpu_lib, q, k, v, SCALE)
    o2, l2 = run_gpu(gpu_lib, q, k, v, SCALE)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_misaligned_device_pointer_rejected(gpu_lib):
    import torch
    buf = torch.zeros(1 * 1 * 128 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(128, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    rc = gpu_lib.load_library().attn_fwd(p + 2, p, p, p, lse.data_ptr(), 1, 1, 128, 128, 128, 0.1, None)
    assert rc == gpu_lib.ATTN_ERR_MISALIGNED


def test_launch_counter_counts_launches(gpu_lib):
    before = gpu_lib.attn_fwd_kernel_count()
    q, k, v = make_qkv(1, 1, 128, 128, seed=10)
    run_gpu(gpu_lib, q, k, v, SCALE)
    assert gpu_lib.attn_fwd_kernel_count() == before + 1


def test_split_workspace_reuse_across_shapes(gpu_lib):
    # Launches on one stream share a workspace; a launch with few split groups followed
    # by one with many must not see arrival counts left over from earlier launches.
    for B, H, Nq, Nk in [(1, 1, 256, 5120), (1, 2, 300, 3000), (1, 1, 256, 5120), (1, 8, 1024, 4096),
                         (1, 2, 300, 3000)]:
        check_case(gpu_lib, B, H, Nq, Nk, seed=Nq + Nk)


# ---- causal mask (query i sees keys 0 .. i + Nk - Nq) ------------------------------------------

@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 256, 256),     # one group: both tiles, the diagonal inside each of the two key tiles
    (1, 2, 512, 512),     # groups of different lengths, longest first
    (2, 3, 384, 640),     # Nq < Nk: the diagonal shifted by 256 keys, an odd number of Q tiles
    (1, 2, 300, 300),     # ragged: partial last Q tile and partial last key tile
    (1, 1, 1, 1),
    (1, 1, 1, 200),       # a single query sees every key
    (1, 1, 129, 129),
    (1, 3, 1000, 1777),
    (4, 2, 768, 768),     # more groups than blocks on a small GPU slice: several waves
])
def test_causal_full_parity(gpu_lib, B, H, Nq, Nk):
    check_case(gpu_lib, B, H, Nq, Nk, seed=7000 + Nq + Nk, causal=True)


def test_causal_first_row_returns_its_own_value(gpu_lib):
    # square: row 0 sees key 0 alone with weight exactly 1, so O[0] is V[0] bit for bit
    q, k, v = make_qkv(1, 2, 384, 384, seed=71)
    o, lse = run_gpu(gpu_lib, q, k, v, SCALE, causal=True)
    assert np.array_equal(o[:, :, 0], bf16_bits_to_f32(v)[:, :, 0])
    expect = SCALE * np.einsum("bhd,bhd->bh", bf16_bits_to_f32(q)[:, :, 0].astype(np.float64),
                               bf16_bits_to_f32(k)[:, :, 0].astype(np.float64))
    assert np.max(np.abs(lse[:, :, 0] - expect)) < 1e-4 * np.maximum(1.0, np.abs(expect)).max()


def test_causal_peaked_and_other_scales(gpu_lib):
    check_case(gpu_lib, 1, 2, 512, 1024, seed=72, qk_mult=3.0, ulp_aware=True, causal=True)
    check_case(gpu_lib, 1, 2, 256, 384, seed=73, scale=-0.0883883461356163, ulp_aware=True, causal=True)
    check_case(gpu_lib, 1, 2, 512, 2048, seed=74, scale=2.0, ulp_aware=True, causal=True)


@pytest.mark.parametrize("name", ["square-4k", "long-16k", "rect-4k-8k", "peaked-8k"])
def test_causal_workload_sampled_rows(gpu_lib, name):
    # every workload under the causal mask as `bench.py --causal` launches it (rect-4k-8k:
    # 128 groups, fewer than two per SM, so their key ranges are split between blocks)
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, qk_mult=w.qk_mult, scale=w.scale, rows=rows, causal=True,
               ulp_aware=w.qk_mult != 1.0)


def test_causal_rejects_more_queries_than_keys(gpu_lib):
    with pytest.raises(gpu_lib.AttnError) as e:
        run_gpu(gpu_lib, *make_qkv(1, 1, 200, 100, seed=75), SCALE, causal=True)
    assert e.value.status == gpu_lib.ATTN_ERR_INVALID_ARG


# ---- additive bias: S = scale * Q K^T + B --------------------------------------------------------

def _bias_shape(kind, B, H, Nq, Nk):
    return {"full": (B, H, Nq, Nk), "shared": (1, 1, Nq, Nk), "per_head": (1, H, Nq, Nk),
            "per_key": (1, 1, 1, Nk)}[kind]


@pytest.mark.parametrize("B,H,Nq,Nk,kind", [
    (1, 2, 256, 256, "full"),
    (2, 3, 300, 1000, "full"),       # ragged query and key tails
    (1, 2, 384, 640, "shared"),
    (1, 3, 1000, 1777, "per_key"),
    (1, 1, 1, 200, "full"),
    (1, 1, 129, 129, "per_key"),
    (1, 2, 256, 5120, "shared"),     # few groups with long rows: key steps split across blocks
    (4, 2, 768, 768, "per_head"),
])
def test_bias_full_parity(gpu_lib, B, H, Nq, Nk, kind):
    bias = make_bias(_bias_shape(kind, B, H, Nq, Nk), seed=9000 + Nq + Nk, std=2.0)
    check_case(gpu_lib, B, H, Nq, Nk, seed=8000 + Nq + Nk, bias=bias)


def test_bias_padding_mask_hides_whole_key_tiles(gpu_lib):
    # keys 0..299 and 900..999 removed for every row: each row starts with two key tiles that
    # are entirely -inf, so its running maximum is still -inf when the first visible key arrives
    Nk = 1000
    bias = make_bias((1, 1, 1, Nk), seed=80)
    bias[..., :300] = BF16_NEG_INF
    bias[..., 900:] = BF16_NEG_INF
    check_case(gpu_lib, 1, 2, 384, Nk, seed=81, bias=bias)


def test_bias_causal_pattern_agrees_with_the_causal_entry_point(gpu_lib):
    Nq, Nk = 384, 640
    bias = np.zeros((1, 1, Nq, Nk), dtype=np.uint16)
    for i in range(Nq):
        bias[0, 0, i, i + Nk - Nq + 1:] = BF16_NEG_INF
    q, k, v = make_qkv(1, 2, Nq, Nk, seed=82)
    check_case(gpu_lib, 1, 2, Nq, Nk, qkv=(q, k, v), bias=bias)
    check_case(gpu_lib, 1, 2, Nq, Nk, qkv=(q, k, v), causal=True)
    ob, lb = run_gpu(gpu_lib, q, k, v, SCALE, bias=bias)
    oc, lc = run_gpu(gpu_lib, q, k, v, SCALE, causal=True)
    assert np.max(np.abs(ob - oc)) <= 2e-2 and np.max(np.abs(lb - lc)) <= 1e-4 * max(1.0, np.max(np.abs(lc)))


def test_bias_peaked_and_negative_scale(gpu_lib):
    # a bias of standard deviation 8 on top of peaked scores: frequent late maxima and O rescales
    check_case(gpu_lib, 1, 2, 512, 2048, seed=83, qk_mult=3.0, ulp_aware=True,
               bias=make_bias((1, 2, 512, 2048), seed=84, std=8.0))
    check_case(gpu_lib, 1, 2, 256, 384, seed=85, scale=-0.0883883461356163,
               bias=make_bias((1, 1, 256, 384), seed=86, std=2.0))


def test_bias_of_zeros_matches_the_plain_entry_point(gpu_lib):
    q, k, v = make_qkv(1, 2, 256, 512, seed=87)
    ob, lb = run_gpu(gpu_lib, q, k, v, SCALE, bias=np.zeros((1, 1, 1, 512), dtype=np.uint16))
    o0, l0 = run_gpu(gpu_lib, q, k, v, SCALE)
    assert np.max(np.abs(ob - o0)) <= 1e-2 and np.max(np.abs(lb - l0)) <= 1e-5 * np.max(np.abs(l0))


@pytest.mark.parametrize("name,kind", [("rect-4k-8k", "shared"), ("rect-4k-8k", "full"), ("square-4k", "shared")])
def test_bias_workload_sampled_rows(gpu_lib, name, kind):
    # the default benchmark shape with one [Nq, Nk] bias shared by every head, or one bias per
    # (batch, head) (537 MB of BF16 for this shape), as `bench.py --bias` times them
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    bias = make_bias(_bias_shape(kind, w.B, w.H, w.Nq, w.Nk), seed=88, std=1.0)
    check_case(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows, bias=bias)


def test_bias_rejects_misaligned_strides(gpu_lib):
    with pytest.raises(gpu_lib.AttnError) as e:
        run_gpu(gpu_lib, *make_qkv(1, 1, 128, 100, seed=89), SCALE, bias=np.zeros((1, 1, 128, 100), np.uint16))
    assert e.value.status == gpu_lib.ATTN_ERR_MISALIGNED


def test_bias_rows_padded_to_16_bytes_for_a_ragged_key_count(gpu_lib):
    # Nk = 129 keys: each bias row is stored with a stride of 136 elements (16-byte rows)
    import torch
    from parity import bf16_to_np, to_device
    Nq, Nk, ld = 200, 129, 136
    q, k, v = make_qkv(1, 2, Nq, Nk, seed=90)
    bias = make_bias((1, 1, Nq, Nk), seed=91, std=2.0)
    padded = np.zeros((1, 1, Nq, ld), dtype=np.uint16)
    padded[..., :Nk] = bias
    bd = to_device(padded)[..., :Nk]
    assert bd.stride(2) == ld
    o = torch.empty(1, 2, Nq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, Nq, dtype=torch.float32, device="cuda")
    gpu_lib.attn_fwd_bias(to_device(q), to_device(k), to_device(v), bd, o, lse, 1, 2, Nq, Nk, 128, SCALE)
    o_ref, l_ref = oracle.attention_rows_bias(q, k, v, bias, SCALE)
    compare(bf16_to_np(o).reshape(-1, 128), lse.cpu().numpy().reshape(-1), o_ref, l_ref)


@pytest.mark.parametrize("bias_kind", [None, "shared"])
def test_split_groups_give_bit_identical_results_on_every_run(gpu_lib, bias_kind):
    # the benchmark shape: every group's key steps are split across blocks, and the block
    # that merges a group is whichever finishes last; the merge order must not depend on it
    import torch
    from parity import to_device
    w = by_name("rect-4k-8k")
    q, k, v = (to_device(x) for x in make_qkv(w.B, w.H, w.Nq, w.Nk, seed=92))
    bias = to_device(make_bias((1, 1, w.Nq, w.Nk), seed=93)) if bias_kind else None
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i in range(6):
        o = torch.empty(w.B, w.H, w.Nq, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
        st = streams[i % 2]
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            if bias is None:
                gpu_lib.attn_fwd(q, k, v, o, lse, w.B, w.H, w.Nq, w.Nk, 128, w.scale, st)
            else:
                gpu_lib.attn_fwd_bias(q, k, v, bias, o, lse, w.B, w.H, w.Nq, w.Nk, 128, w.scale, st)
        torch.cuda.synchronize()
        outs.append((o.cpu(), lse.cpu()))
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


# ---- shapes at the edges of the schedule ---------------------------------------------------------

def test_many_tiny_heads(gpu_lib):
    # 2560 groups of one key step each: many waves of short segments, a 16-key ragged tile
    check_case(gpu_lib, 64, 40, 16, 16, seed=13000)


def test_one_query_over_twenty_thousand_keys(gpu_lib):
    # one group, 157 key steps: every block takes a share of the same group and one merges
    check_case(gpu_lib, 1, 1, 1, 20000, seed=13001)


def test_causal_single_row_over_a_long_sequence(gpu_lib):
    check_case(gpu_lib, 1, 2, 1, 9000, seed=13002, causal=True)


def test_bias_over_a_single_key(gpu_lib):
    # Nk = 1: every row's softmax is exactly 1 whatever the bias; O = V_0
    bias = make_bias((1, 1, 1, 1), seed=13003, std=3.0)
    check_case(gpu_lib, 1, 2, 300, 1, seed=13004, bias=bias)

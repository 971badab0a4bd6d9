"""Parity of the forward at head dimensions above 128 (d = 192 and 256, attn_fwd's one-Q-tile
kernel) against the FP64 oracle, through the C ABI, on seeded inputs.

The tolerance is the d = 128 one (max|dO| <= 1e-2, mean|dO| <= 1e-3, LSE relative error <=
1e-4): the kernel rounds at the same points (S in FP32, P to BF16 for the tensor cores, FP32
accumulation, BF16 O), and a longer dot product per score adds only FP32 rounding, far below
those bounds.
"""
import numpy as np
import pytest

from dense_attention_forward_fwd_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_qkv, sample_rows
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

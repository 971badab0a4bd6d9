"""GPU parity of attn_fwd_mxfp8 (Q, K and V in MXFP8: E4M3 codes with E8M0 scales per 32
elements along the contracted dimension; both products block-scaled on the tensor cores)
against the FP64 oracle on the same codes and scales.

Tolerance: the kernel rounds P to E4M3 (block scale 2^0) for the P V product and nothing
else differs from the definition (each product of two scaled E4M3 values is exact and the
sums are FP32), so the bounds are those of attn_fwd_fp8's P rounding: max|dO| <= 4e-2 and
mean|dO| <= 5e-3 on N(0,1) inputs, 0.2 and 1e-2 on peaked (x3) ones, and the forward's
LSE relative error of 1e-4 (the row sums use the unrounded weights). The derivation of those
bounds is in test_fp8_gpu.py and is rerun on the CPU by test_fp8_tolerance.py. Under the
causal mask (attn_fwd_mxfp8_causal) rows near the diagonal average over few keys, so the
bounds are the causal ones of attn_fwd_fp8_causal (7e-2 and 7e-3 on N(0,1) inputs), which
test_fp8_tolerance.py also checks against an emulation on these MXFP8 inputs.
"""
import math

import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.configs import by_name
from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8, mx_value_layout, sample_rows
from parity import bf16_to_np

pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1 / math.sqrt(128)))


def tolerance(qk_mult, scale=SCALE, causal=False):
    """(max, mean) bounds of |dO|: the N(0,1) ones for scores as sharp as the standard inputs',
    the peaked ones for sharper scores (Q and K x3, or a scale well above 1/sqrt(d))."""
    sharp = qk_mult != 1.0 or abs(scale) > 2 * SCALE
    if sharp:
        return (2e-1, 1e-2)
    return (7e-2, 7e-3) if causal else (4e-2, 5e-3)


def run_mx(attn, q8, sq, k8, sk, v8, sv, scale, causal=False):
    import torch
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    vt8, svt = mx_value_layout(v8, sv)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_mxfp8(dev(q8), dev(sq), dev(k8), dev(sk), dev(vt8), dev(svt), o, lse, B, H, Nq, Nk, d, scale,
                        causal=causal)
    assert attn.attn_fwd_status() == attn.ATTN_OK
    return bf16_to_np(o), lse.cpu().numpy()


def check_mx(attn, B, H, Nq, Nk, seed, qk_mult=1.0, scale=SCALE, rows=None, inputs=None, causal=False):
    q8, sq, k8, sk, v8, sv = inputs if inputs is not None else make_qkv_mxfp8(B, H, Nq, Nk, seed=seed,
                                                                              qk_mult=qk_mult)
    o, lse = run_mx(attn, q8, sq, k8, sk, v8, sv, scale, causal)
    o_ref, lse_ref = oracle.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, scale, rows, causal=causal)
    o, lse = o.reshape(-1, 128), lse.reshape(-1)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), "non-finite output"
    err = np.abs(o.astype(np.float64) - o_ref)
    lse_err = np.abs(lse.astype(np.float64) - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    t_max, t_mean = tolerance(qk_mult, scale, causal)
    print(f"mxfp8 n={err.size} max|dO|={err.max():.3e} mean|dO|={err.mean():.3e} lse_rel={lse_err.max():.3e}")
    assert err.max() <= t_max and err.mean() <= t_mean and lse_err.max() <= 1e-4, \
        f"max {err.max():.3e} mean {err.mean():.3e} lse {lse_err.max():.3e}"
    return err.max(), err.mean()


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),
    (1, 2, 256, 384),
    (2, 3, 300, 1000),     # ragged query and key tails: the last key tile has partial blocks
    (1, 1, 1, 200),
    (1, 2, 129, 129),
    (1, 1, 130, 33),       # a second key block of one key
    (1, 2, 256, 5120),     # key steps split across blocks
    (4, 2, 768, 768),
])
def test_mxfp8_full_parity(gpu_lib, B, H, Nq, Nk):
    check_mx(gpu_lib, B, H, Nq, Nk, seed=15000 + Nq + Nk)


def test_mxfp8_peaked_scores(gpu_lib):
    check_mx(gpu_lib, 1, 2, 512, 2048, seed=15100, qk_mult=3.0)


@pytest.mark.parametrize("scale", [0.0, -0.0883883461356163, 0.5])
def test_mxfp8_other_scales(gpu_lib, scale):
    check_mx(gpu_lib, 1, 2, 256, 640, seed=15200, scale=scale)


def test_mxfp8_scales_vary_per_block(gpu_lib):
    # every block's scale lowered by its own power of two, 2^0 to 2^-3 (codes unchanged), so
    # that blocks of one row differ by up to 8x while the values stay of order one (the
    # bounds are absolute): a scale applied to the wrong row, block or operand moves O or
    # the LSE far outside them
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 2, 256, 640, seed=15300)
    rng = np.random.Generator(np.random.PCG64(15301))
    bump = lambda s: (s.astype(np.int64) - rng.integers(0, 4, size=s.shape)).clip(1, 254).astype(np.uint8)
    inputs = (q8, bump(sq), k8, bump(sk), v8, bump(sv))
    check_mx(gpu_lib, 1, 2, 256, 640, seed=0, inputs=inputs)


@pytest.mark.parametrize("name", ["rect-4k-8k", "square-4k", "long-16k"])
def test_mxfp8_workload_sampled_rows(gpu_lib, name):
    # the measured shapes at full size, in the launch configuration the benchmark times
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    check_mx(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows)


def test_mxfp8_is_deterministic(gpu_lib):
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 2, 256, 5120, seed=15400)
    a = run_mx(gpu_lib, q8, sq, k8, sk, v8, sv, SCALE)
    b = run_mx(gpu_lib, q8, sq, k8, sk, v8, sv, SCALE)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_mxfp8_uniform_scales_equal_the_per_tensor_fp8_entry_point(gpu_lib):
    # one scale per tensor (a power of two): attn_fwd_fp8 with those factors as its descales
    # computes the same products, scaled exactly, with the same rounding of P, so the two
    # entry points agree bit for bit
    import torch
    from test_fp8_gpu import run_fp8pv
    B, H, Nq, Nk = 1, 2, 384, 1000
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(B, H, Nq, Nk, seed=15500)
    eq, ek, ev = 124, 125, 121
    sq, sk, sv = (np.full_like(a, e) for a, e in ((sq, eq), (sk, ek), (sv, ev)))
    o_mx, l_mx = run_mx(gpu_lib, q8, sq, k8, sk, v8, sv, SCALE)
    o_f8, l_f8 = run_fp8pv(gpu_lib, q8, k8, v8, SCALE, 2.0 ** (eq - 127), 2.0 ** (ek - 127), 2.0 ** (ev - 127))
    assert np.array_equal(o_mx, o_f8) and np.array_equal(l_mx, l_f8)


# ---- under the causal mask: attn_fwd_mxfp8_causal ----------------------------------------------

@pytest.mark.parametrize("B,H,Nq,Nk,seed", [
    (1, 1, 128, 128, 19256),
    (1, 2, 256, 384, 19640),     # Nq < Nk: the mask's corner at key Nk - Nq
    (2, 3, 300, 1000, 20300),    # ragged, partial key blocks in the last tile
    (1, 1, 1, 200, 19201),
    (1, 2, 129, 129, 19258),
    (1, 2, 1000, 1000, 21000),
])
def test_mxfp8_causal_parity(gpu_lib, B, H, Nq, Nk, seed):
    # the inputs test_fp8_tolerance.py checks the causal bounds on by emulation
    check_mx(gpu_lib, B, H, Nq, Nk, seed=seed, causal=True)


def test_mxfp8_causal_peaked(gpu_lib):
    check_mx(gpu_lib, 1, 2, 512, 1024, seed=19100, qk_mult=3.0, causal=True)


def test_mxfp8_causal_scales_vary_per_block(gpu_lib):
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 2, 256, 640, seed=19300)
    rng = np.random.Generator(np.random.PCG64(19301))
    bump = lambda s: (s.astype(np.int64) - rng.integers(0, 4, size=s.shape)).clip(1, 254).astype(np.uint8)
    check_mx(gpu_lib, 1, 2, 256, 640, seed=0, inputs=(q8, bump(sq), k8, bump(sk), v8, bump(sv)), causal=True)


@pytest.mark.parametrize("name", ["square-4k", "long-16k"])
def test_mxfp8_causal_workload_sampled_rows(gpu_lib, name):
    w = by_name(name)
    rows = sample_rows(w.B, w.H, w.Nq, per_head=16)
    check_mx(gpu_lib, w.B, w.H, w.Nq, w.Nk, seed=w.seed, scale=w.scale, rows=rows, causal=True)


def test_mxfp8_causal_uniform_scales_equal_the_per_tensor_fp8_entry_point(gpu_lib):
    # as the unmasked case: one power-of-two scale per tensor makes the two entry points agree
    # bit for bit, here through the causal path of both
    from test_fp8_gpu import run_fp8pv
    B, H, Nq, Nk = 1, 2, 384, 1000
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(B, H, Nq, Nk, seed=19500)
    eq, ek, ev = 124, 125, 121
    sq, sk, sv = (np.full_like(a, e) for a, e in ((sq, eq), (sk, ek), (sv, ev)))
    o_mx, l_mx = run_mx(gpu_lib, q8, sq, k8, sk, v8, sv, SCALE, causal=True)
    o_f8, l_f8 = run_fp8pv(gpu_lib, q8, k8, v8, SCALE, 2.0 ** (eq - 127), 2.0 ** (ek - 127), 2.0 ** (ev - 127),
                           causal=True)
    assert np.array_equal(o_mx, o_f8) and np.array_equal(l_mx, l_f8)


def test_mxfp8_causal_keys_past_the_diagonal_do_not_matter(gpu_lib):
    # the codes and scales of keys a row cannot see are changed (NaN scales for V's last
    # blocks, large codes for K's last keys): rows that see none of them keep their outputs
    B, H, Nq, Nk = 1, 1, 256, 256
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(B, H, Nq, Nk, seed=19600)
    o1, l1 = run_mx(gpu_lib, q8, sq, k8, sk, v8, sv, SCALE, causal=True)
    k8b, v8b = k8.copy(), v8.copy()
    k8b[:, :, 200:] = 0x7E     # 448, the largest finite E4M3 code
    v8b[:, :, 200:] = 0x7E
    o2, l2 = run_mx(gpu_lib, q8, sq, k8b, sk, v8b, sv, SCALE, causal=True)
    assert np.array_equal(o1[:, :, :200], o2[:, :, :200]) and np.array_equal(l1[:, :, :200], l2[:, :, :200])
    assert not np.array_equal(o1[:, :, 200:], o2[:, :, 200:])

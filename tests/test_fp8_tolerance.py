"""Where the tolerance of attn_fwd_fp8 comes from, recomputed on the CPU.

attn_fwd_fp8 rounds P to E4M3 before the P V product, so its O differs from the definition
by more than the BF16 path's 1e-2. This test emulates the kernel's rounding points in numpy
(written from the kernel's documented steps; it shares no code with it): scores in FP32
from the exact products of the E4M3 inputs; per 128-key tile the running maximum, moved
only when a tile's maximum exceeds it by more than 8 (log2 units); weights
p = 2^(s * scale * log2 e - m) in FP32, rounded to E4M3 for P V; l the FP32 sum of the
unrounded weights plus the E4M3 rounding error of each tile's largest weight; O = v_descale
* (P8 V8) / l rounded to BF16. It compares that against the FP64 oracle and checks that the
GPU tests' bounds (tests/test_fp8_gpu.py) hold at least 1.5 times the emulated error, on
N(0,1) and peaked (x3) inputs of the shapes the GPU tests use. Under the causal mask
(attn_fwd_fp8_causal) rows near the diagonal average over few keys, so one weight's E4M3
rounding weighs more in their O: the emulation with the mask gives up to 3.6e-2 (max) and
3.6e-3 (mean) on N(0,1) inputs, and the causal GPU tests take their own bounds (CAUSAL_BOUNDS).
attn_fwd_mxfp8 rounds P the same way (E4M3 under a block scale of 2^0) and its products of
scaled E4M3 values are exact, so the same emulation on the decoded MXFP8 values (with a V
descale of 1) gives its error too; the last test checks the MXFP8 GPU tests' inputs.
With an additive bias (attn_fwd_fp8_bias) rows are sharper still: a bias of standard
deviation 2 (8 on peaked rows) gives up to 7.0e-2 (max) and 4.3e-3 (mean), and those GPU
tests take BIAS_BOUNDS.
"""
import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.inputs import bf16_bits_to_f32, make_bias, make_qkv_e4m3, make_qkv_mxfp8

torch = pytest.importorskip("torch")

SCALE = float(np.float32(1 / np.sqrt(128)))
# the GPU tests' bounds: (max, mean) for N(0,1) inputs and for peaked inputs
BOUNDS = {1.0: (4e-2, 5e-3), 3.0: (2e-1, 1e-2)}
CAUSAL_BOUNDS = {1.0: (7e-2, 7e-3), 3.0: (2e-1, 1e-2)}
BIAS_BOUNDS = (1.2e-1, 8e-3)   # attn_fwd_fp8_bias, N(0,1) scores with a bias of std 2 to 8


def to_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float32).numpy()


def to_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def emulate_head(q, k, v8, scale, dv, tau=8.0, causal=False, bias=None):
    """q [Nq, d], k [Nk, d] real inputs (float64), v8 [Nk, d] E4M3 values; returns O [Nq, d].
    causal: row i sees keys 0 .. i + Nk - Nq (a masked weight is exactly 0). bias [Nq, Nk]
    (float64): added to the scaled scores in FP32, then the whole scaled by log2 e."""
    if bias is None:
        t = (q @ k.T).astype(np.float32) * np.float32(scale * 1.4426950408889634)
    else:
        t = ((q @ k.T).astype(np.float32) * np.float32(scale) + bias.astype(np.float32)) * np.float32(1.4426950408889634)
    Nq, Nk = t.shape
    if causal:
        t[np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + (Nk - Nq)] = -np.inf
    m = np.full(Nq, -np.inf, np.float32)
    l = np.zeros(Nq, np.float32)
    corr = np.zeros(Nq, np.float32)
    acc = np.zeros((Nq, v8.shape[1]), np.float64)
    for j0 in range(0, Nk, 128):
        tt = t[:, j0:j0 + 128]
        mt = tt.max(axis=1)
        move = mt > m + tau
        alpha = np.where(move, np.exp2(np.where(np.isinf(m), -np.inf, m - mt)), 1.0).astype(np.float32)
        l, corr, acc = l * alpha, corr * alpha, acc * alpha[:, None]
        m = np.where(move, mt, m)
        with np.errstate(invalid="ignore"):   # a tile fully masked for a row: its weights are 0
            pm = np.where(np.isinf(mt), 0.0, np.exp2(mt - m)).astype(np.float32)
            p = np.where(np.isinf(tt), 0.0, np.exp2(tt - m[:, None])).astype(np.float32)
        corr += to_e4m3(pm) - pm
        l += p.sum(axis=1, dtype=np.float32)
        acc += to_e4m3(p).astype(np.float64) @ v8[j0:j0 + 128]
    return to_bf16(acc * dv / (l + corr)[:, None])


@pytest.mark.parametrize("B,H,Nq,Nk,qk_mult,seed,causal", [
    (1, 1, 128, 128, 1.0, 14256, False),
    (1, 2, 129, 129, 1.0, 14258, False),
    (1, 2, 256, 384, 1.0, 14640, False),
    (4, 2, 768, 768, 1.0, 15536, False),
    (1, 2, 512, 2048, 3.0, 14100, False),
    # the causal GPU tests' inputs (tests/test_fp8_gpu.py)
    (1, 1, 128, 128, 1.0, 16256, True),
    (1, 2, 256, 384, 1.0, 16640, True),
    (1, 2, 129, 129, 1.0, 16258, True),
    (1, 2, 1000, 1000, 1.0, 18000, True),
    (1, 2, 512, 1024, 3.0, 16100, True),
])
def test_gpu_bounds_cover_the_emulated_rounding_error(B, H, Nq, Nk, qk_mult, seed, causal):
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(B, H, Nq, Nk, seed=seed, qk_mult=qk_mult)
    o_ref, _ = oracle.attention_rows_e4m3(q8, k8, v8, SCALE, dq, dk, dv, causal=causal)
    o_ref = o_ref.reshape(B, H, Nq, -1)
    errs = []
    for b in range(B):
        for h in range(H):
            o = emulate_head(oracle.e4m3_to_f64(q8[b, h]) * dq, oracle.e4m3_to_f64(k8[b, h]) * dk,
                             oracle.e4m3_to_f64(v8[b, h]), SCALE, dv, causal=causal)
            errs.append(np.abs(o - o_ref[b, h]))
    err = np.stack(errs)
    t_max, t_mean = (CAUSAL_BOUNDS if causal else BOUNDS)[qk_mult]
    assert err.max() * 1.5 <= t_max, f"emulated max {err.max():.3e} leaves too little margin under {t_max}"
    assert err.mean() * 1.5 <= t_mean, f"emulated mean {err.mean():.3e} leaves too little margin under {t_mean}"
    # and the rounding is visible at all: the bounds are not loose by orders of magnitude
    assert err.max() * 20 >= t_max


def test_the_emulation_without_p_rounding_matches_the_definition():
    # with P kept in FP32 the emulated kernel is the definition up to FP32 and BF16 rounding,
    # so the E4M3 rounding of P is what the bounds above pay for
    global to_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 1, 128, 384, seed=14999)
    o_ref, _ = oracle.attention_rows_e4m3(q8, k8, v8, SCALE, dq, dk, dv)
    keep = to_e4m3
    try:
        to_e4m3 = lambda x: np.asarray(x, dtype=np.float32)   # noqa: E731
        o = emulate_head(oracle.e4m3_to_f64(q8[0, 0]) * dq, oracle.e4m3_to_f64(k8[0, 0]) * dk,
                         oracle.e4m3_to_f64(v8[0, 0]), SCALE, dv)
    finally:
        to_e4m3 = keep
    assert np.abs(o - o_ref).max() <= 1e-2 and np.abs(o - o_ref).mean() <= 1e-3


def mx_decode(codes, scales, axis):
    """E4M3 codes times their E8M0 block scales, the blocks of 32 along `axis`."""
    n = codes.shape[axis]
    f = np.repeat(oracle.e8m0_to_f64(scales), 32, axis=axis)
    return oracle.e4m3_to_f64(codes) * np.take(f, np.arange(n), axis=axis)


@pytest.mark.parametrize("B,H,Nq,Nk,qk_mult,seed,causal", [
    (1, 2, 256, 384, 1.0, 15640, False),
    (4, 2, 768, 768, 1.0, 16536, False),
    (1, 2, 512, 2048, 3.0, 15100, False),
    # the causal MXFP8 GPU tests' inputs (tests/test_mxfp8_gpu.py)
    (1, 1, 128, 128, 1.0, 19256, True),
    (1, 2, 256, 384, 1.0, 19640, True),
    (2, 3, 300, 1000, 1.0, 20300, True),
    (1, 2, 129, 129, 1.0, 19258, True),
    (1, 2, 1000, 1000, 1.0, 21000, True),
    (1, 2, 512, 1024, 3.0, 19100, True),
])
def test_mxfp8_bounds_cover_the_emulated_rounding_error(B, H, Nq, Nk, qk_mult, seed, causal):
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(B, H, Nq, Nk, seed=seed, qk_mult=qk_mult)
    o_ref, _ = oracle.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, SCALE, causal=causal)
    o_ref = o_ref.reshape(B, H, Nq, -1)
    q, k, v = mx_decode(q8, sq, 3), mx_decode(k8, sk, 3), mx_decode(v8, sv, 2)
    err = np.stack([np.abs(emulate_head(q[b, h], k[b, h], v[b, h], SCALE, 1.0, causal=causal) - o_ref[b, h])
                    for b in range(B) for h in range(H)])
    t_max, t_mean = (CAUSAL_BOUNDS if causal else BOUNDS)[qk_mult]
    assert err.max() * 1.5 <= t_max, f"emulated max {err.max():.3e} leaves too little margin under {t_max}"
    assert err.mean() * 1.5 <= t_mean, f"emulated mean {err.mean():.3e} leaves too little margin under {t_mean}"
    assert err.max() * 20 >= t_max


def bias_shape(kind, B, H, Nq, Nk):
    return {"full": (B, H, Nq, Nk), "shared": (1, 1, Nq, Nk), "key": (1, 1, 1, Nk)}[kind]


@pytest.mark.parametrize("B,H,Nq,Nk,seed,kind,std", [
    # the biased FP8 GPU tests' inputs (tests/test_fp8_gpu.py)
    (1, 2, 256, 384, 22640, "full", 2.0),
    (2, 3, 300, 1000, 23300, "shared", 2.0),
    (1, 2, 129, 136, 22265, "key", 2.0),
    (1, 2, 256, 5120, 27376, "full", 2.0),
    (1, 2, 512, 1024, 22100, "full", 8.0),
])
def test_bias_bounds_cover_the_emulated_rounding_error(B, H, Nq, Nk, seed, kind, std):
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(B, H, Nq, Nk, seed=seed)
    bias = make_bias(bias_shape(kind, B, H, Nq, Nk), seed=seed + 1, std=std)
    o_ref, _ = oracle.attention_rows_e4m3(q8, k8, v8, SCALE, dq, dk, dv, bias=bias)
    o_ref = o_ref.reshape(B, H, Nq, -1)
    bf = np.broadcast_to(bf16_bits_to_f32(bias).astype(np.float64), (B, H, Nq, Nk))
    err = np.stack([np.abs(emulate_head(oracle.e4m3_to_f64(q8[b, h]) * dq, oracle.e4m3_to_f64(k8[b, h]) * dk,
                                        oracle.e4m3_to_f64(v8[b, h]), SCALE, dv, bias=bf[b, h]) - o_ref[b, h])
                    for b in range(B) for h in range(H)])
    t_max, t_mean = BIAS_BOUNDS
    assert err.max() * 1.5 <= t_max, f"emulated max {err.max():.3e} leaves too little margin under {t_max}"
    assert err.mean() * 1.5 <= t_mean, f"emulated mean {err.mean():.3e} leaves too little margin under {t_mean}"
    assert err.max() * 20 >= t_max

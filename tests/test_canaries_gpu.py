"""Every entry point writes all of its outputs and nothing else.

Each output (O, LSE, dQ, dK, dV) is the middle of a larger device allocation whose head and
tail hold a NaN canary pattern (tests/canary.py). After the call the canaries must be
intact (no write outside the tensor) and the tensor finite (every element written), on
ragged shapes whose last query and key tiles are partial, and on a shape whose key steps
are split across blocks (the merge writes O and LSE from another block)."""
import math

import numpy as np
import pytest

from canary import fully_written, guarded, intact
from dense_attention_forward_fwd_gb300.inputs import (make_bias, make_qk_e4m3, make_qkv, make_qkv_e4m3, make_qkv_mxfp8,
                                                      mx_value_layout)
from parity import to_device

pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1 / math.sqrt(128)))
SHAPES = [(2, 3, 300, 1000), (1, 1, 1, 200), (1, 2, 256, 5120), (1, 2, 129, 257)]


def outputs(B, H, Nq):
    fo, o = guarded((B, H, Nq, 128), "bf16", "cuda")
    fl, lse = guarded((B, H, Nq), "f32", "cuda")
    return (fo, o), (fl, lse)


def check(attn, *pairs):
    assert attn.attn_fwd_status() == attn.ATTN_OK and attn.attn_bwd_status() == attn.ATTN_OK
    for (flat, view), kind in pairs:
        assert intact(flat, kind), "a write outside the output tensor"
        assert fully_written(view), "an output element left unwritten"


@pytest.mark.parametrize("B,H,Nq,Nk", SHAPES)
def test_forward_entry_points(gpu_lib, B, H, Nq, Nk):
    q, k, v = (to_device(a) for a in make_qkv(B, H, Nq, Nk, seed=17000 + Nq + Nk))
    calls = {
        "attn_fwd": lambda o, l: gpu_lib.attn_fwd(q, k, v, o, l, B, H, Nq, Nk, 128, SCALE),
        "attn_fwd_noalloc": lambda o, l: gpu_lib.attn_fwd_noalloc(q, k, v, o, l, B, H, Nq, Nk, 128, SCALE),
        "attn_fwd_causal": lambda o, l: gpu_lib.attn_fwd_causal(q, k, v, o, l, B, H, Nq, Nk, 128, SCALE),
    }
    # the FP32-output diagnostic: its O is FP32, guarded the same way
    (fo32, o32), (fl32, l32) = guarded((B, H, Nq, 128), "f32", "cuda"), guarded((B, H, Nq), "f32", "cuda")
    gpu_lib.attn_fwd_o32(q, k, v, o32, l32, B, H, Nq, Nk, 128, SCALE)
    check(gpu_lib, ((fo32, o32), "f32"), ((fl32, l32), "f32"))
    bias = to_device(make_bias((B, H, Nq, Nk), seed=17100, std=1.0)) if Nk % 8 == 0 else None
    if bias is not None:   # rows of Nk BF16 values on 16-byte boundaries
        calls["attn_fwd_bias"] = lambda o, l: gpu_lib.attn_fwd_bias(q, k, v, bias, o, l, B, H, Nq, Nk, 128, SCALE)
    for name, call in calls.items():
        (fo, o), (fl, lse) = outputs(B, H, Nq)
        call(o, lse)
        check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,H,Nq,Nk", SHAPES)
def test_forward_wide_head_dims(gpu_lib, d, B, H, Nq, Nk):
    # attn_fwd at d > 128 (the one-Q-tile kernel): each thread stores its own row of O
    q, k, v = (to_device(a) for a in make_qkv(B, H, Nq, Nk, d=d, seed=17300 + Nq + Nk + d))
    (fo, o), (fl, lse) = guarded((B, H, Nq, d), "bf16", "cuda"), guarded((B, H, Nq), "f32", "cuda")
    gpu_lib.attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, d ** -0.5)
    check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
    if Nk % 8 == 0:   # attn_fwd_bias at the same head dimension (bias rows on 16-byte boundaries)
        bias = to_device(make_bias((B, H, Nq, Nk), seed=17400 + Nq + Nk + d, std=1.0))
        (fo, o), (fl, lse) = guarded((B, H, Nq, d), "bf16", "cuda"), guarded((B, H, Nq), "f32", "cuda")
        gpu_lib.attn_fwd_bias(q, k, v, bias, o, lse, B, H, Nq, Nk, d, d ** -0.5)
        check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
    # attn_fwd_fp8qk at the same head dimension (Q and K as E4M3 codes)
    import torch
    q8, k8, v8b, dq, dk = make_qk_e4m3(B, H, Nq, Nk, d=d, seed=17500 + Nq + Nk + d)
    (fo, o), (fl, lse) = guarded((B, H, Nq, d), "bf16", "cuda"), guarded((B, H, Nq), "f32", "cuda")
    gpu_lib.attn_fwd_fp8qk(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), to_device(v8b), o, lse, B, H,
                           Nq, Nk, d, d ** -0.5, dq, dk)
    check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
    # attn_fwd_fp8 at the same head dimension (V^T as E4M3 codes too)
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(B, H, Nq, Nk, d=d, seed=17600 + Nq + Nk + d)
    ldv = (Nk + 15) // 16 * 16
    vt = np.zeros((B, H, d, ldv), dtype=np.uint8)
    vt[..., :Nk] = np.swapaxes(v8, 2, 3)
    (fo, o), (fl, lse) = guarded((B, H, Nq, d), "bf16", "cuda"), guarded((B, H, Nq), "f32", "cuda")
    gpu_lib.attn_fwd_fp8(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), torch.from_numpy(vt).cuda(), o, lse,
                         B, H, Nq, Nk, d, d ** -0.5, dq, dk, dv)
    check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))


@pytest.mark.parametrize("B,H,Nq,Nk", SHAPES)
def test_fp8_entry_points(gpu_lib, B, H, Nq, Nk):
    import torch
    q8, k8, v, dq, dk = make_qk_e4m3(B, H, Nq, Nk, seed=17200 + Nq + Nk)
    q8d, k8d = torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda()
    (fo, o), (fl, lse) = outputs(B, H, Nq)
    gpu_lib.attn_fwd_fp8qk(q8d, k8d, to_device(v), o, lse, B, H, Nq, Nk, 128, SCALE, dq, dk)
    check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(B, H, Nq, Nk, seed=17300 + Nq + Nk)
    ldv = (Nk + 15) // 16 * 16
    vt = np.zeros((B, H, 128, ldv), dtype=np.uint8)
    vt[..., :Nk] = np.swapaxes(v8, 2, 3)
    (fo, o), (fl, lse) = outputs(B, H, Nq)
    gpu_lib.attn_fwd_fp8(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), torch.from_numpy(vt).cuda(), o, lse,
                         B, H, Nq, Nk, 128, SCALE, dq, dk, dv)
    check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
    if Nk % 8 == 0:   # the biased variants (bias rows on 16-byte boundaries)
        bias = to_device(make_bias((B, H, Nq, Nk), seed=17350, std=1.0))
        (fo, o), (fl, lse) = outputs(B, H, Nq)
        gpu_lib.attn_fwd_fp8qk(q8d, k8d, to_device(v), o, lse, B, H, Nq, Nk, 128, SCALE, dq, dk, bias=bias)
        check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
        (fo, o), (fl, lse) = outputs(B, H, Nq)
        gpu_lib.attn_fwd_fp8(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), torch.from_numpy(vt).cuda(), o,
                             lse, B, H, Nq, Nk, 128, SCALE, dq, dk, dv, bias=bias)
        check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
    if Nq <= Nk:   # the causal variants
        (fo, o), (fl, lse) = outputs(B, H, Nq)
        gpu_lib.attn_fwd_fp8qk(q8d, k8d, to_device(v), o, lse, B, H, Nq, Nk, 128, SCALE, dq, dk, causal=True)
        check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))
        (fo, o), (fl, lse) = outputs(B, H, Nq)
        gpu_lib.attn_fwd_fp8(torch.from_numpy(q8).cuda(), torch.from_numpy(k8).cuda(), torch.from_numpy(vt).cuda(), o,
                             lse, B, H, Nq, Nk, 128, SCALE, dq, dk, dv, causal=True)
        check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))


@pytest.mark.parametrize("B,H,Nq,Nk", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_entry_points(gpu_lib, B, H, Nq, Nk, causal):
    import torch
    if causal and Nq > Nk:
        pytest.skip("the causal mask needs Nq <= Nk")
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(B, H, Nq, Nk, seed=17500 + Nq + Nk)
    vt8, svt = mx_value_layout(v8, sv)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    (fo, o), (fl, lse) = outputs(B, H, Nq)
    gpu_lib.attn_fwd_mxfp8(dev(q8), dev(sq), dev(k8), dev(sk), dev(vt8), dev(svt), o, lse, B, H, Nq, Nk, 128, SCALE,
                           causal=causal)
    check(gpu_lib, ((fo, o), "bf16"), ((fl, lse), "f32"))


@pytest.mark.parametrize("B,H,Nq,Nk", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_backward(gpu_lib, B, H, Nq, Nk, causal):
    import torch
    q, k, v = (to_device(a) for a in make_qkv(B, H, Nq, Nk, seed=17400 + Nq + Nk))
    do = torch.randn(B, H, Nq, 128, device="cuda").to(torch.bfloat16)
    o = torch.empty(B, H, Nq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, Nq, dtype=torch.float32, device="cuda")
    (gpu_lib.attn_fwd_causal if causal else gpu_lib.attn_fwd)(q, k, v, o, lse, B, H, Nq, Nk, 128, SCALE)
    fq, dq = guarded((B, H, Nq, 128), "bf16", "cuda")
    fk, dk = guarded((B, H, Nk, 128), "bf16", "cuda")
    fv, dv = guarded((B, H, Nk, 128), "bf16", "cuda")
    gpu_lib.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, Nq, Nk, 128, SCALE, causal=causal)
    check(gpu_lib, ((fq, dq), "bf16"), ((fk, dk), "bf16"), ((fv, dv), "bf16"))
    if not causal and Nk % 8 == 0:   # the biased backward (bias rows on 16-byte boundaries)
        bias = to_device(make_bias((B, H, Nq, Nk), seed=17450, std=1.0))
        gpu_lib.attn_fwd_bias(q, k, v, bias, o, lse, B, H, Nq, Nk, 128, SCALE)
        fq, dq = guarded((B, H, Nq, 128), "bf16", "cuda")
        fk, dk = guarded((B, H, Nk, 128), "bf16", "cuda")
        fv, dv = guarded((B, H, Nk, 128), "bf16", "cuda")
        gpu_lib.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, Nq, Nk, 128, SCALE, bias=bias)
        check(gpu_lib, ((fq, dq), "bf16"), ((fk, dk), "bf16"), ((fv, dv), "bf16"))

"""GPU parity of the backward pass (attn_bwd) against the FP64 oracle's exact gradient.

The CUDA path is fed what a training step has: the forward's own BF16 O and FP32 LSE from
attn_fwd, then an upstream gradient dO. The oracle differentiates the definition exactly
from the same BF16 Q, K, V and dO.

Tolerance, per gradient G in {dQ, dK, dV}: max|dG| <= 2e-2 * max|G_ref| and
mean|dG| <= 1.5e-2 * mean|G_ref|. It comes from a CPU emulation of the kernels' rounding
points (FP32 scores and P, P and dS rounded to BF16 for the tensor cores, D from the
forward's BF16 O, FP32 accumulation, BF16 outputs) against the FP64 oracle: worst case
6.3e-3 of max|G_ref| and 5.8e-3 of mean|G_ref| (peaked inputs), about 2e-3 on N(0,1)
inputs, where BF16 output rounding alone gives 2^-9. A dropped term, a wrong scale or a
transposed operand moves the gradient by O(1) of its size.
"""
import math

import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.inputs import f32_to_bf16_bits, make_qkv
from parity import bf16_to_np, to_device

pytestmark = pytest.mark.gpu

SCALE = float(np.float32(1 / math.sqrt(128)))
MAX_REL = 2e-2
MEAN_REL = 1.5e-2


def make_dout(B, H, Nq, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return f32_to_bf16_bits(rng.standard_normal((B, H, Nq, 128), dtype=np.float32))


def run_fwd_bwd(attn, q, k, v, do, scale, stream=None, causal=False, bias=None):
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    qd, kd, vd, dod = to_device(q), to_device(k), to_device(v), to_device(do)
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())
    bd = None if bias is None else to_device(bias)
    if bd is not None:
        attn.attn_fwd_bias(qd, kd, vd, bd, o, lse, B, H, Nq, Nk, d, scale, stream)
    else:
        (attn.attn_fwd_causal if causal else attn.attn_fwd)(qd, kd, vd, o, lse, B, H, Nq, Nk, d, scale, stream)
    dq = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dk = torch.full((B, H, Nk, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dv = torch.full((B, H, Nk, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    if stream is not None:   # the inputs and outputs were made on the current stream
        stream.wait_stream(torch.cuda.current_stream())
    attn.attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, stream, causal=causal, bias=bd)
    assert attn.attn_fwd_status(stream) == attn.ATTN_OK
    assert attn.attn_bwd_status(stream) == attn.ATTN_OK
    return bf16_to_np(dq), bf16_to_np(dk), bf16_to_np(dv)


def check_bwd(attn, B, H, Nq, Nk, seed, qk_mult=1.0, scale=SCALE, causal=False, bias=None):
    q, k, v = make_qkv(B, H, Nq, Nk, seed=seed, qk_mult=qk_mult)
    do = make_dout(B, H, Nq, seed + 1)
    got = run_fwd_bwd(attn, q, k, v, do, scale, causal=causal, bias=bias)
    ref = oracle.attention_bwd(q, k, v, do, scale, causal=causal, bias=bias)
    report = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(g)), f"{name}: non-finite output"
        err = np.abs(g.astype(np.float64) - r)
        mx, mean = float(err.max()), float(err.mean())
        report[name] = (mx / np.abs(r).max(), mean / np.abs(r).mean())
        assert mx <= MAX_REL * np.abs(r).max(), f"{name}: max err {mx:.3e} vs max|ref| {np.abs(r).max():.3e}"
        assert mean <= MEAN_REL * np.abs(r).mean(), f"{name}: mean err {mean:.3e} vs mean|ref| {np.abs(r).mean():.3e}"
    return report


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 128, 128),      # one tile each way
    (1, 2, 256, 384),      # several query and key tiles
    (2, 3, 300, 1000),     # ragged query and key tails
    (1, 1, 1, 200),        # a single query row
    (1, 2, 129, 129),      # one row / one key past a tile
    (1, 4, 1024, 640),
])
def test_bwd_parity(gpu_lib, B, H, Nq, Nk):
    check_bwd(gpu_lib, B, H, Nq, Nk, seed=11000 + Nq + Nk)


def test_bwd_peaked_scores(gpu_lib):
    check_bwd(gpu_lib, 1, 2, 512, 512, seed=11100, qk_mult=3.0)


def test_bwd_other_scales(gpu_lib):
    check_bwd(gpu_lib, 1, 1, 256, 256, seed=11200, scale=-0.0883883461356163)
    check_bwd(gpu_lib, 1, 1, 256, 512, seed=11201, scale=0.5)


def test_bwd_one_head_of_the_square_workload(gpu_lib):
    # the sequence lengths of the square-4k workload, one head (the oracle's cost grows as Nq*Nk*d)
    check_bwd(gpu_lib, 1, 1, 4096, 4096, seed=11300)


def test_bwd_key_gradients_sum_to_zero_on_the_gpu(gpu_lib):
    # sum_j dK_j = scale * sum_i q_i sum_j dS_ij = 0: BF16 rounding leaves far less than 2 % of
    # sum_j |dK_j| in every (head, column)
    q, k, v = make_qkv(1, 2, 384, 512, seed=11400)
    do = make_dout(1, 2, 384, 11401)
    _, dk, _ = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE)
    dk = dk.astype(np.float64)
    assert np.all(np.abs(dk.sum(axis=2)) <= 2e-2 * np.abs(dk).sum(axis=2))


def test_bwd_is_deterministic_across_runs_and_streams(gpu_lib):
    import torch
    q, k, v = make_qkv(1, 2, 512, 768, seed=11500)
    do = make_dout(1, 2, 512, 11501)
    first = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE)
    st = torch.cuda.Stream()
    for stream in (None, st):
        again = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE, stream)
        for a, b in zip(first, again):
            assert np.array_equal(a, b)


def test_bwd_rejects_bad_arguments(gpu_lib):
    import torch
    t = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    a, b = t.data_ptr(), lse.data_ptr()
    with pytest.raises(gpu_lib.AttnError) as e:
        gpu_lib.attn_bwd(a, a, a, a, a, b, a, a, a, 1, 1, 128, 128, 64, SCALE)
    assert e.value.status == gpu_lib.ATTN_ERR_UNSUPPORTED


# ---- causal backward (the gradient of attn_fwd_causal) --------------------------------------------

@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 256, 256),      # two tiles each way: one diagonal tile per block
    (1, 2, 384, 640),      # Nq < Nk: the diagonal shifted by 256 keys
    (2, 3, 300, 300),      # ragged tails on the diagonal
    (1, 1, 1, 200),        # a single query row sees every key
    (1, 2, 129, 257),      # the shift not a multiple of the tile
    (1, 2, 1024, 1024),    # blocks of very different lengths
])
def test_causal_bwd_parity(gpu_lib, B, H, Nq, Nk):
    check_bwd(gpu_lib, B, H, Nq, Nk, seed=12000 + Nq + Nk, causal=True)


def test_causal_bwd_peaked_and_other_scale(gpu_lib):
    check_bwd(gpu_lib, 1, 2, 512, 768, seed=12100, qk_mult=3.0, causal=True)
    check_bwd(gpu_lib, 1, 1, 256, 384, seed=12101, scale=-0.0883883461356163, causal=True)


def test_causal_bwd_rejects_more_queries_than_keys(gpu_lib):
    import torch
    t = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 256, dtype=torch.float32, device="cuda")
    a, b = t.data_ptr(), lse.data_ptr()
    with pytest.raises(gpu_lib.AttnError) as e:
        gpu_lib.attn_bwd_causal(a, a, a, a, a, b, a, a, a, 1, 1, 256, 128, 128, SCALE)
    assert e.value.status == gpu_lib.ATTN_ERR_INVALID_ARG


# ---- the measured workloads at full size: one launch over every head, sampled heads checked ---------

@pytest.mark.parametrize("name,causal,heads", [
    ("rect-4k-8k", False, ((0, 7),)),              # one head: about 20 s of FP64 oracle on 8 cores
    ("square-4k", False, ((0, 0), (3, 15))),
    ("square-4k", True, ((0, 0), (3, 15))),
])
def test_bwd_workload_sampled_heads(gpu_lib, name, causal, heads):
    """attn_bwd (or attn_bwd_causal) over all B*H heads of a measured workload, as the backward
    bench launches it; the sampled heads (the last one always) are compared with the exact FP64
    gradient on every row of dQ and every key of dK and dV."""
    from dense_attention_forward_fwd_gb300.configs import by_name
    w = by_name(name)
    q, k, v = make_qkv(w.B, w.H, w.Nq, w.Nk, seed=w.seed, qk_mult=w.qk_mult)
    do = make_dout(w.B, w.H, w.Nq, w.seed + 1)
    got = run_fwd_bwd(gpu_lib, q, k, v, do, w.scale, causal=causal)
    assert (w.B - 1, w.H - 1) in heads
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attention_bwd(q[sl], k[sl], v[sl], do[sl], w.scale, causal=causal)
        for gname, g, r in zip(("dq", "dk", "dv"), got, ref):
            g = g[sl]
            assert np.all(np.isfinite(g)), f"{gname} head ({b},{h}): non-finite output"
            err = np.abs(g.astype(np.float64) - r)
            assert err.max() <= MAX_REL * np.abs(r).max(), f"{gname} head ({b},{h}): max err {err.max():.3e}"
            assert err.mean() <= MEAN_REL * np.abs(r).mean(), f"{gname} head ({b},{h}): mean err {err.mean():.3e}"


# ---- the backward of the biased forward (attn_bwd_bias), the bias held fixed ------------------

def bias_shape(kind, B, H, Nq, Nk):
    return {"full": (B, H, Nq, Nk), "shared": (1, 1, Nq, Nk), "key": (1, 1, 1, Nk)}[kind]


@pytest.mark.parametrize("B,H,Nq,Nk,kind", [
    (1, 1, 128, 128, "full"),
    (1, 2, 256, 384, "full"),
    (2, 3, 300, 1000, "shared"),   # ragged query and key tails; one [Nq, Nk] bias for every head
    (1, 1, 1, 200, "full"),        # a single query row; keys end inside a 64-key group
    (1, 2, 129, 136, "key"),       # one bias per key
    (1, 4, 1024, 640, "full"),
])
def test_bwd_bias_parity(gpu_lib, B, H, Nq, Nk, kind):
    from dense_attention_forward_fwd_gb300.inputs import make_bias
    bias = make_bias(bias_shape(kind, B, H, Nq, Nk), seed=12500 + Nq + Nk, std=2.0)
    check_bwd(gpu_lib, B, H, Nq, Nk, seed=12400 + Nq + Nk, bias=bias)


def test_bwd_bias_peaked_and_negative_scale(gpu_lib):
    from dense_attention_forward_fwd_gb300.inputs import make_bias
    check_bwd(gpu_lib, 1, 2, 512, 768, seed=12600, qk_mult=3.0, bias=make_bias((1, 2, 512, 768), seed=12601, std=8.0))
    check_bwd(gpu_lib, 1, 1, 256, 384, seed=12602, scale=-0.0883883461356163,
              bias=make_bias((1, 1, 256, 384), seed=12603, std=2.0))


def test_bwd_bias_masks(gpu_lib):
    # -inf entries remove keys, two whole key tiles of them included, and a causal-pattern bias
    # gives the causal backward's gradients
    from dense_attention_forward_fwd_gb300.inputs import BF16_NEG_INF, make_bias
    bias = make_bias((1, 1, 1, 1024), seed=12700)
    bias[..., :300] = BF16_NEG_INF
    bias[..., 900:] = BF16_NEG_INF
    check_bwd(gpu_lib, 1, 2, 384, 1024, seed=12701, bias=bias)
    Nq, Nk = 256, 384
    mask = np.zeros((1, 1, Nq, Nk), dtype=np.uint16)
    for i in range(Nq):
        mask[0, 0, i, i + Nk - Nq + 1:] = BF16_NEG_INF
    q, k, v = make_qkv(1, 2, Nq, Nk, seed=12702)
    do = make_dout(1, 2, Nq, 12703)
    gb = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE, bias=mask)
    gc = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE, causal=True)
    for a, b in zip(gb, gc):
        assert np.max(np.abs(a - b)) <= 2e-2 * np.abs(b).max()


def test_bwd_bias_zero_is_the_plain_gradient(gpu_lib):
    q, k, v = make_qkv(1, 2, 256, 512, seed=12704)
    do = make_dout(1, 2, 256, 12705)
    gb = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE, bias=np.zeros((1, 1, 1, 512), dtype=np.uint16))
    g0 = run_fwd_bwd(gpu_lib, q, k, v, do, SCALE)
    for a, b in zip(gb, g0):
        assert np.max(np.abs(a - b)) <= 2e-2 * np.abs(b).max()


@pytest.mark.parametrize("kind", ["shared", "full"])
def test_bwd_bias_one_head_of_the_square_workload(gpu_lib, kind):
    # square-4k's shape for one head, with a shared or per-head bias, as `bench.py --backward --bias` times it
    from dense_attention_forward_fwd_gb300.inputs import make_bias
    bias = make_bias(bias_shape(kind, 1, 1, 4096, 4096), seed=12706, std=1.0)
    check_bwd(gpu_lib, 1, 1, 4096, 4096, seed=12707, bias=bias)

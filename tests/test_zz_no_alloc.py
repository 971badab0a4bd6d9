"""attn_fwd_noalloc, the entry point for callers that cannot allocate device memory
(applications with a fixed memory budget, allocation-free hot loops, programs whose
own allocator owns the device), must give the same results as attn_fwd.

It runs the same kernel with its split-merge workspace in a fixed array inside the
library. Two calls in a row check that what the first call leaves in the shared array
does not leak into the second. The file is named to be collected last, and passes both
alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

from dense_attention_forward_fwd_gb300.inputs import make_qkv
from parity import LSE_REL, MAX_ABS, MEAN_ABS, bf16_to_np, to_device

pytestmark = pytest.mark.gpu


def _same_within_tolerance(o_a, l_a, o_b, l_b):
    err = np.abs(o_a.astype(np.float64) - o_b.astype(np.float64))
    lse_err = np.abs(l_a.astype(np.float64) - l_b.astype(np.float64)) / np.maximum(1.0, np.abs(l_b))
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS and lse_err.max() <= LSE_REL, \
        (err.max(), err.mean(), lse_err.max())


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 256, 5120),    # one group split five ways: every share goes through the workspace
    (1, 8, 4096, 8192),   # 128 groups on all SMs, split two or three ways
    (2, 3, 520, 1290),    # ragged tails, uneven split points
])
def test_noalloc_matches_attn_fwd_on_two_calls(gpu_lib, B, H, Nq, Nk):
    import torch
    attn = gpu_lib
    lib = attn.load_library()
    q, k, v = make_qkv(B, H, Nq, Nk, seed=Nq + Nk)
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    scale = float(np.float32(1 / np.sqrt(128)))

    o_ref = torch.empty((B, H, Nq, 128), dtype=torch.bfloat16, device="cuda")
    l_ref = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    attn.attn_fwd(qd, kd, vd, o_ref, l_ref, B, H, Nq, Nk, 128, scale)
    assert attn.attn_fwd_status() == attn.ATTN_OK
    o_ref_np, l_ref_np = bf16_to_np(o_ref), l_ref.cpu().numpy()

    for call in range(2):
        o = torch.full((B, H, Nq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.attn_fwd_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  B, H, Nq, Nk, 128, scale, stream)
        assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
        assert attn.attn_fwd_status() == attn.ATTN_OK
        o_np, l_np = bf16_to_np(o), lse.cpu().numpy()
        assert np.all(np.isfinite(o_np)) and np.all(np.isfinite(l_np)), f"call {call}: unwritten output"
        _same_within_tolerance(o_np, l_np, o_ref_np, l_ref_np)


def test_noalloc_rejects_bad_arguments_like_attn_fwd(gpu_lib):
    lib = gpu_lib.load_library()
    a = 1 << 20
    assert lib.attn_fwd_noalloc(a, a, a, a, a, 1, 1, 128, 128, 64, 0.1, None) == gpu_lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_noalloc(a + 2, a, a, a, a, 1, 1, 128, 128, 128, 0.1, None) == gpu_lib.ATTN_ERR_MISALIGNED
    assert lib.attn_fwd_noalloc(None, a, a, a, a, 1, 1, 128, 128, 128, 0.1, None) == gpu_lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_noalloc(a, a, a, a, a, 0, 1, 128, 128, 128, 0.1, None) == gpu_lib.ATTN_OK

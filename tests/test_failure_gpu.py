"""Failure detection without a GPU fault: a launch that never receives one K/V tile must
give up its bounded waits, exit cleanly and report ATTN_ERR_TIMEOUT through
attn_fwd_status, after which the device keeps working normally.

The missing tile is withheld by the library's test hook (attn_fwd_set_wait_limit): the
producer simply skips one load, so the consumer's wait runs out after the short limit
set here. Nothing traps, faults or hangs.
"""
import pytest

from dense_attention_forward_fwd_gb300.inputs import make_qkv
from parity import check_case, to_device

pytestmark = pytest.mark.gpu

SHORT_LIMIT = 20_000_000   # SM cycles per wait, about 10 ms at 2 GHz


def test_withheld_tile_times_out_cleanly(gpu_lib):
    import torch
    attn = gpu_lib
    q, k, v = make_qkv(1, 2, 512, 1024, seed=21)
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    o = torch.zeros((1, 2, 512, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 512), dtype=torch.float32, device="cuda")
    assert attn.attn_fwd_status() == attn.ATTN_OK
    attn.attn_fwd_set_wait_limit(SHORT_LIMIT, withhold_tile=True)
    try:
        attn.attn_fwd(qd, kd, vd, o, lse, 1, 2, 512, 1024, 128, 0.0883883461356163)
        status = attn.attn_fwd_status()
    finally:
        attn.attn_fwd_set_wait_limit(0, withhold_tile=False)
    assert status == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_fwd_status() == attn.ATTN_OK   # reading the status clears it
    # the context is still usable and the next launch is exact again
    check_case(attn, 1, 2, 512, 1024, seed=21)


def test_backward_withheld_tile_times_out_cleanly(gpu_lib):
    # the dK/dV kernel's loader stops before the second query tile: every waiting role of
    # every block gives up after the short limit, the call reports ATTN_ERR_TIMEOUT, and
    # the next backward is exact again
    import torch
    attn = gpu_lib
    from test_bwd_gpu import check_bwd, make_dout
    q, k, v = make_qkv(1, 2, 512, 384, seed=22)
    do = make_dout(1, 2, 512, 23)
    qd, kd, vd, dod = (to_device(x) for x in (q, k, v, do))
    o = torch.empty((1, 2, 512, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 2, 512), dtype=torch.float32, device="cuda")
    attn.attn_fwd(qd, kd, vd, o, lse, 1, 2, 512, 384, 128, 0.0883883461356163)
    assert attn.attn_fwd_status() == attn.ATTN_OK
    grads = [torch.zeros((1, 2, n, 128), dtype=torch.bfloat16, device="cuda") for n in (512, 384, 384)]
    assert attn.attn_bwd_status() == attn.ATTN_OK
    attn.attn_bwd_set_wait_limit(SHORT_LIMIT, withhold_tile=True)
    try:
        attn.attn_bwd(qd, kd, vd, o, dod, lse, *grads, 1, 2, 512, 384, 128, 0.0883883461356163)
        status = attn.attn_bwd_status()
    finally:
        attn.attn_bwd_set_wait_limit(0, withhold_tile=False)
    assert status == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_bwd_status() == attn.ATTN_OK
    check_bwd(attn, 1, 2, 512, 384, seed=24)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_withheld_tile_times_out_cleanly(gpu_lib, d):
    # d > 128 (the one-query-tile kernel): every block skips its first V unit; the softmax
    # thread that checks V before handing P over gives up, the other roles see the abort
    # flag, and the launch ends with ATTN_ERR_TIMEOUT
    import torch
    attn = gpu_lib
    q, k, v = make_qkv(1, 2, 384, 640, d=d, seed=25 + d)
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    o = torch.zeros((1, 2, 384, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 384), dtype=torch.float32, device="cuda")
    assert attn.attn_fwd_status() == attn.ATTN_OK
    attn.attn_fwd_set_wait_limit(SHORT_LIMIT, withhold_tile=True)
    try:
        attn.attn_fwd(qd, kd, vd, o, lse, 1, 2, 384, 640, d, d ** -0.5)
        status = attn.attn_fwd_status()
    finally:
        attn.attn_fwd_set_wait_limit(0, withhold_tile=False)
    assert status == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_fwd_status() == attn.ATTN_OK
    check_case(attn, 1, 2, 384, 640, seed=25 + d, d=d)

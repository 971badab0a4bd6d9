"""attn_fwd_noalloc, the entry point for callers that cannot allocate device memory
(applications that budget all GPU memory up front, allocation-free hot loops, programs
whose own allocator owns the device), must give attn_fwd's results and allocate nothing.

It runs the same kernel with the same work split and a merge whose order does not depend
on timing, so its O and LSE must equal attn_fwd's bit for bit. The workspace for split
work is a fixed array inside the library that keeps the previous call's contents: two
calls in a row, and a second call on another shape, check that nothing of an earlier call
leaks into a later one. The allocation check reads the device's default memory pool (the
pool cudaMallocAsync draws from) through the driver API around a call on a fresh stream,
where attn_fwd would have to allocate its workspace, and checks that attn_fwd on another
fresh stream does move the pool, so the probe can see an allocation.

The file is named to be collected last; it passes alone in a fresh process and after the
rest of the suite.
"""
import ctypes

import numpy as np
import pytest

from dense_attention_forward_fwd_gb300.inputs import make_qkv
from parity import bf16_to_np, to_device

pytestmark = pytest.mark.gpu

class Driver:
    """The few CUDA driver calls the allocation check needs, on the current context."""
    RESERVED_MEM_CURRENT, USED_MEM_CURRENT = 5, 7   # CUmemPool_attribute values

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def pool_bytes(self):
        out = []
        for attr in (self.RESERVED_MEM_CURRENT, self.USED_MEM_CURRENT):
            v = ctypes.c_uint64()
            assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
            out.append(v.value)
        return tuple(out)

    def new_stream(self) -> int:
        """A stream no earlier call has used (torch's streams come from a reused pool)."""
        s = ctypes.c_void_p()
        assert self.cu.cuStreamCreate(ctypes.byref(s), 1) == 0   # CU_STREAM_NON_BLOCKING
        return s.value


def _prepare(shape, d=128):
    """Seeded inputs and NaN-filled outputs on the device, ready before any timed or probed call."""
    import torch
    B, H, Nq, Nk = shape
    q, k, v = make_qkv(B, H, Nq, Nk, d=d, seed=Nq + Nk)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    bufs = (to_device(q), to_device(k), to_device(v), o, lse)
    torch.cuda.synchronize()   # a call on another stream must see the copies and fills done
    return bufs


def _call(attn, fn_name, shape, bufs, stream=None, d=128):
    """One call of attn_fwd or attn_fwd_noalloc through the C ABI, waited for."""
    import torch
    B, H, Nq, Nk = shape
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = getattr(attn.load_library(), fn_name)(*(t.data_ptr() for t in bufs), B, H, Nq, Nk, d, d ** -0.5, st)
    assert rc == attn.ATTN_OK, attn.attn_status_string(rc)
    assert attn.attn_fwd_status(st) == attn.ATTN_OK   # synchronises the stream


def _result(bufs):
    return bf16_to_np(bufs[3]), bufs[4].cpu().numpy()


def _run(attn, fn_name, shape, stream=None, d=128):
    bufs = _prepare(shape, d)
    _call(attn, fn_name, shape, bufs, stream, d)
    return _result(bufs)


def _assert_same(got, want, what):
    (o, lse), (o_ref, lse_ref) = got, want
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: an output element left unwritten"
    assert np.array_equal(o, o_ref), f"{what}: O differs from attn_fwd's"
    assert np.array_equal(lse, lse_ref), f"{what}: LSE differs from attn_fwd's"


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 1, 256, 5120),    # one group split five ways: every share goes through the workspace
    (1, 8, 4096, 8192),   # 128 groups on all SMs, split two or three ways
    (2, 3, 520, 1290),    # ragged tails, uneven split points
])
def test_noalloc_equals_attn_fwd_on_two_calls(gpu_lib, B, H, Nq, Nk):
    want = _run(gpu_lib, "attn_fwd", (B, H, Nq, Nk))
    for call in range(2):
        _assert_same(_run(gpu_lib, "attn_fwd_noalloc", (B, H, Nq, Nk)), want, f"call {call}")


def test_noalloc_second_call_on_another_shape(gpu_lib):
    # the first call leaves partial records and counters of a many-group split in the array;
    # the second splits fewer, longer groups at other points and must not see them
    first, second = (1, 8, 4096, 8192), (2, 3, 520, 1290)
    want = {s: _run(gpu_lib, "attn_fwd", s) for s in (first, second)}
    for s in (first, second, first):
        _assert_same(_run(gpu_lib, "attn_fwd_noalloc", s), want[s], f"shape {s}")


def test_noalloc_allocates_nothing(gpu_lib):
    import torch
    if torch.cuda.get_allocator_backend() != "native":
        pytest.skip("torch's own allocations come from the probed pool under this allocator backend")
    drv = Driver()
    shape = (1, 8, 4096, 8192)   # split work: attn_fwd needs its workspace here
    want = _run(gpu_lib, "attn_fwd", shape)   # also loads the library's kernels on this device
    s1, s2 = drv.new_stream(), drv.new_stream()
    bufs1, bufs2 = _prepare(shape), _prepare(shape)

    before = drv.pool_bytes()
    _call(gpu_lib, "attn_fwd_noalloc", shape, bufs1, stream=s1)
    after = drv.pool_bytes()
    assert after == before, f"attn_fwd_noalloc changed the memory pool: {before} -> {after}"
    _assert_same(_result(bufs1), want, "noalloc on a fresh stream")

    # the probe sees an allocation: attn_fwd allocates its workspace on a stream it has not used
    _call(gpu_lib, "attn_fwd", shape, bufs2, stream=s2)
    assert drv.pool_bytes()[1] > after[1], "attn_fwd on a fresh stream did not allocate: the probe sees nothing"
    _assert_same(_result(bufs2), want, "attn_fwd on a fresh stream")


def test_noalloc_rejects_bad_arguments_like_attn_fwd(gpu_lib):
    lib = gpu_lib.load_library()
    a = 1 << 20
    assert lib.attn_fwd_noalloc(a, a, a, a, a, 1, 1, 128, 128, 64, 0.1, None) == gpu_lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_noalloc(a + 2, a, a, a, a, 1, 1, 128, 128, 128, 0.1, None) == gpu_lib.ATTN_ERR_MISALIGNED
    assert lib.attn_fwd_noalloc(None, a, a, a, a, 1, 1, 128, 128, 128, 0.1, None) == gpu_lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_noalloc(a, a, a, a, a, 0, 1, 128, 128, 128, 0.1, None) == gpu_lib.ATTN_OK


@pytest.mark.parametrize("d", [192, 256])
def test_noalloc_wide_head_dims(gpu_lib, d):
    # d = 192 / 256: the kernel of attn_fwd at those head dimensions, bit for bit, and no
    # change to the memory pool on a fresh stream
    import torch
    shape = (2, 3, 520, 1290)
    want = _run(gpu_lib, "attn_fwd", shape, d=d)
    bufs = _prepare(shape, d)
    if torch.cuda.get_allocator_backend() == "native":
        drv = Driver()
        s1 = drv.new_stream()
        before = drv.pool_bytes()
        _call(gpu_lib, "attn_fwd_noalloc", shape, bufs, stream=s1, d=d)
        assert drv.pool_bytes() == before, "attn_fwd_noalloc changed the memory pool"
    else:
        _call(gpu_lib, "attn_fwd_noalloc", shape, bufs, d=d)
    _assert_same(_result(bufs), want, f"noalloc at d = {d}")

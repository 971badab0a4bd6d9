"""Dense, non-causal BF16 attention forward (head_dim 128) for GB300, sm_103a.

A thin ctypes binding over the C ABI declared in ``include/attn_fwd.h``; every step of
the computation runs in the CUDA kernels of ``libattn_fwd.so``. The Python side only
checks that tensors match the sizes it passes and marshals pointers and streams.
There is no CPU fallback: if the library cannot be built or loaded, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import threading

from ._build import LIB_PATH, build_library

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED", "ATTN_ERR_CUDA",
    "ATTN_ERR_TIMEOUT", "AttnError", "load_library", "attn_fwd", "attn_fwd_causal", "attn_fwd_bias", "attn_fwd_fp8qk", "attn_fwd_fp8", "attn_fwd_mxfp8", "attn_fwd_o32", "attn_fwd_noalloc", "attn_fwd_status", "attn_status_string",
    "attn_fwd_set_wait_limit", "attn_fwd_kernel_count", "attention", "attn_bwd", "attn_bwd_causal", "attn_bwd_status",
    "attn_bwd_kernel_count", "attn_bwd_set_wait_limit",
]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_MISALIGNED = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TIMEOUT = -5

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str = "attn_fwd"):
        self.status = status
        super().__init__(f"{where} failed: {attn_status_string(status)} ({status})")


def load_library(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load libattn_fwd.so (building it first when it is missing or older than its sources)."""
    global _lib
    with _lock:
        if _lib is None:
            path = build_library() if build_if_stale else LIB_PATH
            lib = ctypes.CDLL(path)
            vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
            lib.attn_fwd.restype = i32
            lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
            lib.attn_fwd_o32.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
            lib.attn_fwd_o32.restype = i32
            lib.attn_fwd_causal.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
            lib.attn_fwd_fp8qk.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, f32, f32, vp]
            lib.attn_fwd_fp8qk.restype = i32
            lib.attn_fwd_fp8.argtypes = [vp, vp, vp, ctypes.c_longlong, vp, vp, i32, i32, i32, i32, i32, f32, f32, f32,
                                         f32, vp]
            lib.attn_fwd_fp8.restype = i32
            lib.attn_fwd_fp8qk_causal.argtypes = lib.attn_fwd_fp8qk.argtypes
            lib.attn_fwd_fp8qk_causal.restype = i32
            lib.attn_fwd_fp8_causal.argtypes = lib.attn_fwd_fp8.argtypes
            lib.attn_fwd_fp8_causal.restype = i32
            ll = ctypes.c_longlong
            lib.attn_fwd_fp8qk_bias.argtypes = [vp, vp, vp, vp, ll, ll, ll, vp, vp, i32, i32, i32, i32, i32, f32, f32,
                                                f32, vp]
            lib.attn_fwd_fp8qk_bias.restype = i32
            lib.attn_fwd_fp8_bias.argtypes = [vp, vp, vp, ll, vp, ll, ll, ll, vp, vp, i32, i32, i32, i32, i32, f32,
                                              f32, f32, f32, vp]
            lib.attn_fwd_fp8_bias.restype = i32
            lib.attn_fwd_mxfp8.argtypes = [vp, vp, vp, vp, vp, ctypes.c_longlong, vp, ctypes.c_longlong, vp, vp, i32, i32,
                                           i32, i32, i32, f32, vp]
            lib.attn_fwd_mxfp8.restype = i32
            lib.attn_fwd_mxfp8_causal.argtypes = lib.attn_fwd_mxfp8.argtypes
            lib.attn_fwd_mxfp8_causal.restype = i32
            i64 = ctypes.c_longlong
            lib.attn_fwd_bias.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, i32, i32, i32, i32, i32, f32, vp]
            lib.attn_fwd_noalloc.restype = i32
            lib.attn_fwd_status.argtypes = [vp]
            lib.attn_fwd_status.restype = i32
            lib.attn_status_string.argtypes = [i32]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_fwd_set_wait_limit.argtypes = [ctypes.c_ulonglong, i32]
            lib.attn_fwd_set_wait_limit.restype = i32
            lib.attn_fwd_kernel_count.argtypes = []
            lib.attn_fwd_kernel_count.restype = ctypes.c_ulonglong
            lib.attn_bwd.argtypes = [vp] * 9 + [i32] * 5 + [f32, vp]
            lib.attn_bwd.restype = i32
            lib.attn_bwd_causal.argtypes = lib.attn_bwd.argtypes
            lib.attn_bwd_bias.argtypes = [vp] * 7 + [ctypes.c_longlong] * 3 + [vp] * 3 + [i32] * 5 + [f32, vp]
            lib.attn_bwd_bias.restype = i32
            lib.attn_bwd_causal.restype = i32
            lib.attn_bwd_status.argtypes = [vp]
            lib.attn_bwd_status.restype = i32
            lib.attn_bwd_kernel_count.argtypes = []
            lib.attn_bwd_kernel_count.restype = ctypes.c_ulonglong
            lib.attn_bwd_set_wait_limit.argtypes = [ctypes.c_ulonglong, i32]
            lib.attn_bwd_set_wait_limit.restype = i32
            _lib = lib
    return _lib


def _is_tensor(x) -> bool:
    return hasattr(x, "data_ptr") and hasattr(x, "is_cuda")


def _ptr(x, name: str, numel: int | None, dtype_name: str):
    """Raw device pointer of a torch tensor (checked against the element count) or an int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if _is_tensor(x):
        import torch
        want = {"bf16": (torch.bfloat16,), "f32": (torch.float32,),
                "e4m3": (torch.float8_e4m3fn, torch.uint8)}[dtype_name]   # E4M3 codes, or their bytes
        if not x.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if x.dtype not in want:
            raise TypeError(f"{name} must be {' or '.join(map(str, want))}, got {x.dtype}")
        if not x.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if numel is not None and x.numel() != numel:
            raise ValueError(f"{name} has {x.numel()} elements, the sizes given need {numel}")
        return x.data_ptr()
    raise TypeError(f"{name}: expected a torch tensor or an integer device pointer, got {type(x).__name__}")


def _stream_handle(stream, *tensors):
    if stream is None:
        for t in tensors:
            if _is_tensor(t):
                import torch
                return torch.cuda.current_stream(t.device).cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def attn_fwd(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, stream=None) -> None:
    """Enqueue O = softmax(scale * Q K^T) V and LSE on ``stream`` (see include/attn_fwd.h).

    q, k, v, o: BF16 [B,H,N,d] CUDA tensors (or integer device pointers); lse: FP32 [B,H,Nq].
    ``stream`` defaults to torch's current stream on the tensors' device. Raises AttnError
    with the library's status code when the call is rejected.
    """
    lib = load_library()
    args = (
        _ptr(q, "q", B * H * Nq * d, "bf16"), _ptr(k, "k", B * H * Nk * d, "bf16"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), _ptr(o, "o", B * H * Nq * d, "bf16"),
        _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    rc = lib.attn_fwd(*args, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                      _stream_handle(stream, q, k, v, o, lse))
    if rc != ATTN_OK:
        raise AttnError(rc)


def attn_fwd_causal(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, stream=None) -> None:
    """Like :func:`attn_fwd`, under the causal mask: query i sees keys 0 .. i + Nk - Nq
    (the mask aligned to the bottom-right corner of the score matrix); needs Nq <= Nk."""
    lib = load_library()
    args = (
        _ptr(q, "q", B * H * Nq * d, "bf16"), _ptr(k, "k", B * H * Nk * d, "bf16"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), _ptr(o, "o", B * H * Nq * d, "bf16"),
        _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    rc = lib.attn_fwd_causal(*args, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                             _stream_handle(stream, q, k, v, o, lse))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_causal")


def attn_fwd_fp8qk(q8, k8, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                   q_descale: float = 1.0, k_descale: float = 1.0, stream=None, causal: bool = False,
                   bias=None, bias_strides=None) -> None:
    """Like :func:`attn_fwd`, with Q and K given as FP8 E4M3 codes (torch.float8_e4m3fn or
    uint8 CUDA tensors [B,H,N,d]) and one positive descale factor each:
    S = scale * q_descale * k_descale * (Q8 K8^T); V, O and LSE as in attn_fwd. causal: under
    the causal mask of attn_fwd_causal (attn_fwd_fp8qk_causal). bias: the additive bias of
    :func:`attn_fwd_bias` (attn_fwd_fp8qk_bias; not with causal)."""
    lib = load_library()
    if bias is not None and causal:
        raise ValueError("bias and causal together are not supported (put the mask in the bias)")
    args = (
        _ptr(q8, "q8", B * H * Nq * d, "e4m3"), _ptr(k8, "k8", B * H * Nk * d, "e4m3"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), _ptr(o, "o", B * H * Nq * d, "bf16"),
        _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    tail = (int(B), int(H), int(Nq), int(Nk), int(d), float(scale), float(q_descale), float(k_descale),
            _stream_handle(stream, q8, k8, v, o, lse))
    if bias is not None:
        name = "attn_fwd_fp8qk_bias"
        rc = lib.attn_fwd_fp8qk_bias(*args[:3], *_bias_arg(bias, B, H, Nq, Nk, bias_strides), *args[3:], *tail)
    else:
        name = "attn_fwd_fp8qk_causal" if causal else "attn_fwd_fp8qk"
        rc = getattr(lib, name)(*args, *tail)
    if rc != ATTN_OK:
        raise AttnError(rc, name)


def attn_fwd_fp8(q8, k8, vt8, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                 q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0, stream=None,
                 ldv: int | None = None, causal: bool = False, bias=None, bias_strides=None) -> None:
    """Like :func:`attn_fwd_fp8qk`, with V as E4M3 codes too, passed transposed: ``vt8`` is
    [B,H,d,ldv] (keys innermost, ldv >= Nk a multiple of 16; a tensor's last dimension is
    taken as ldv). P is rounded to E4M3 for the P V product (see include/attn_fwd.h for the
    accuracy this costs). causal: under the causal mask (attn_fwd_fp8_causal). bias: the
    additive bias of :func:`attn_fwd_bias` (attn_fwd_fp8_bias; not with causal)."""
    lib = load_library()
    if bias is not None and causal:
        raise ValueError("bias and causal together are not supported (put the mask in the bias)")
    if _is_tensor(vt8):
        if vt8.dim() != 4 or tuple(vt8.shape[:3]) != (B, H, d):
            raise ValueError(f"vt8 must be [B, H, d, ldv] = [{B}, {H}, {d}, ldv], got {tuple(vt8.shape)}")
        ldv = int(vt8.shape[3])
    elif ldv is None:
        raise ValueError("ldv is required when vt8 is an integer pointer")
    args = (
        _ptr(q8, "q8", B * H * Nq * d, "e4m3"), _ptr(k8, "k8", B * H * Nk * d, "e4m3"),
        _ptr(vt8, "vt8", B * H * d * ldv, "e4m3"),
    )
    outs = (_ptr(o, "o", B * H * Nq * d, "bf16"), _ptr(lse, "lse", B * H * Nq, "f32"))
    tail = (int(B), int(H), int(Nq), int(Nk), int(d), float(scale), float(q_descale), float(k_descale),
            float(v_descale), _stream_handle(stream, q8, k8, vt8, o, lse))
    if bias is not None:
        name = "attn_fwd_fp8_bias"
        rc = lib.attn_fwd_fp8_bias(*args, int(ldv), *_bias_arg(bias, B, H, Nq, Nk, bias_strides), *outs, *tail)
    else:
        name = "attn_fwd_fp8_causal" if causal else "attn_fwd_fp8"
        rc = getattr(lib, name)(*args, int(ldv), *outs, *tail)
    if rc != ATTN_OK:
        raise AttnError(rc, name)


def attn_fwd_mxfp8(q8, sq, k8, sk, vt8, svt, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                   stream=None, ldv: int | None = None, ldsv: int | None = None, causal: bool = False) -> None:
    """Attention from MXFP8 inputs (see include/attn_fwd.h): E4M3 codes q8 [B,H,Nq,d] and
    k8 [B,H,Nk,d] with E8M0 scales sq [B,H,Nq,d/32] and sk [B,H,Nk,d/32] (32 elements along
    d), V transposed as codes vt8 [B,H,d,ldv] (keys innermost) with scales svt [B,H,d,ldsv]
    (byte t of a row: keys 32t .. 32t+31). A tensor's last dimension is taken as ldv / ldsv.
    O (BF16) and LSE (FP32) as in attn_fwd. causal: under the causal mask (attn_fwd_mxfp8_causal)."""
    lib = load_library()
    for name, t, want in (("vt8", vt8, (B, H, d)), ("svt", svt, (B, H, d))):
        if _is_tensor(t) and (t.dim() != 4 or tuple(t.shape[:3]) != want):
            raise ValueError(f"{name} must be [B, H, d, row bytes] = [{B}, {H}, {d}, ...], got {tuple(t.shape)}")
    if _is_tensor(vt8):
        ldv = int(vt8.shape[3])
    if _is_tensor(svt):
        ldsv = int(svt.shape[3])
    if ldv is None or ldsv is None:
        raise ValueError("ldv and ldsv are required with integer pointers")
    args = (
        _ptr(q8, "q8", B * H * Nq * d, "e4m3"), _ptr(sq, "sq", B * H * Nq * (d // 32), "e4m3"),
        _ptr(k8, "k8", B * H * Nk * d, "e4m3"), _ptr(sk, "sk", B * H * Nk * (d // 32), "e4m3"),
        _ptr(vt8, "vt8", B * H * d * ldv, "e4m3"), int(ldv), _ptr(svt, "svt", B * H * d * ldsv, "e4m3"), int(ldsv),
        _ptr(o, "o", B * H * Nq * d, "bf16"), _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    fn = lib.attn_fwd_mxfp8_causal if causal else lib.attn_fwd_mxfp8
    rc = fn(*args, int(B), int(H), int(Nq), int(Nk), int(d), float(scale), _stream_handle(stream, q8, k8, vt8, o, lse))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_mxfp8_causal" if causal else "attn_fwd_mxfp8")


def _bias_arg(bias, B: int, H: int, Nq: int, Nk: int, bias_strides):
    """(device pointer, stride_b, stride_h, stride_q) of a bias argument (see attn_fwd_bias)."""
    if _is_tensor(bias):
        import torch
        if not bias.is_cuda or bias.dtype != torch.bfloat16:
            raise TypeError("bias must be a BF16 CUDA tensor")
        if bias.dim() != 4 or bias.shape[3] != Nk or bias.stride(3) != 1:
            raise ValueError("bias must be (Bb, Hb, Nqb, Nk) with unit stride over keys")
        Bb, Hb, Nqb, _ = bias.shape
        if Bb not in (1, B) or Hb not in (1, H) or Nqb not in (1, Nq):
            raise ValueError(f"bias shape {tuple(bias.shape)} does not broadcast to {(B, H, Nq, Nk)}")
        if bias_strides is None:
            bias_strides = tuple(bias.stride(i) if n > 1 else 0 for i, n in enumerate((Bb, Hb, Nqb)))
        bptr = bias.data_ptr()
    elif isinstance(bias, int):
        if bias_strides is None:
            raise ValueError("bias_strides are needed with an integer bias pointer")
        bptr = bias
    else:
        raise TypeError(f"bias: expected a torch tensor or an integer device pointer, got {type(bias).__name__}")
    sb, sh, sq = (int(x) for x in bias_strides)
    return bptr, sb, sh, sq


def attn_fwd_bias(q, k, v, bias, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, stream=None,
                  bias_strides=None) -> None:
    """Like :func:`attn_fwd`, with an additive bias: S = scale * Q K^T + bias.

    ``bias`` is a BF16 CUDA tensor of shape (Bb, Hb, Nqb, Nk), Bb in {1, B}, Hb in {1, H},
    Nqb in {1, Nq}, with unit stride over keys; a dimension of size 1 (or of stride 0, as
    from ``expand``) is shared. Its element strides are passed as they are, or given as
    ``bias_strides`` = (stride_b, stride_h, stride_q) when ``bias`` is an integer pointer.
    Entries of -inf remove keys; see include/attn_fwd.h for the rules.
    """
    lib = load_library()
    bptr, sb, sh, sq = _bias_arg(bias, B, H, Nq, Nk, bias_strides)
    args = (
        _ptr(q, "q", B * H * Nq * d, "bf16"), _ptr(k, "k", B * H * Nk * d, "bf16"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), bptr, sb, sh, sq, _ptr(o, "o", B * H * Nq * d, "bf16"),
        _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    rc = lib.attn_fwd_bias(*args, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                           _stream_handle(stream, q, k, v, o, lse))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_bias")


def attn_fwd_o32(q, k, v, o32, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, stream=None) -> None:
    """Like :func:`attn_fwd`, with O written as FP32 [B,H,Nq,d] (``o32``) before its rounding to
    BF16: the same kernel code, for checking the computation's own error."""
    lib = load_library()
    args = (
        _ptr(q, "q", B * H * Nq * d, "bf16"), _ptr(k, "k", B * H * Nk * d, "bf16"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), _ptr(o32, "o32", B * H * Nq * d, "f32"),
        _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    rc = lib.attn_fwd_o32(*args, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                          _stream_handle(stream, q, k, v, o32, lse))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_o32")


def attn_fwd_noalloc(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, stream=None) -> None:
    """Like :func:`attn_fwd`, for callers that cannot allocate device memory.

    The library never allocates on this path: work split between thread blocks uses a
    fixed array inside the library (see include/attn_fwd.h). Calls that run at the same
    time on the GPU share that array and must be ordered, e.g. issued on one stream.
    """
    lib = load_library()
    args = (
        _ptr(q, "q", B * H * Nq * d, "bf16"), _ptr(k, "k", B * H * Nk * d, "bf16"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), _ptr(o, "o", B * H * Nq * d, "bf16"),
        _ptr(lse, "lse", B * H * Nq, "f32"),
    )
    rc = lib.attn_fwd_noalloc(*args, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                              _stream_handle(stream, q, k, v, o, lse))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_noalloc")


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
             stream=None, causal: bool = False, bias=None, bias_strides=None) -> None:
    """Enqueue the gradients dQ, dK, dV of the forward for upstream gradient ``dout`` (see
    include/attn_bwd.h). q, o, dout, dq: BF16 [B,H,Nq,d]; k, v, dk, dv: BF16 [B,H,Nk,d];
    lse: the forward's FP32 [B,H,Nq]. CUDA tensors or integer device pointers. causal: of
    the causal forward (attn_bwd_causal). bias: of the biased forward (attn_bwd_bias; the
    bias as in :func:`attn_fwd_bias`, held fixed; not with causal)."""
    lib = load_library()
    if bias is not None and causal:
        raise ValueError("bias and causal together are not supported (put the mask in the bias)")
    args = (
        _ptr(q, "q", B * H * Nq * d, "bf16"), _ptr(k, "k", B * H * Nk * d, "bf16"),
        _ptr(v, "v", B * H * Nk * d, "bf16"), _ptr(o, "o", B * H * Nq * d, "bf16"),
        _ptr(dout, "dout", B * H * Nq * d, "bf16"), _ptr(lse, "lse", B * H * Nq, "f32"),
        _ptr(dq, "dq", B * H * Nq * d, "bf16"), _ptr(dk, "dk", B * H * Nk * d, "bf16"),
        _ptr(dv, "dv", B * H * Nk * d, "bf16"),
    )
    tail = (int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
            _stream_handle(stream, q, k, v, o, dout, lse, dq, dk, dv))
    if bias is not None:
        name = "attn_bwd_bias"
        rc = lib.attn_bwd_bias(*args[:6], *_bias_arg(bias, B, H, Nq, Nk, bias_strides), *args[6:], *tail)
    else:
        name = "attn_bwd_causal" if causal else "attn_bwd"
        rc = getattr(lib, name)(*args, *tail)
    if rc != ATTN_OK:
        raise AttnError(rc, name)


def attn_bwd_causal(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                    stream=None) -> None:
    """:func:`attn_bwd` of the causal forward (query i sees keys 0 .. i + Nk - Nq; Nq <= Nk)."""
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, stream, causal=True)


def attn_bwd_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the backward kernels' timeout status."""
    return load_library().attn_bwd_status(_stream_handle(stream))


def attn_bwd_set_wait_limit(cycles: int = 0, withhold_tile: bool = False) -> None:
    """Test hook: per-wait time limit of backward launches in SM cycles (0 = default) and the
    withheld-tile switch."""
    load_library().attn_bwd_set_wait_limit(int(cycles), 1 if withhold_tile else 0)


def attn_bwd_kernel_count() -> int:
    """Backward kernel launches made by the library in this process."""
    return int(load_library().attn_bwd_kernel_count())


def attn_fwd_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device's timeout status."""
    return load_library().attn_fwd_status(_stream_handle(stream))


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_fwd_set_wait_limit(cycles: int = 0, withhold_tile: bool = False) -> None:
    """Test hook: per-wait time limit in SM cycles (0 = default) and the withheld-tile switch."""
    load_library().attn_fwd_set_wait_limit(int(cycles), 1 if withhold_tile else 0)


def attn_fwd_kernel_count() -> int:
    """Kernel launches made by the library in this process."""
    return int(load_library().attn_fwd_kernel_count())


def attention(q, k, v, scale: float | None = None, stream=None):
    """Allocate O and LSE with torch and run :func:`attn_fwd` on [B,H,N,128] BF16 CUDA tensors."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, stream)
    return o, lse

"""The C-ABI library on a host without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import math
import os
import re

import pytest

import dense_attention_forward_fwd_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_fwd.h")
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+|unsigned\s+long\s+long\s+)?[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(",
                                text, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_causal", "attn_fwd_bias", "attn_fwd_fp8qk", "attn_fwd_fp8", "attn_fwd_o32", "attn_fwd_noalloc", "attn_bwd", "attn_bwd_causal",
            "attn_fwd_fp8qk_causal", "attn_fwd_fp8_causal", "attn_fwd_mxfp8", "attn_fwd_mxfp8_causal",
            "attn_fwd_fp8qk_bias", "attn_fwd_fp8_bias", "attn_bwd_bias",
            "attn_bwd_status", "attn_bwd_set_wait_limit",
            "attn_bwd_kernel_count", "attn_fwd_status", "attn_status_string",
            "attn_fwd_set_wait_limit", "attn_fwd_kernel_count"} <= set(names)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(attn.load_library()._name)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in attn_fwd.h but not exported"


def test_status_strings():
    for code, name in [(0, "ATTN_OK"), (-1, "ATTN_ERR_INVALID_ARG"), (-2, "ATTN_ERR_UNSUPPORTED"),
                       (-3, "ATTN_ERR_MISALIGNED"), (-4, "ATTN_ERR_CUDA"), (-5, "ATTN_ERR_TIMEOUT")]:
        assert attn.attn_status_string(code) == name
    assert attn.attn_status_string(7) == "ATTN_ERR_UNKNOWN"


def test_header_codes_match_binding():
    text = open(HEADER).read()
    for name in ["ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED",
                 "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT"]:
        m = re.search(rf"#define\s+{name}\s+\(?(-?\d+)\)?", text)
        assert m and int(m.group(1)) == getattr(attn, name)


A = 1 << 20  # fake, 16-byte aligned addresses: every call below is rejected before any CUDA call


def call(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125):
    return attn.load_library().attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=A + 8), attn.ATTN_ERR_MISALIGNED),    # FP32 rows are stored in 16-byte vectors
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0, q=None, o=None), attn.ATTN_OK),
])
def test_o32_rejects_like_attn_fwd(kw, code):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125)
    a.update(kw)
    lib = attn.load_library()
    assert lib.attn_fwd_o32(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                            a["scale"], None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Nk=-3), attn.ATTN_ERR_INVALID_ARG),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.inf), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=160), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=320), attn.ATTN_ERR_UNSUPPORTED),
    # head dimensions above 128 (the one-Q-tile kernel): the same checks, before any CUDA call
    (dict(d=256, q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=192, Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=256, scale=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=256, k=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(d=192, lse=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(d=256, B=1 << 16, H=1 << 16), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=256, B=0, q=None, o=None), attn.ATTN_OK),
    (dict(q=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(v=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(o=A + 4), attn.ATTN_ERR_MISALIGNED),
    (dict(lse=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 16), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=0, q=None, o=None), attn.ATTN_OK),        # empty batch: nothing read or written
    (dict(Nq=0, lse=None), attn.ATTN_OK),
    (dict(H=0, Nk=0), attn.ATTN_OK),
])
def test_argument_checks(kw, code):
    assert call(**kw) == code


def call_causal(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125):
    return attn.load_library().attn_fwd_causal(q, k, v, o, lse, B, H, Nq, Nk, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=129, Nk=128), attn.ATTN_ERR_INVALID_ARG),   # a query row would see no key
    (dict(Nq=1, Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(k=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(o=A + 4), attn.ATTN_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 16), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nq=0, Nk=0, lse=None), attn.ATTN_OK),
    (dict(B=0), attn.ATTN_OK),
    # d > 128 (the one-Q-tile kernel): the same checks, before any CUDA call
    (dict(Nq=129, Nk=128, d=256), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=192, o=A + 4), attn.ATTN_ERR_MISALIGNED),
    (dict(d=256, k=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=320), attn.ATTN_ERR_UNSUPPORTED),
])
def test_causal_argument_checks(kw, code):
    before = attn.attn_fwd_kernel_count()
    assert call_causal(**kw) == code
    assert attn.attn_fwd_kernel_count() == before


def call_bias(q=A, k=A, v=A, bias=A, sb=0, sh=0, sq=128, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125):
    return attn.load_library().attn_fwd_bias(q, k, v, bias, sb, sh, sq, o, lse, B, H, Nq, Nk, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bias=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sq=-128), attn.ATTN_ERR_INVALID_ARG),
    (dict(sb=-8, B=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(sh=1 << 62, H=4), attn.ATTN_ERR_INVALID_ARG),     # the last element's offset overflows
    (dict(bias=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(sq=130, Nk=130), attn.ATTN_ERR_MISALIGNED),       # rows not on 16-byte boundaries
    (dict(sh=12, H=2), attn.ATTN_ERR_MISALIGNED),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_OK),
    (dict(Nq=0, bias=None), attn.ATTN_OK),
    # d = 192 / 256 (the one-query-tile kernel) applies the same bias rules
    (dict(d=256, bias=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=256, sq=-128), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=192, sh=1 << 62, H=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=256, bias=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(d=192, sq=130, Nk=130), attn.ATTN_ERR_MISALIGNED),
    (dict(d=256, Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=256, B=0, bias=None), attn.ATTN_OK),
])
def test_bias_argument_checks(kw, code):
    before = attn.attn_fwd_kernel_count()
    assert call_bias(**kw) == code
    assert attn.attn_fwd_kernel_count() == before


@pytest.mark.parametrize("d,kw,code", [
    (256, dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (192, dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (256, dict(o=A + 8), attn.ATTN_ERR_MISALIGNED),
    (192, dict(B=0), attn.ATTN_OK),
    (64, dict(), attn.ATTN_ERR_UNSUPPORTED),
])
def test_noalloc_argument_checks(d, kw, code):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Nq=128, Nk=128)
    args.update(kw)
    before = attn.attn_fwd_kernel_count()
    assert attn.load_library().attn_fwd_noalloc(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                                                args["H"], args["Nq"], args["Nk"], d, 0.1, None) == code
    assert attn.attn_fwd_kernel_count() == before


def call_fp8(q8=A, k8=A, v=A, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125, dq=0.01, dk=0.02,
             causal=False):
    lib = attn.load_library()
    fn = lib.attn_fwd_fp8qk_causal if causal else lib.attn_fwd_fp8qk
    return fn(q8, k8, v, o, lse, B, H, Nq, Nk, d, scale, dq, dk, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dq=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=-0.5), attn.ATTN_ERR_INVALID_ARG),
    (dict(dq=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=math.inf), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=3e38, dq=10.0, dk=10.0), attn.ATTN_ERR_INVALID_ARG),   # the combined scale overflows FP32
    (dict(scale=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(q8=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(k8=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0, q8=None), attn.ATTN_OK),
    (dict(Nq=0, lse=None), attn.ATTN_OK),
])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [128, 256])   # d = 256: the one-query-tile kernel's checks
def test_fp8qk_argument_checks(kw, code, causal, d):
    before = attn.attn_fwd_kernel_count()
    assert call_fp8(causal=causal, **dict({"d": d}, **kw)) == code
    assert attn.attn_fwd_kernel_count() == before


def test_fp8_causal_rejects_more_queries_than_keys():
    assert call_fp8(Nq=129, Nk=128, causal=True) == attn.ATTN_ERR_INVALID_ARG
    assert call_fp8pv(Nq=129, Nk=128, causal=True) == attn.ATTN_ERR_INVALID_ARG


def test_fp8qk_binding_checks_types():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):   # a CPU tensor is refused before any pointer is passed
        attn.attn_fwd_fp8qk(torch.zeros(1, 1, 128, 128, dtype=torch.uint8), A, A, A, A, 1, 1, 128, 128, 128, 0.1)
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_fp8qk(A, A, A, A, A, 1, 1, 128, 128, 128, 0.1, q_descale=0.0)


def call_fp8pv(q8=A, k8=A, vt8=A, ldv=128, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125, dq=0.01,
               dk=0.02, dv=0.03, causal=False):
    lib = attn.load_library()
    fn = lib.attn_fwd_fp8_causal if causal else lib.attn_fwd_fp8
    return fn(q8, k8, vt8, ldv, o, lse, B, H, Nq, Nk, d, scale, dq, dk, dv, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dv=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(dv=math.inf), attn.ATTN_ERR_INVALID_ARG),
    (dict(dq=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ldv=120), attn.ATTN_ERR_INVALID_ARG),              # shorter than Nk
    (dict(ldv=136, Nk=130), attn.ATTN_ERR_MISALIGNED),       # rows not on 16-byte boundaries
    (dict(ldv=1 << 60, B=1 << 10), attn.ATTN_ERR_INVALID_ARG),   # offsets overflow
    (dict(vt8=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(vt8=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_OK),
])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [128, 256])   # d = 256: the one-query-tile kernel's checks
def test_fp8_argument_checks(kw, code, causal, d):
    before = attn.attn_fwd_kernel_count()
    assert call_fp8pv(causal=causal, **dict({"d": d}, **kw)) == code
    assert attn.attn_fwd_kernel_count() == before


def call_fp8_bias(pv=False, q8=A, k8=A, v=A, ldv=128, bias=A, sb=0, sh=0, sq=128, o=A, lse=A, B=1, H=1, Nq=128,
                  Nk=128, d=128, scale=0.125, dq=0.01, dk=0.02, dv=0.03):
    lib = attn.load_library()
    if pv:
        return lib.attn_fwd_fp8_bias(q8, k8, v, ldv, bias, sb, sh, sq, o, lse, B, H, Nq, Nk, d, scale, dq, dk, dv, None)
    return lib.attn_fwd_fp8qk_bias(q8, k8, v, bias, sb, sh, sq, o, lse, B, H, Nq, Nk, d, scale, dq, dk, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bias=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sq=-128), attn.ATTN_ERR_INVALID_ARG),
    (dict(sb=1 << 62, B=2), attn.ATTN_ERR_INVALID_ARG),      # the last element's offset overflows
    (dict(bias=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(sq=100), attn.ATTN_ERR_MISALIGNED),                # rows not on 16-byte boundaries
    (dict(dq=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=3e38, dq=10.0, dk=10.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(q8=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_OK),
])
@pytest.mark.parametrize("pv", [False, True])
def test_fp8_bias_argument_checks(kw, code, pv):
    before = attn.attn_fwd_kernel_count()
    assert call_fp8_bias(pv=pv, **kw) == code
    assert attn.attn_fwd_kernel_count() == before


def test_fp8_bias_value_operand_checks():
    before = attn.attn_fwd_kernel_count()
    assert call_fp8_bias(pv=True, dv=0.0) == attn.ATTN_ERR_INVALID_ARG
    assert call_fp8_bias(pv=True, ldv=120) == attn.ATTN_ERR_INVALID_ARG
    assert call_fp8_bias(pv=True, ldv=136, Nk=130, sq=136) == attn.ATTN_ERR_MISALIGNED
    assert attn.attn_fwd_kernel_count() == before


def test_fp8_bias_binding_refuses_causal():
    with pytest.raises(ValueError):
        attn.attn_fwd_fp8qk(A, A, A, A, A, 1, 1, 128, 128, 128, 0.1, causal=True, bias=A, bias_strides=(0, 0, 128))
    with pytest.raises(ValueError):
        attn.attn_fwd_fp8(A, A, A, A, A, 1, 1, 128, 128, 128, 0.1, ldv=128, causal=True, bias=A,
                          bias_strides=(0, 0, 128))


def call_mx(q8=A, sq=A, k8=A, sk=A, vt8=A, ldv=128, svt=A, ldsv=16, o=A, lse=A, B=1, H=1, Nq=128, Nk=128, d=128,
            scale=0.125, causal=False):
    lib = attn.load_library()
    fn = lib.attn_fwd_mxfp8_causal if causal else lib.attn_fwd_mxfp8
    return fn(q8, sq, k8, sk, vt8, ldv, svt, ldsv, o, lse, B, H, Nq, Nk, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(sq=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sk=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(svt=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sq=A + 2), attn.ATTN_ERR_MISALIGNED),              # scale rows are read as words
    (dict(ldsv=0), attn.ATTN_ERR_INVALID_ARG),               # under 4 bytes per key tile
    (dict(ldsv=8), attn.ATTN_ERR_MISALIGNED),                # not a 16-byte multiple
    (dict(ldsv=16, Nk=640, ldv=640), attn.ATTN_ERR_INVALID_ARG),   # 5 key tiles need 20 bytes
    (dict(ldsv=24, Nk=640, ldv=640), attn.ATTN_ERR_MISALIGNED),
    (dict(ldv=120), attn.ATTN_ERR_INVALID_ARG),
    (dict(vt8=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(scale=math.nan), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_OK),
])
@pytest.mark.parametrize("causal", [False, True])
def test_mxfp8_argument_checks(kw, code, causal):
    before = attn.attn_fwd_kernel_count()
    assert call_mx(causal=causal, **kw) == code
    assert attn.attn_fwd_kernel_count() == before


def test_mxfp8_causal_rejects_more_queries_than_keys():
    before = attn.attn_fwd_kernel_count()
    assert call_mx(Nq=129, Nk=128, causal=True) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_kernel_count() == before


def test_bias_binding_checks_shapes():
    torch = pytest.importorskip("torch")
    with pytest.raises(TypeError):   # a CPU tensor is refused before any pointer is passed
        attn.attn_fwd_bias(A, A, A, torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16), A, A,
                           1, 1, 128, 128, 128, 0.1)
    with pytest.raises(ValueError):  # an integer pointer needs its strides
        attn.attn_fwd_bias(A, A, A, A, A, A, 1, 1, 128, 128, 128, 0.1)


def call_bwd(q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125):
    return attn.load_library().attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(do=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.inf), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(dq=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(lse=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 16), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=0), attn.ATTN_OK),
    (dict(Nq=0, Nk=0), attn.ATTN_OK),
])
def test_bwd_argument_checks(kw, code):
    before = attn.attn_bwd_kernel_count()
    assert call_bwd(**kw) == code
    assert attn.attn_bwd_kernel_count() == before


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=129, Nk=128), attn.ATTN_ERR_INVALID_ARG),   # a query row would see no key
    (dict(do=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=0), attn.ATTN_OK),
])
def test_bwd_causal_argument_checks(kw, code):
    args = dict(q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.125)
    args.update(kw)
    before = attn.attn_bwd_kernel_count()
    assert attn.load_library().attn_bwd_causal(*args.values(), None) == code
    assert attn.attn_bwd_kernel_count() == before


def test_binding_raises_on_rejected_call():
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(A, A, A, A, A, 1, 1, 128, 128, 64, 0.1)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED


def test_binding_checks_tensor_sizes():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # a CPU tensor is refused before any pointer is passed
        attn.attn_fwd(q, q, q, q, torch.zeros(1, 1, 128), 1, 1, 128, 128, 128, 0.1)


def test_no_launch_without_gpu_calls():
    before = attn.attn_fwd_kernel_count()
    call(d=64)
    assert attn.attn_fwd_kernel_count() == before


def call_bwd_bias(q=A, k=A, v=A, o=A, do=A, lse=A, bias=A, sb=0, sh=0, sq=128, dq=A, dk=A, dv=A, B=1, H=1, Nq=128,
                  Nk=128, d=128, scale=0.125):
    return attn.load_library().attn_bwd_bias(q, k, v, o, do, lse, bias, sb, sh, sq, dq, dk, dv, B, H, Nq, Nk, d, scale,
                                             None)


@pytest.mark.parametrize("kw,code", [
    (dict(bias=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sh=-8), attn.ATTN_ERR_INVALID_ARG),
    (dict(sb=1 << 62, B=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(bias=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(sq=100), attn.ATTN_ERR_MISALIGNED),
    (dict(do=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_OK),
])
def test_bwd_bias_argument_checks(kw, code):
    before = attn.attn_bwd_kernel_count()
    assert call_bwd_bias(**kw) == code
    assert attn.attn_bwd_kernel_count() == before


def test_bwd_bias_binding_refuses_causal():
    with pytest.raises(ValueError):
        attn.attn_bwd(A, A, A, A, A, A, A, A, A, 1, 1, 128, 128, 128, 0.1, causal=True, bias=A,
                      bias_strides=(0, 0, 128))


def plan(n_groups, n_kv, sms=152):
    lib = attn.load_library()
    fn = lib.attn_fwd_plan
    dp = ctypes.c_longlong()
    cuts = (ctypes.c_longlong * 161)()
    grid, split = ctypes.c_int(), ctypes.c_int()
    assert fn(ctypes.c_longlong(n_groups), n_kv, sms, ctypes.byref(dp), cuts, ctypes.byref(grid), ctypes.byref(split)) == 0
    return dp.value, list(cuts)[:grid.value + 1], grid.value, bool(split.value)


@pytest.mark.parametrize("n_groups,n_kv", [(128, 64), (8, 8), (1, 1), (3, 40), (152, 32), (1024, 32), (300, 17),
                                           (151, 128), (64, 128), (2, 3)])
def test_plan_shares_cover_the_split_region(n_groups, n_kv):
    # the shares partition the split region in order, every one non-empty
    dp, cuts, grid, split = plan(n_groups, n_kv)
    total = (n_groups - dp) * n_kv
    assert 1 <= grid <= 152 and dp % 152 == 0 and dp <= n_groups
    if total == 0:
        return
    assert cuts[0] == 0 and cuts[-1] == total and len(cuts) == grid + 1
    assert all(b > a for a, b in zip(cuts, cuts[1:]))
    assert split == any(c % n_kv != 0 for c in cuts[1:-1])
    if dp > 0:
        assert grid == 152


def test_plan_shares_are_even():
    # rect-4k-8k's 128 groups of 64 steps on 152 blocks: shares of 53 or 54 steps
    dp, cuts, grid, split = plan(128, 64)
    assert dp == 0 and split and grid == 152
    sizes = [b - a for a, b in zip(cuts, cuts[1:])]
    assert set(sizes) <= {53, 54}


def test_plan_rejects_bad_arguments():
    lib = attn.load_library()
    assert lib.attn_fwd_plan(ctypes.c_longlong(0), 1, 152, None, None, None, None) == attn.ATTN_ERR_INVALID_ARG

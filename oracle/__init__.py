"""FP64 CPU oracle for dense scaled-dot-product attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library under test never does, and
this package imports nothing from it: the two share no code. Inputs are BF16
bit patterns (uint16 numpy arrays), or for the 8-bit functions E4M3 codes and E8M0
block scales (uint8 arrays), as produced by the seeded generators; the oracle decodes
the 8-bit formats itself.

The arithmetic lives in ``attn_ref.c`` (plain C, double precision, OpenMP over
query rows); this module compiles it with gcc on first use and marshals numpy
arrays. See ``attn_ref.c`` for the definition it follows and its citations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = ["build", "Oracle", "default", "attention_rows", "attention_rows_causal", "attention_rows_bias",
           "attention", "attention_dense", "attention_bwd", "probs", "max_threads", "LIB_PATH",
           "attention_rows_e4m3qk", "attention_rows_e4m3", "attention_rows_mxfp8", "e4m3_to_f64", "e8m0_to_f64"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
LIB_PATH = os.path.join(_HERE, "libattn_ref.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = LIB_PATH) -> str:
    """Compile attn_ref.c into a shared library (gcc, -O2, OpenMP when available)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """The oracle bound to one compiled copy of attn_ref.c (the default one, or a test's own build)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.attn_ref_rows_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, vp, i64, vp, vp, ctypes.c_int]
        lib.attn_ref_rows_f64.restype = ctypes.c_int
        lib.attn_ref_rows_causal_f64.argtypes = lib.attn_ref_rows_f64.argtypes
        lib.attn_ref_rows_causal_f64.restype = ctypes.c_int
        lib.attn_ref_rows_bias_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, i64, dbl,
                                               vp, i64, vp, vp, ctypes.c_int]
        lib.attn_ref_rows_bias_f64.restype = ctypes.c_int
        lib.attn_ref_rows_e4m3qk_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, dbl, dbl, vp, i64, vp,
                                                 vp, ctypes.c_int]
        lib.attn_ref_rows_e4m3qk_f64.restype = ctypes.c_int
        lib.attn_ref_rows_e4m3qk_causal_f64.argtypes = lib.attn_ref_rows_e4m3qk_f64.argtypes
        lib.attn_ref_rows_e4m3qk_causal_f64.restype = ctypes.c_int
        lib.attn_ref_rows_e4m3_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, dbl, dbl, dbl, vp, i64,
                                               vp, vp, ctypes.c_int]
        lib.attn_ref_rows_e4m3_f64.restype = ctypes.c_int
        lib.attn_ref_rows_e4m3_causal_f64.argtypes = lib.attn_ref_rows_e4m3_f64.argtypes
        lib.attn_ref_rows_e4m3_causal_f64.restype = ctypes.c_int
        bias_args = [vp, i64, i64, i64, i64]   # bias, H, sb, sh, sq after the three operands
        lib.attn_ref_rows_e4m3qk_bias_f64.argtypes = (lib.attn_ref_rows_e4m3qk_f64.argtypes[:3] + bias_args
                                                      + lib.attn_ref_rows_e4m3qk_f64.argtypes[3:])
        lib.attn_ref_rows_e4m3qk_bias_f64.restype = ctypes.c_int
        lib.attn_ref_rows_e4m3_bias_f64.argtypes = (lib.attn_ref_rows_e4m3_f64.argtypes[:3] + bias_args
                                                    + lib.attn_ref_rows_e4m3_f64.argtypes[3:])
        lib.attn_ref_rows_e4m3_bias_f64.restype = ctypes.c_int
        lib.attn_ref_rows_mxfp8_f64.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, vp, i64, vp,
                                                vp, ctypes.c_int]
        lib.attn_ref_rows_mxfp8_f64.restype = ctypes.c_int
        lib.attn_ref_rows_mxfp8_causal_f64.argtypes = lib.attn_ref_rows_mxfp8_f64.argtypes
        lib.attn_ref_rows_mxfp8_causal_f64.restype = ctypes.c_int
        lib.attn_ref_e8m0_to_f64.argtypes = [vp, i64, vp]
        lib.attn_ref_e8m0_to_f64.restype = None
        lib.attn_ref_e4m3_to_f64.argtypes = [vp, i64, vp]
        lib.attn_ref_e4m3_to_f64.restype = None
        lib.attn_ref_dense_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, vp, vp]
        lib.attn_ref_dense_f64.restype = ctypes.c_int
        lib.attn_ref_bwd_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, vp, vp, vp, ctypes.c_int]
        lib.attn_ref_bwd_f64.restype = ctypes.c_int
        lib.attn_ref_dense_causal_f64.argtypes = lib.attn_ref_dense_f64.argtypes
        lib.attn_ref_dense_causal_f64.restype = ctypes.c_int
        lib.attn_ref_bwd_causal_f64.argtypes = lib.attn_ref_bwd_f64.argtypes
        lib.attn_ref_bwd_causal_f64.restype = ctypes.c_int
        dense_bias = [vp, i64, i64, i64, i64]   # bias, H, sb, sh, sq
        lib.attn_ref_dense_bias_f64.argtypes = lib.attn_ref_dense_f64.argtypes[:3] + dense_bias + \
            lib.attn_ref_dense_f64.argtypes[3:]
        lib.attn_ref_dense_bias_f64.restype = ctypes.c_int
        lib.attn_ref_bwd_bias_f64.argtypes = lib.attn_ref_bwd_f64.argtypes[:4] + dense_bias + \
            lib.attn_ref_bwd_f64.argtypes[4:]
        lib.attn_ref_bwd_bias_f64.restype = ctypes.c_int
        lib.attn_ref_probs_f64.argtypes = [vp, vp, i64, i64, i64, i64, dbl, vp]
        lib.attn_ref_probs_f64.restype = ctypes.c_int
        lib.attn_ref_max_threads.argtypes = []
        lib.attn_ref_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def max_threads(self) -> int:
        return self.lib.attn_ref_max_threads()

    def attention_rows(self, q, k, v, scale: float, rows=None, nthreads: int = 0):
        """O and LSE (float64) for selected query rows.

        q [B,H,Nq,d], k [B,H,Nk,d], v [B,H,Nk,dv] as uint16 BF16 bits. ``rows`` holds
        flat ids ``(b*H + h)*Nq + i``; None means every row. Returns
        (o [len(rows), dv], lse [len(rows)]).
        """
        q, k, v = _u16(q, 4), _u16(k, 4), _u16(v, 4)
        B, H, Nq, d = q.shape
        Nk, dv = k.shape[2], v.shape[3]
        if k.shape != (B, H, Nk, d) or v.shape[:3] != (B, H, Nk):
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
        if rows is None:
            rows = np.arange(B * H * Nq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, dv), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        rc = self.lib.attn_ref_rows_f64(_ptr(q), _ptr(k), _ptr(v), B * H, Nq, Nk, d, dv, float(scale),
                                        _ptr(rows), rows.size, _ptr(o), _ptr(lse), int(nthreads))
        if rc != 0:
            raise ValueError(f"attn_ref_rows_f64 failed with status {rc}")
        return o, lse

    def attention_rows_causal(self, q, k, v, scale: float, rows=None, nthreads: int = 0):
        """As attention_rows, under the causal mask: query i sees keys 0 .. i + Nk - Nq
        (bottom-right alignment; needs Nq <= Nk)."""
        q, k, v = _u16(q, 4), _u16(k, 4), _u16(v, 4)
        B, H, Nq, d = q.shape
        Nk, dv = k.shape[2], v.shape[3]
        if k.shape != (B, H, Nk, d) or v.shape[:3] != (B, H, Nk):
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
        if rows is None:
            rows = np.arange(B * H * Nq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, dv), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        rc = self.lib.attn_ref_rows_causal_f64(_ptr(q), _ptr(k), _ptr(v), B * H, Nq, Nk, d, dv, float(scale),
                                               _ptr(rows), rows.size, _ptr(o), _ptr(lse), int(nthreads))
        if rc != 0:
            raise ValueError(f"attn_ref_rows_causal_f64 failed with status {rc}")
        return o, lse

    @staticmethod
    def _bias_strides(bias, B, H, Nq, Nk):
        """(bias as uint16 [Bb,Hb,Nqb,Nk], sb, sh, sq) for a bias that broadcasts to [B,H,Nq,Nk]."""
        bias = _u16(bias, 4)
        Bb, Hb, Nqb, Nkb = bias.shape
        if Bb not in (1, B) or Hb not in (1, H) or Nqb not in (1, Nq) or Nkb != Nk:
            raise ValueError(f"bias shape {bias.shape} does not broadcast to {(B, H, Nq, Nk)}")
        sb, sh, sq = (st // 2 if n > 1 else 0 for st, n in zip(bias.strides[:3], (Bb, Hb, Nqb)))
        return bias, sb, sh, sq

    def attention_rows_bias(self, q, k, v, bias, scale: float, rows=None, nthreads: int = 0):
        """As attention_rows, with the additive bias B: S = scale * Q K^T + B.

        ``bias`` holds BF16 bits (uint16) of shape (Bb, Hb, Nqb, Nk) with Bb in {1, B},
        Hb in {1, H}, Nqb in {1, Nq}; a dimension of size 1 is repeated (numpy
        broadcasting). A C-contiguous view into a larger buffer is used in place.
        """
        q, k, v, bias = _u16(q, 4), _u16(k, 4), _u16(v, 4), _u16(bias, 4)
        B, H, Nq, d = q.shape
        Nk, dv = k.shape[2], v.shape[3]
        if k.shape != (B, H, Nk, d) or v.shape[:3] != (B, H, Nk):
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
        Bb, Hb, Nqb, Nkb = bias.shape
        if Bb not in (1, B) or Hb not in (1, H) or Nqb not in (1, Nq) or Nkb != Nk:
            raise ValueError(f"bias shape {bias.shape} does not broadcast to {(B, H, Nq, Nk)}")
        sb, sh, sq = (st // 2 if n > 1 else 0 for st, n in zip(bias.strides[:3], (Bb, Hb, Nqb)))
        if rows is None:
            rows = np.arange(B * H * Nq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, dv), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        rc = self.lib.attn_ref_rows_bias_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), H, sb, sh, sq, B * H, Nq, Nk,
                                             d, dv, float(scale), _ptr(rows), rows.size, _ptr(o), _ptr(lse),
                                             int(nthreads))
        if rc != 0:
            raise ValueError(f"attn_ref_rows_bias_f64 failed with status {rc}")
        return o, lse

    def e4m3_to_f64(self, codes):
        """Values of FP8 E4M3 codes (uint8 array of any shape) as float64 (NaN for the NaN codes)."""
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.attn_ref_e4m3_to_f64(_ptr(c), c.size, _ptr(out))
        return out

    def attention_rows_e4m3qk(self, q8, k8, v, scale: float, q_descale: float = 1.0, k_descale: float = 1.0,
                              rows=None, nthreads: int = 0, causal: bool = False, bias=None):
        """As attention_rows with Q and K given as FP8 E4M3 codes (uint8 [B,H,N,d]) and their
        per-tensor descale factors: the scores are scale * (q_descale Q8)(k_descale K8)^T.
        causal: under the causal mask of attention_rows_causal (needs Nq <= Nk). bias: the
        additive B of attention_rows_bias (same shapes and broadcasting; not with causal)."""
        q8 = np.ascontiguousarray(q8)
        k8 = np.ascontiguousarray(k8)
        if q8.dtype != np.uint8 or k8.dtype != np.uint8:
            raise TypeError("q8 and k8 must be uint8 E4M3 codes")
        v = _u16(v, 4)
        B, H, Nq, d = q8.shape
        Nk, dv = k8.shape[2], v.shape[3]
        if k8.shape != (B, H, Nk, d) or v.shape[:3] != (B, H, Nk):
            raise ValueError(f"shape mismatch q8{q8.shape} k8{k8.shape} v{v.shape}")
        if rows is None:
            rows = np.arange(B * H * Nq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, dv), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        tail = (B * H, Nq, Nk, d, dv, float(scale), float(q_descale), float(k_descale), _ptr(rows), rows.size,
                _ptr(o), _ptr(lse), int(nthreads))
        if bias is not None:
            if causal:
                raise ValueError("bias and causal together are not supported (put the mask in the bias)")
            bias, sb, sh, sq = self._bias_strides(bias, B, H, Nq, Nk)
            rc = self.lib.attn_ref_rows_e4m3qk_bias_f64(_ptr(q8), _ptr(k8), _ptr(v), _ptr(bias), H, sb, sh, sq, *tail)
        else:
            fn = self.lib.attn_ref_rows_e4m3qk_causal_f64 if causal else self.lib.attn_ref_rows_e4m3qk_f64
            rc = fn(_ptr(q8), _ptr(k8), _ptr(v), *tail)
        if rc != 0:
            raise ValueError(f"attn_ref_rows_e4m3qk_f64 failed with status {rc}")
        return o, lse

    def attention_rows_e4m3(self, q8, k8, v8, scale: float, q_descale: float = 1.0, k_descale: float = 1.0,
                            v_descale: float = 1.0, rows=None, nthreads: int = 0, causal: bool = False, bias=None):
        """As attention_rows_e4m3qk with V given as E4M3 codes too (uint8 [B,H,Nk,dv], real
        values v_descale * V8); P is not rounded: this is the definition on the real inputs.
        causal: under the causal mask of attention_rows_causal (needs Nq <= Nk). bias: the
        additive B of attention_rows_bias (not with causal)."""
        q8, k8, v8 = (np.ascontiguousarray(a) for a in (q8, k8, v8))
        if q8.dtype != np.uint8 or k8.dtype != np.uint8 or v8.dtype != np.uint8:
            raise TypeError("q8, k8 and v8 must be uint8 E4M3 codes")
        B, H, Nq, d = q8.shape
        Nk, dv = k8.shape[2], v8.shape[3]
        if k8.shape != (B, H, Nk, d) or v8.shape[:3] != (B, H, Nk):
            raise ValueError(f"shape mismatch q8{q8.shape} k8{k8.shape} v8{v8.shape}")
        if rows is None:
            rows = np.arange(B * H * Nq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, dv), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        tail = (B * H, Nq, Nk, d, dv, float(scale), float(q_descale), float(k_descale), float(v_descale),
                _ptr(rows), rows.size, _ptr(o), _ptr(lse), int(nthreads))
        if bias is not None:
            if causal:
                raise ValueError("bias and causal together are not supported (put the mask in the bias)")
            bias, sb, sh, sq = self._bias_strides(bias, B, H, Nq, Nk)
            rc = self.lib.attn_ref_rows_e4m3_bias_f64(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(bias), H, sb, sh, sq, *tail)
        else:
            fn = self.lib.attn_ref_rows_e4m3_causal_f64 if causal else self.lib.attn_ref_rows_e4m3_f64
            rc = fn(_ptr(q8), _ptr(k8), _ptr(v8), *tail)
        if rc != 0:
            raise ValueError(f"attn_ref_rows_e4m3_f64 failed with status {rc}")
        return o, lse

    def e8m0_to_f64(self, codes):
        """Values 2^(e - 127) of E8M0 scale codes (uint8 array of any shape); NaN for 255."""
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.attn_ref_e8m0_to_f64(_ptr(c), c.size, _ptr(out))
        return out

    def attention_rows_mxfp8(self, q8, sq, k8, sk, v8, sv, scale: float, rows=None, nthreads: int = 0,
                             causal: bool = False):
        """O and LSE (float64) of selected rows from MXFP8 inputs: E4M3 codes q8 [B,H,Nq,d],
        k8 [B,H,Nk,d], v8 [B,H,Nk,dv] with E8M0 block scales sq [B,H,Nq,d/32] and
        sk [B,H,Nk,d/32] (32 elements along d) and sv [B,H,ceil(Nk/32),dv] (32 keys per column).
        causal: under the causal mask of attention_rows_causal (needs Nq <= Nk)."""
        arrs = [np.ascontiguousarray(a) for a in (q8, sq, k8, sk, v8, sv)]
        if any(a.dtype != np.uint8 for a in arrs):
            raise TypeError("MXFP8 codes and scales must be uint8")
        q8, sq, k8, sk, v8, sv = arrs
        B, H, Nq, d = q8.shape
        Nk, dv = k8.shape[2], v8.shape[3]
        if (k8.shape != (B, H, Nk, d) or v8.shape[:3] != (B, H, Nk) or d % 32 != 0
                or sq.shape != (B, H, Nq, d // 32) or sk.shape != (B, H, Nk, d // 32)
                or sv.shape != (B, H, (Nk + 31) // 32, dv)):
            raise ValueError(f"shape mismatch q8{q8.shape} sq{sq.shape} k8{k8.shape} sk{sk.shape} v8{v8.shape} "
                             f"sv{sv.shape}")
        if rows is None:
            rows = np.arange(B * H * Nq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.empty((rows.size, dv), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
        fn = self.lib.attn_ref_rows_mxfp8_causal_f64 if causal else self.lib.attn_ref_rows_mxfp8_f64
        rc = fn(_ptr(q8), _ptr(sq), _ptr(k8), _ptr(sk), _ptr(v8), _ptr(sv), B * H, Nq, Nk, d, dv, float(scale),
                _ptr(rows), rows.size, _ptr(o), _ptr(lse), int(nthreads))
        if rc != 0:
            raise ValueError(f"attn_ref_rows_mxfp8_f64 failed with status {rc}")
        return o, lse

    def attention(self, q, k, v, scale: float, nthreads: int = 0):
        """Full O [B,H,Nq,dv] and LSE [B,H,Nq] in float64."""
        B, H, Nq, _ = q.shape
        dv = v.shape[3]
        o, lse = self.attention_rows(q, k, v, scale, None, nthreads)
        return o.reshape(B, H, Nq, dv), lse.reshape(B, H, Nq)

    @staticmethod
    def _dense_bias(bias, B, H, Nq, Nk):
        """(float64 C-contiguous bias [Bb,Hb,Nqb,Nk], sb, sh, sq) for a float64 or BF16-bit bias
        that broadcasts to [B,H,Nq,Nk] (a dimension of size 1 is shared)."""
        bias = _f64(bias)
        Bb, Hb, Nqb, Nkb = bias.shape
        if Bb not in (1, B) or Hb not in (1, H) or Nqb not in (1, Nq) or Nkb != Nk:
            raise ValueError(f"bias shape {bias.shape} does not broadcast to {(B, H, Nq, Nk)}")
        sb, sh, sq = (st // 8 if n > 1 else 0 for st, n in zip(bias.strides[:3], (Bb, Hb, Nqb)))
        return bias, sb, sh, sq

    def attention_dense(self, q, k, v, scale: float, causal: bool = False, bias=None):
        """Forward on float64 (or BF16-bit uint16, widened exactly) inputs: (o [B,H,Nq,dv], lse [B,H,Nq]).
        causal: the causal mask of attention_rows_causal (needs Nq <= Nk). bias: the additive
        B of attention_rows_bias, float64 or BF16 bits (not with causal)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Nq, d = q.shape
        Nk, dv = k.shape[2], v.shape[3]
        if k.shape != (B, H, Nk, d) or v.shape[:3] != (B, H, Nk):
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
        o = np.empty((B, H, Nq, dv), dtype=np.float64)
        lse = np.empty((B, H, Nq), dtype=np.float64)
        tail = (B * H, Nq, Nk, d, dv, float(scale), _ptr(o), _ptr(lse))
        if bias is not None:
            if causal:
                raise ValueError("bias and causal together are not supported (put the mask in the bias)")
            bias, sb, sh, sq = self._dense_bias(bias, B, H, Nq, Nk)
            rc = self.lib.attn_ref_dense_bias_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), H, sb, sh, sq, *tail)
        else:
            fn = self.lib.attn_ref_dense_causal_f64 if causal else self.lib.attn_ref_dense_f64
            rc = fn(_ptr(q), _ptr(k), _ptr(v), *tail)
        if rc != 0:
            raise ValueError(f"attn_ref_dense_f64 failed with status {rc}")
        return o, lse

    def attention_bwd(self, q, k, v, dout, scale: float, nthreads: int = 0, causal: bool = False, bias=None):
        """Gradients (dq, dk, dv) in float64 of the forward for upstream gradient dout [B,H,Nq,dv].

        Inputs are float64 arrays, or BF16 bits (uint16) widened exactly. causal: of the
        causal forward (needs Nq <= Nk). bias: of the biased forward (as attention_dense), the
        bias held fixed."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, Nq, d = q.shape
        Nk, dv = k.shape[2], v.shape[3]
        if k.shape != (B, H, Nk, d) or v.shape[:3] != (B, H, Nk) or dout.shape != (B, H, Nq, dv):
            raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape} dout{dout.shape}")
        dq = np.empty((B, H, Nq, d), dtype=np.float64)
        dk = np.empty((B, H, Nk, d), dtype=np.float64)
        dvv = np.empty((B, H, Nk, dv), dtype=np.float64)
        tail = (B * H, Nq, Nk, d, dv, float(scale), _ptr(dq), _ptr(dk), _ptr(dvv), int(nthreads))
        if bias is not None:
            if causal:
                raise ValueError("bias and causal together are not supported (put the mask in the bias)")
            bias, sb, sh, sq = self._dense_bias(bias, B, H, Nq, Nk)
            rc = self.lib.attn_ref_bwd_bias_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(bias), H, sb, sh, sq,
                                                *tail)
        else:
            fn = self.lib.attn_ref_bwd_causal_f64 if causal else self.lib.attn_ref_bwd_f64
            rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), *tail)
        if rc != 0:
            raise ValueError(f"attn_ref_bwd_f64 failed with status {rc}")
        return dq, dk, dvv

    def probs(self, q, k, scale: float):
        """Full P = softmax_row(scale * Q K^T) as float64 [B,H,Nq,Nk] (small shapes only)."""
        q, k = _u16(q, 4), _u16(k, 4)
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        p = np.empty((B, H, Nq, Nk), dtype=np.float64)
        rc = self.lib.attn_ref_probs_f64(_ptr(q), _ptr(k), B * H, Nq, Nk, d, float(scale), _ptr(p))
        if rc != 0:
            raise ValueError(f"attn_ref_probs_f64 failed with status {rc}")
        return p


def default() -> Oracle:
    """The oracle built from this directory's attn_ref.c (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = Oracle(LIB_PATH)
    return _lib


def _u16(a: np.ndarray, ndim: int) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns as uint16, got {a.dtype}")
    if a.ndim != ndim:
        raise ValueError(f"expected {ndim} dims, got shape {a.shape}")
    return a


def _f64(a: np.ndarray) -> np.ndarray:
    """float64 C-contiguous copy of a float array, or of BF16 bits (uint16) widened exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if a.ndim != 4:
        raise ValueError(f"expected 4 dims, got shape {a.shape}")
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return default().max_threads()


def attention_rows(q, k, v, scale: float, rows=None, nthreads: int = 0):
    return default().attention_rows(q, k, v, scale, rows, nthreads)


def attention_rows_causal(q, k, v, scale: float, rows=None, nthreads: int = 0):
    return default().attention_rows_causal(q, k, v, scale, rows, nthreads)


def attention_rows_bias(q, k, v, bias, scale: float, rows=None, nthreads: int = 0):
    return default().attention_rows_bias(q, k, v, bias, scale, rows, nthreads)


def e4m3_to_f64(codes):
    return default().e4m3_to_f64(codes)


def attention_rows_e4m3qk(q8, k8, v, scale: float, q_descale: float = 1.0, k_descale: float = 1.0, rows=None,
                          nthreads: int = 0, causal: bool = False, bias=None):
    return default().attention_rows_e4m3qk(q8, k8, v, scale, q_descale, k_descale, rows, nthreads, causal, bias)


def attention_rows_e4m3(q8, k8, v8, scale: float, q_descale: float = 1.0, k_descale: float = 1.0,
                        v_descale: float = 1.0, rows=None, nthreads: int = 0, causal: bool = False, bias=None):
    return default().attention_rows_e4m3(q8, k8, v8, scale, q_descale, k_descale, v_descale, rows, nthreads,
                                         causal, bias)


def e8m0_to_f64(codes):
    return default().e8m0_to_f64(codes)


def attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, scale: float, rows=None, nthreads: int = 0, causal: bool = False):
    return default().attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, scale, rows, nthreads, causal)


def attention(q, k, v, scale: float, nthreads: int = 0):
    return default().attention(q, k, v, scale, nthreads)


def probs(q, k, scale: float):
    return default().probs(q, k, scale)


def attention_dense(q, k, v, scale: float, causal: bool = False, bias=None):
    return default().attention_dense(q, k, v, scale, causal, bias)


def attention_bwd(q, k, v, dout, scale: float, nthreads: int = 0, causal: bool = False, bias=None):
    return default().attention_bwd(q, k, v, dout, scale, nthreads, causal, bias)

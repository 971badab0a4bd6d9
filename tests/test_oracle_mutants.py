"""The oracle's pins must catch plausible slips: each mutant below plants one in a private
copy of attn_ref.c (compiled into a temporary directory, on the CPU; at every occurrence
of the mutated text) and at least one pin of tests/test_oracle.py must fail against it.
The committed oracle is never modified.
"""
import os
import shutil

import pytest

import oracle
from test_oracle import PINS

MUTANTS = {
    "scale dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "exponent sign flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "missing 1/l": ("o[c] = acc / l;", "o[c] = acc;"),
    "max not added back to lse": ("*lse = m + log(l);", "*lse = log(l);"),
    "log2 instead of ln": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "value rows with key stride": ("vh[j * dv + c]", "vh[j * d + c]"),
    "key head stride uses Nq": ("k + bh * Nk * d, v", "k + bh * Nq * d, v"),
    "query row stride uses Nk": ("attend_row(q + (bh * Nq + i) * d", "attend_row(q + (bh * Nk + i) * d"),
    "minimum instead of maximum": ("if (s[j] > m) m = s[j];", "if (s[j] < m) m = s[j];"),
    "last key dropped from PV": ("for (int64_t j = 0; j < Nk; j++)\n            acc += s[j]",
                                 "for (int64_t j = 0; j < Nk - 1; j++)\n            acc += s[j]"),
    "keys used as values": ("bf16_to_f64(vh[j * dv + c])", "bf16_to_f64(kh[j * d + c])"),
    "causal mask one key short": ("int64_t visible = i + (Nk - Nq) + 1;", "int64_t visible = i + (Nk - Nq) + (i > 0);"),
    "causal mask aligned top-left": ("int64_t visible = i + (Nk - Nq) + 1;", "int64_t visible = i + 1;"),
    "bias ignored": ("s[j] += bf16_to_f64(bh_bias[i * sq + j]);", "s[j] += 0.0;"),
    "bias inside the scale": ("s[j] += bf16_to_f64(bh_bias[i * sq + j]);",
                              "s[j] += scale * bf16_to_f64(bh_bias[i * sq + j]);"),
    "bias transposed": ("bh_bias[i * sq + j]", "bh_bias[j * sq + i]"),
    "bias row stride dropped": ("bh_bias[i * sq + j]", "bh_bias[j]"),
    "bias head and batch strides swapped": ("bias + (bh / H) * sb + (bh % H) * sh", "bias + (bh / H) * sh + (bh % H) * sb"),
    "bwd row term D dropped": ("double ds = p[j] * (dp[j] - D);", "double ds = p[j] * dp[j];"),
    "bwd dq without the scale": ("dqi[c] += scale * ds * kh[j * d + c];", "dqi[c] += ds * kh[j * d + c];"),
    "bwd dk from keys": ("dkh[j * d + c] += scale * ds * qi[c];", "dkh[j * d + c] += scale * ds * kh[j * d + c];"),
    "bwd dv from dp": ("dvh[j * dv + c] += p[j] * doi[c];", "dvh[j * dv + c] += dp[j] * doi[c];"),
    "bwd probabilities not normalised": ("for (int64_t j = 0; j < nvis; j++) p[j] /= l;", ""),
    "dense forward without 1/l": ("oi[c] = acc / l;", "oi[c] = acc;"),
    "causal bwd mask half offset": ("nvis = causal ? i + (Nk - Nq) + 1", "nvis = causal ? i + (Nk - Nq) / 2 + 1"),
    "e4m3 exponent bias 8": ("mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3 subnormals one binade low": ("ldexp((double)m / 8.0, 1 - 7)", "ldexp((double)m / 8.0, -7)"),
    "e4m3 sign dropped": ("return sign ? -mag : mag;", "return mag;"),
    "e4m3 mantissa without the implicit one": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp((double)m / 8.0, e - 7)"),
    "e4m3 key descale dropped": ("(k_descale * e4m3_to_f64(kh[j * d + c]))", "(e4m3_to_f64(kh[j * d + c]))"),
    "e4m3 query descale squared": ("(q_descale * e4m3_to_f64(qi[c]))", "(q_descale * q_descale * e4m3_to_f64(qi[c]))"),
    "e4m3 values from the keys": ("num += s[j] * bf16_to_f64(vrows[j * dv + c]);",
                                  "num += s[j] * (double)kh[j * d + c];"),
    "e4m3 value descale dropped": ("(v_descale * e4m3_to_f64(vhead[j * dv + c]))", "(e4m3_to_f64(vhead[j * dv + c]))"),
    "e4m3 value rows with the key stride": ("vhead[j * dv + c]", "vhead[j * d + c]"),
    "mx scale bias 128": ("return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 128);"),
    "mx key scales taken from the query": ("(e8m0_to_f64(ks[j * db + c / 32]) * e4m3_to_f64(kh[j * d + c]))",
                                           "(e8m0_to_f64(qs[c / 32]) * e4m3_to_f64(kh[j * d + c]))"),
    "mx value scales ignored": ("(e8m0_to_f64(vs[(j / 32) * dv + c]) * e4m3_to_f64(vh[j * dv + c]))",
                                "(1.0 * e4m3_to_f64(vh[j * dv + c]))"),
    "mx query scales of the first block only": ("(e8m0_to_f64(qs[c / 32]) * e4m3_to_f64(qi[c]))",
                                                "(e8m0_to_f64(qs[0]) * e4m3_to_f64(qi[c]))"),
    "bwd bias ignored": ("for (int64_t j = 0; j < nvis; j++) p[j] += brow[j];",
                         "for (int64_t j = 0; j < nvis; j++) p[j] += 0.0;"),
    "bwd bias rows transposed": ("const double *brow = dbias_row(bias, bh, i);", "const double *brow = dbias_row(bias, bh, 0);"),
    "dense bias ignored": ("for (int64_t j = 0; j < nv; j++) s[j] += bi[j];", "for (int64_t j = 0; j < nv; j++) s[j] += 0.0;"),
    "double bias head and batch strides swapped": ("(bh / b->H) * b->sb + (bh % b->H) * b->sh",
                                                   "(bh / b->H) * b->sh + (bh % b->H) * b->sb"),
    "e4m3 bias ignored": ("for (int64_t j = 0; j < nk; j++) s[j] += bf16_to_f64(brow[j]);",
                          "for (int64_t j = 0; j < nk; j++) s[j] += 0.0;"),
    "e4m3 bias row stride dropped": ("(bh % H) * sh + i * sq;\n                    for (int64_t j = 0; j < nk; j++) s[j]",
                                     "(bh % H) * sh;\n                    for (int64_t j = 0; j < nk; j++) s[j]"),
    "e4m3 bias head and batch strides swapped": ("const uint16_t *brow = bias + (bh / H) * sb + (bh % H) * sh",
                                                 "const uint16_t *brow = bias + (bh / H) * sh + (bh % H) * sb"),
    "e4m3-value bias ignored": ("for (int64_t j = 0; j < nk; j++) w[j] += bf16_to_f64(bq[j]);",
                                "for (int64_t j = 0; j < nk; j++) w[j] += 0.0;"),
    "e4m3-value bias scaled": ("w[j] += bf16_to_f64(bq[j]);", "w[j] += scale * bf16_to_f64(bq[j]);"),
    "e4m3 causal mask one key short": ("const int64_t nk = causal ? i + (Nk - Nq) + 1 : Nk;",
                                       "const int64_t nk = causal ? i + (Nk - Nq) + (i > 0) : Nk;"),
    "e4m3 causal mask aligned top-left": ("const int64_t nk = causal ? i + (Nk - Nq) + 1 : Nk;",
                                          "const int64_t nk = causal ? i + 1 : Nk;"),
    "e4m3-value and mx causal masks ignored": ("const int64_t nk = causal ? i + (Nk - Nq) + 1 : Nk;   /* the row's keys */\n                /* step 1 on the real inputs */\n                for (int64_t j = 0; j < nk; j++) {\n                    double dot",
                               "const int64_t nk = Nk;\n                /* step 1 on the real inputs */\n                for (int64_t j = 0; j < nk; j++) {\n                    double dot"),
    "causal dense forward one key short": ("const int64_t nv = causal ? i + (Nk - Nq) + 1 : Nk;",
                                           "const int64_t nv = causal ? i + (Nk - Nq) + (i > 0) : Nk;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")).read()
    # a slip in code that two row functions share is planted in both
    assert src.count(old) >= 1, f"mutation site for {name!r} not found"
    mut_src = tmp_path / "attn_ref.c"
    mut_src.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / "libmut.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
        except pytest.skip.Exception:
            pass
    assert caught, f"no pin caught mutant {name!r}"
    shutil.rmtree(tmp_path, ignore_errors=True)

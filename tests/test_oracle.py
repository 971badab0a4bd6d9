"""Pins for the FP64 oracle against facts fixed by the mathematics, not by the oracle itself.

The definition being pinned is S = scale*QK^T, P = softmax_row(S), O = PV, plus the
natural log-sum-exp of each score row ("FlashAttention'ı Anlamak Bölüm 1", section 0.2
Notasyon; "Flash Attention на 5090 в CUDA C++", Алгоритм Flash Attention 2). Each test
below is chosen so that a plausible slip in the oracle (a dropped scale, a sign flip in
the exponent, value rows indexed with the key stride, a missing 1/l, a head-stride
error, a wrong logarithm base) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from dense_attention_forward_fwd_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_qkv

SCALE = float(np.float32(1 / math.sqrt(128)))


def bf16(x):
    """Exact BF16 bits of values that are representable (asserts no rounding happened)."""
    x = np.asarray(x, dtype=np.float32)
    b = f32_to_bf16_bits(x)
    assert np.array_equal(bf16_bits_to_f32(b), x), "test value not exactly representable in BF16"
    return b


def widen(b):
    return bf16_bits_to_f32(b).astype(np.float64)


# ---- invariants ---------------------------------------------------------------------------

def pin_probability_rows_sum_to_one(orc):
    q, k, _ = make_qkv(2, 3, 7, 11, d=16, seed=5, qk_mult=2.0)
    p = orc.probs(q, k, 0.37)
    assert p.shape == (2, 3, 7, 11)
    assert np.all(p >= 0)
    assert np.max(np.abs(p.sum(-1) - 1.0)) < 1e-12


def pin_constant_v_returns_that_row(orc):
    q, k, _ = make_qkv(1, 2, 9, 13, d=32, seed=1)
    c = np.array([((i % 7) - 3) * 0.25 for i in range(32)], dtype=np.float32)
    v = np.broadcast_to(bf16(c), (1, 2, 13, 32)).copy()
    o, _ = orc.attention(q, k, v, SCALE)
    assert np.max(np.abs(o - c.astype(np.float64))) < 1e-12


def pin_zero_query_gives_mean_of_v_and_log_nk(orc):
    _, k, v = make_qkv(2, 2, 5, 37, d=128, seed=2)
    q = np.zeros((2, 2, 5, 128), dtype=np.uint16)  # +0.0 in BF16
    o, lse = orc.attention(q, k, v, SCALE)
    mean_v = widen(v).mean(axis=2)  # [B,H,dv]
    assert np.max(np.abs(o - mean_v[:, :, None, :])) < 1e-12
    assert np.max(np.abs(lse - math.log(37))) < 1e-12


def pin_single_key_returns_its_value_and_score(orc):
    q, k, v = make_qkv(1, 3, 4, 1, d=128, seed=3)
    o, lse = orc.attention(q, k, v, SCALE)
    assert np.max(np.abs(o - widen(v)[:, :, 0:1, :])) < 1e-15
    s = SCALE * np.einsum("bhic,bhc->bhi", widen(q), widen(k)[:, :, 0, :])
    assert np.max(np.abs(lse - s)) < 1e-12


def pin_two_keys_logistic_closed_form(orc):
    # softmax over two scores is the logistic function of their difference
    q, k, v = make_qkv(1, 1, 6, 2, d=8, seed=4, qk_mult=3.0)
    scale = 0.5
    o, lse = orc.attention(q, k, v, scale)
    qw, kw, vw = widen(q)[0, 0], widen(k)[0, 0], widen(v)[0, 0]
    for i in range(6):
        s0 = scale * float(qw[i] @ kw[0])
        s1 = scale * float(qw[i] @ kw[1])
        t = s1 - s0
        sig = 1.0 / (1.0 + math.exp(-t)) if t >= 0 else math.exp(t) / (1.0 + math.exp(t))
        want_o = vw[0] + sig * (vw[1] - vw[0])
        want_lse = max(s0, s1) + math.log1p(math.exp(-abs(t)))
        assert np.max(np.abs(o[0, 0, i] - want_o)) < 1e-12
        assert abs(lse[0, 0, i] - want_lse) < 1e-12


def pin_key_permutation_invariance(orc):
    q, k, v = make_qkv(1, 2, 8, 50, d=64, seed=6)
    perm = np.random.Generator(np.random.PCG64(9)).permutation(50)
    o1, l1 = orc.attention(q, k, v, SCALE)
    o2, l2 = orc.attention(q, k[:, :, perm], v[:, :, perm], SCALE)
    assert np.max(np.abs(o1 - o2)) < 1e-13
    assert np.max(np.abs(l1 - l2)) < 1e-13


def pin_linear_in_v(orc):
    q, k, _ = make_qkv(1, 1, 5, 20, d=16, seed=7)
    g = np.random.Generator(np.random.PCG64(10))
    v1 = g.integers(-8, 9, size=(1, 1, 20, 16)).astype(np.float32)
    v2 = g.integers(-8, 9, size=(1, 1, 20, 16)).astype(np.float32)
    o1, _ = orc.attention(q, k, bf16(v1), SCALE)
    o2, _ = orc.attention(q, k, bf16(v2), SCALE)
    o3, _ = orc.attention(q, k, bf16(2 * v1 + v2), SCALE)
    assert np.max(np.abs(o3 - (2 * o1 + o2))) < 1e-12


def pin_common_key_shift_moves_only_lse(orc):
    # K_j -> K_j + u adds scale*q.u to every score of a row: P unchanged, LSE shifted
    g = np.random.Generator(np.random.PCG64(11))
    kq = g.integers(-8, 9, size=(1, 1, 30, 8)).astype(np.float32) * 0.25
    u = g.integers(-8, 9, size=(8,)).astype(np.float32) * 0.25
    qf = g.integers(-4, 5, size=(1, 1, 6, 8)).astype(np.float32) * 0.5
    _, _, v = make_qkv(1, 1, 6, 30, d=8, seed=12)
    o1, l1 = orc.attention(bf16(qf), bf16(kq), v, 0.3)
    o2, l2 = orc.attention(bf16(qf), bf16(kq + u), v, 0.3)
    shift = 0.3 * (qf[0, 0].astype(np.float64) @ u.astype(np.float64))
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs((l2 - l1)[0, 0] - shift)) < 1e-12


def pin_heads_and_batches_are_independent(orc):
    q, k, v = make_qkv(2, 3, 9, 17, d=32, seed=13)
    o, lse = orc.attention(q, k, v, SCALE)
    for b in range(2):
        for h in range(3):
            oo, ll = orc.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], SCALE)
            assert np.array_equal(oo[0, 0], o[b, h])
            assert np.array_equal(ll[0, 0], lse[b, h])


def pin_scale_zero_is_uniform_and_sign_of_scale_matches_negated_keys(orc):
    q, k, v = make_qkv(1, 2, 4, 19, d=16, seed=14)
    o, lse = orc.attention(q, k, v, 0.0)
    assert np.max(np.abs(o - widen(v).mean(axis=2)[:, :, None, :])) < 1e-12
    assert np.max(np.abs(lse - math.log(19))) < 1e-12
    kneg = k ^ np.uint16(0x8000)  # flip the BF16 sign bit
    o1, l1 = orc.attention(q, k, v, -0.2)
    o2, l2 = orc.attention(q, kneg, v, 0.2)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13


def pin_huge_scores_do_not_overflow(orc):
    # one key's score is ~1000 above the rest: exp() of raw scores would overflow
    d = 4
    qf = np.array([[[[8.0, 0, 0, 0]]]], dtype=np.float32)
    kf = np.zeros((1, 1, 5, d), dtype=np.float32)
    kf[0, 0, 3, 0] = 128.0
    kf[0, 0, 1, 0] = 1.0
    _, _, v = make_qkv(1, 1, 1, 5, d=d, seed=15)
    o, lse = orc.attention(bf16(qf), bf16(kf), v, 1.0)
    assert np.all(np.isfinite(o)) and np.isfinite(lse).all()
    assert np.max(np.abs(o[0, 0, 0] - widen(v)[0, 0, 3])) < 1e-300 + 1e-15
    assert abs(lse[0, 0, 0] - 1024.0) < 1e-12


def pin_row_subset_matches_full_rows(orc):
    q, k, v = make_qkv(2, 2, 33, 40, d=128, seed=16)
    o, lse = orc.attention(q, k, v, SCALE)
    rows = np.array([0, 5, 32, 33, 70, 131], dtype=np.int64)
    os_, ls = orc.attention_rows(q, k, v, SCALE, rows)
    assert np.array_equal(os_, o.reshape(-1, 128)[rows])
    assert np.array_equal(ls, lse.reshape(-1)[rows])


def pin_value_head_dim_may_differ(orc):
    q, k, v = make_qkv(1, 2, 3, 6, d=4, seed=17, dv=3)
    o, _ = orc.attention(q, k, v, 0.7)
    assert o.shape == (1, 2, 3, 3)
    p = orc.probs(q, k, 0.7)
    assert np.max(np.abs(o - np.einsum("bhij,bhjc->bhic", p, widen(v)))) < 1e-12


def test_rejects_bad_sizes():
    orc = oracle.default()
    q, k, v = make_qkv(1, 1, 2, 2, d=4, seed=0)
    with pytest.raises(ValueError):
        orc.attention_rows(q, k, v, 1.0, np.array([4], dtype=np.int64))
    with pytest.raises(TypeError):
        orc.attention(q.astype(np.float32), k, v, 1.0)


# ---- brute force in arbitrary precision -----------------------------------------------------

def _mp_attention(qw, kw, vw, scale):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    Nq, Nk, dv = qw.shape[0], kw.shape[0], vw.shape[1]
    o = np.zeros((Nq, dv))
    lse = np.zeros(Nq)
    for i in range(Nq):
        e = [mp.exp(mp.mpf(scale) * mp.fsum(mp.mpf(float(a)) * mp.mpf(float(b)) for a, b in zip(qw[i], kw[j])))
             for j in range(Nk)]  # no max subtraction: exact arithmetic needs none
        den = mp.fsum(e)
        for c in range(dv):
            o[i, c] = float(mp.fsum(e[j] * mp.mpf(float(vw[j, c])) for j in range(Nk)) / den)
        lse[i] = float(mp.log(den))
    return o, lse


BRUTE_CASES = [(1, 1, 1, 1.0, 1.0), (2, 3, 4, 1.0, 0.5), (3, 5, 4, 3.0, SCALE), (5, 2, 128, 1.0, SCALE),
               (2, 5, 128, 3.0, SCALE), (3, 4, 6, 1.0, 0.8, 5),
               (3, 4, 256, 1.0, 1 / 16, 192)]   # a head dim past 128 (and a different value dim)


def pin_matches_high_precision_brute_force(orc, cases=BRUTE_CASES):
    for case in cases:
        Nq, Nk, d, mult, scale = case[:5]
        dv = case[5] if len(case) > 5 else d
        q, k, v = make_qkv(2, 2, Nq, Nk, d=d, seed=Nq * 100 + Nk, qk_mult=mult, dv=dv)
        o, lse = orc.attention(q, k, v, scale)
        for b in range(2):
            for h in range(2):
                wo, wl = _mp_attention(widen(q)[b, h], widen(k)[b, h], widen(v)[b, h], scale)
                assert np.max(np.abs(o[b, h] - wo)) < 1e-13
                assert np.max(np.abs(lse[b, h] - wl)) < 1e-12 * max(1.0, np.max(np.abs(wl)))


# ---- a library routine as an independent special case ---------------------------------------

def pin_matches_torch_float64_softmax_on_the_256_workload(orc):
    torch = pytest.importorskip("torch")
    q, k, v = make_qkv(1, 1, 256, 256, d=128, seed=0)
    o, lse = orc.attention(q, k, v, SCALE)
    qt, kt, vt = (torch.from_numpy(widen(x)) for x in (q, k, v))
    s = (qt @ kt.transpose(-1, -2)) * SCALE
    ot = torch.softmax(s, dim=-1) @ vt
    lt = torch.logsumexp(s, dim=-1)
    assert np.max(np.abs(o - ot.numpy())) < 1e-12
    assert np.max(np.abs(lse - lt.numpy())) < 1e-12


# ---- causal mask: the definition's optional mask B, aligned to the bottom-right corner --------

def pin_causal_rows_are_plain_attention_over_the_visible_prefix(orc):
    # row i sees keys 0 .. i + Nk - Nq: the plain oracle on that prefix of K and V
    for Nq, Nk, seed in ((5, 9, 30), (7, 7, 31), (1, 4, 32), (6, 11, 33)):
        q, k, v = make_qkv(2, 1, Nq, Nk, d=8, seed=seed)
        o, lse = orc.attention_rows_causal(q, k, v, 0.9)
        o, lse = o.reshape(2, Nq, 8), lse.reshape(2, Nq)
        for b in range(2):
            for i in range(Nq):
                n = i + Nk - Nq + 1
                op, lp = orc.attention_rows(q[b:b + 1, :, i:i + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], 0.9)
                assert np.max(np.abs(o[b, i] - op[0])) < 1e-14
                assert abs(lse[b, i] - lp[0]) < 1e-14


def pin_causal_square_first_row_is_its_own_key(orc):
    # Nq = Nk: row 0 sees key 0 alone, with weight exactly 1: O = V[0], LSE = scale * q0.k0
    q, k, v = make_qkv(1, 2, 6, 6, d=16, seed=34)
    o, lse = orc.attention_rows_causal(q, k, v, 0.5, rows=np.array([0, 6], dtype=np.int64))
    for r, h in ((0, 0), (1, 1)):
        assert np.array_equal(o[r], widen(v)[0, h, 0])
        assert abs(lse[r] - 0.5 * float(np.dot(widen(q)[0, h, 0], widen(k)[0, h, 0]))) < 1e-12


def pin_causal_last_row_sees_every_key(orc):
    q, k, v = make_qkv(1, 1, 4, 10, d=8, seed=35)
    rows = np.array([3], dtype=np.int64)
    oc, lc = orc.attention_rows_causal(q, k, v, 0.8, rows=rows)
    of, lf = orc.attention_rows(q, k, v, 0.8, rows=rows)
    assert np.array_equal(oc, of) and np.array_equal(lc, lf)


def pin_causal_row_ignores_keys_past_its_diagonal(orc):
    # Nq = 5, Nk = 8: row i sees keys 0 .. i + 3, so rewriting keys 5..7 leaves rows 0 and 1
    q, k, v = make_qkv(1, 1, 5, 8, d=8, seed=36)
    o1, l1 = orc.attention_rows_causal(q, k, v, 0.7)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, 5:] = k[0, 0, :3][::-1]
    v2[0, 0, 5:] = v[0, 0, 1:4]
    o2, l2 = orc.attention_rows_causal(q, k2, v2, 0.7)
    assert np.array_equal(o1[:2], o2[:2]) and np.array_equal(l1[:2], l2[:2])
    assert not np.array_equal(o1[4], o2[4])


def test_causal_rejects_more_queries_than_keys():
    q, k, v = make_qkv(1, 1, 5, 4, d=8, seed=37)
    with pytest.raises(ValueError):
        oracle.default().attention_rows_causal(q, k, v, 1.0)


# ---- additive bias: S = scale * Q K^T + B ------------------------------------------------------

NEG_INF_BF16 = np.uint16(0xFF80)


def pin_bias_constant_per_row_moves_only_lse(orc):
    # softmax is unchanged by adding c_i to every score of row i; the log-sum-exp grows by c_i
    q, k, v = make_qkv(2, 2, 6, 6, d=16, seed=40)
    c = np.array([0.5, -3.0, 2.25, 0.0, 7.5, -0.125], dtype=np.float32)
    bias = np.broadcast_to(bf16(c)[None, None, :, None], (1, 1, 6, 6)).copy()
    o0, l0 = orc.attention_rows(q, k, v, 0.6)
    ob, lb = orc.attention_rows_bias(q, k, v, bias, 0.6)
    assert np.max(np.abs(ob - o0)) < 1e-14
    assert np.max(np.abs(lb - (l0 + np.tile(c.astype(np.float64), 4)))) < 1e-13


def pin_bias_single_visible_key_per_row(orc):
    # -inf everywhere but key j(i) = (2i + 1) mod 7: O_i = V_j(i) exactly, LSE_i = scale q_i.k_j(i) + B_i,j(i)
    Nq = Nk = 7
    q, k, v = make_qkv(1, 2, Nq, Nk, d=8, seed=41)
    bias = np.full((1, 2, Nq, Nk), NEG_INF_BF16, dtype=np.uint16)
    keep = [(2 * i + 1) % Nk for i in range(Nq)]
    val = np.float32(0.75)
    for i, j in enumerate(keep):
        bias[0, :, i, j] = bf16([val])[0]
    o, lse = orc.attention_rows_bias(q, k, v, bias, 0.4)
    o, lse = o.reshape(2, Nq, 8), lse.reshape(2, Nq)
    qw, kw, vw = widen(q), widen(k), widen(v)
    for h in range(2):
        for i, j in enumerate(keep):
            assert np.array_equal(o[h, i], vw[0, h, j])
            assert abs(lse[h, i] - (0.4 * float(np.dot(qw[0, h, i], kw[0, h, j])) + 0.75)) < 1e-12


def pin_bias_causal_pattern_equals_the_causal_oracle(orc):
    # 0 on and left of the bottom-right diagonal, -inf right of it: the causal oracle's mask
    for Nq, Nk, seed in ((6, 6, 42), (4, 9, 43)):
        q, k, v = make_qkv(2, 2, Nq, Nk, d=8, seed=seed)
        full = np.zeros((1, 1, Nk, Nk), dtype=np.uint16)   # rows past Nq pad the buffer
        for i in range(Nk):
            full[0, 0, i, i + Nk - Nq + 1:] = NEG_INF_BF16
        oc, lc = orc.attention_rows_causal(q, k, v, 0.9)
        ob, lb = orc.attention_rows_bias(q, k, v, full[:, :, :Nq], 0.9)
        assert np.max(np.abs(ob - oc)) < 1e-14 and np.max(np.abs(lb - lc)) < 1e-13


def pin_bias_matches_high_precision_brute_force(orc):
    # a bias that differs by row, key, head and batch, against exp(s + b) / sum exp(s + b) in 50 digits
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    B, H, N, d = 2, 2, 5, 4
    q, k, v = make_qkv(B, H, N, N, d=d, seed=44)
    rng = np.random.default_rng(45)
    bias = f32_to_bf16_bits(rng.normal(0.0, 2.0, size=(B, H, N, N)).astype(np.float32))
    o, lse = orc.attention_rows_bias(q, k, v, bias, 0.7)
    o, lse = o.reshape(B, H, N, d), lse.reshape(B, H, N)
    qw, kw, vw, bw = widen(q), widen(k), widen(v), widen(bias)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                e = [mp.exp(mp.mpf(0.7) * mp.fsum(mp.mpf(float(x)) * mp.mpf(float(y)) for x, y in zip(qw[b, h, i], kw[b, h, j]))
                            + mp.mpf(float(bw[b, h, i, j]))) for j in range(N)]
                den = mp.fsum(e)
                for c in range(d):
                    assert abs(o[b, h, i, c] - float(mp.fsum(e[j] * mp.mpf(float(vw[b, h, j, c])) for j in range(N)) / den)) < 1e-13
                assert abs(lse[b, h, i] - float(mp.log(den))) < 1e-12


def pin_bias_broadcast_strides_equal_materialised_bias(orc):
    # one [Nq, Nk] bias shared by every head and batch, and one bias per key, against the same
    # values written out in full
    q, k, v = make_qkv(2, 3, 5, 5, d=8, seed=46)
    rng = np.random.default_rng(47)
    shared = f32_to_bf16_bits(rng.normal(size=(1, 1, 5, 5)).astype(np.float32))
    per_key = f32_to_bf16_bits(rng.normal(size=(1, 1, 1, 5)).astype(np.float32))
    for small in (shared, per_key):
        o1, l1 = orc.attention_rows_bias(q, k, v, small, 0.5)
        # the full copy sits at the start of a buffer three times its size, so that an oracle
        # with mixed-up strides reads spare memory rather than past the end
        full = np.zeros((6, 3, 5, 5), dtype=np.uint16)
        full[:2] = np.broadcast_to(small, (2, 3, 5, 5))
        o2, l2 = orc.attention_rows_bias(q, k, v, full[:2], 0.5)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and a per-head bias really is per head: head 1 with head 0's bias differs
    per_head = f32_to_bf16_bits(rng.normal(size=(1, 3, 5, 5)).astype(np.float32))
    o3, _ = orc.attention_rows_bias(q, k, v, per_head, 0.5)
    o4, _ = orc.attention_rows_bias(q, k, v, per_head[:, [0, 0, 0]].copy(), 0.5)
    assert np.array_equal(o3.reshape(2, 3, 5, 8)[:, 0], o4.reshape(2, 3, 5, 8)[:, 0])
    assert not np.array_equal(o3.reshape(2, 3, 5, 8)[:, 1], o4.reshape(2, 3, 5, 8)[:, 1])


def test_bias_rejects_a_shape_that_does_not_broadcast():
    q, k, v = make_qkv(1, 2, 4, 4, d=8, seed=48)
    with pytest.raises(ValueError):
        oracle.default().attention_rows_bias(q, k, v, np.zeros((1, 1, 4, 3), np.uint16), 1.0)
    with pytest.raises(ValueError):
        oracle.default().attention_rows_bias(q, k, v, np.zeros((1, 2, 2, 4), np.uint16), 1.0)


# ---- backward: the gradient of the forward for an upstream gradient dO ------------------------

def pin_dense_forward_equals_the_bf16_oracle_on_bf16_inputs(orc):
    # the double-input forward (used for finite differences) is the pinned forward on the BF16 lattice
    q, k, v = make_qkv(2, 2, 5, 7, d=8, seed=50)
    o1, l1 = orc.attention(q, k, v, 0.6)
    o2, l2 = orc.attention_dense(q, k, v, 0.6)
    assert np.max(np.abs(o1 - o2)) < 1e-15 and np.max(np.abs(l1 - l2)) < 1e-14


def pin_bwd_matches_central_differences(orc):
    # L = sum(dO * O): dL/dx by central differences of the forward for every element of q, k, v
    rng = np.random.default_rng(51)
    # dv > d: a mutant oracle that indexes value rows with the key stride stays inside v
    B, H, Nq, Nk, d, dv = 1, 2, 3, 4, 3, 5
    q, k = rng.normal(size=(B, H, Nq, d)), rng.normal(size=(B, H, Nk, d))
    v, dout = rng.normal(size=(B, H, Nk, dv)), rng.normal(size=(B, H, Nq, dv))
    scale = 0.8
    grads = dict(zip("qkv", orc.attention_bwd(q, k, v, dout, scale)))
    h = 1e-6
    for name in "qkv":
        base = {"q": q, "k": k, "v": v}
        x, g = base[name], grads[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            lo, hi = dict(base), dict(base)
            hi[name] = x.copy()
            hi[name][idx] += h
            lo[name] = x.copy()
            lo[name][idx] -= h
            l_hi = np.sum(orc.attention_dense(hi["q"], hi["k"], hi["v"], scale)[0] * dout)
            l_lo = np.sum(orc.attention_dense(lo["q"], lo["k"], lo["v"], scale)[0] * dout)
            fd[idx] = (l_hi - l_lo) / (2 * h)
        assert np.max(np.abs(fd - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), name


def pin_bwd_key_gradients_sum_to_zero(orc):
    # a common shift of every key changes no probability, so sum_j dK_j = 0 in every head
    q, k, v = make_qkv(2, 3, 9, 11, d=8, seed=52, qk_mult=2.0)
    dout = np.random.default_rng(53).normal(size=(2, 3, 9, 8))
    _, dk, _ = orc.attention_bwd(q, k, v, dout, 0.5)
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-12 * max(1.0, np.max(np.abs(dk)))
    assert np.max(np.abs(dk)) > 1e-3


def pin_bwd_dv_is_probabilities_transposed_times_dout(orc):
    q, k, v = make_qkv(1, 2, 6, 5, d=8, seed=54)
    dout = np.random.default_rng(55).normal(size=(1, 2, 6, 8))
    _, _, dv = orc.attention_bwd(q, k, v, dout, 0.9)
    p = orc.probs(q, k, 0.9)
    assert np.max(np.abs(dv - np.einsum("bhij,bhic->bhjc", p, dout))) < 1e-13


def pin_bwd_zero_upstream_gradient_gives_zero(orc):
    q, k, v = make_qkv(1, 1, 4, 6, d=8, seed=56)
    for g in orc.attention_bwd(q, k, v, np.zeros((1, 1, 4, 8)), 0.7):
        assert np.all(g == 0.0)


def pin_bwd_equal_value_rows_give_no_query_or_key_gradient(orc):
    # every value row equal: O is that row whatever the probabilities, so dQ = dK = 0
    q, k, _ = make_qkv(1, 2, 5, 7, d=8, seed=57)
    v = np.broadcast_to(np.random.default_rng(58).normal(size=(1, 2, 1, 8)), (1, 2, 7, 8)).copy()
    dout = np.random.default_rng(59).normal(size=(1, 2, 5, 8))
    dq, dk, dv = orc.attention_bwd(q, k, v, dout, 0.6)
    assert np.max(np.abs(dq)) < 1e-13 and np.max(np.abs(dk)) < 1e-13
    assert np.max(np.abs(dv)) > 1e-2


def pin_causal_dense_forward_equals_the_bf16_causal_oracle(orc):
    q, k, v = make_qkv(2, 2, 5, 8, d=8, seed=60)
    o1, l1 = orc.attention_rows_causal(q, k, v, 0.6)
    o2, l2 = orc.attention_dense(q, k, v, 0.6, causal=True)
    assert np.max(np.abs(o1 - o2.reshape(-1, 8))) < 1e-15 and np.max(np.abs(l1 - l2.reshape(-1))) < 1e-14


def pin_causal_bwd_matches_central_differences(orc):
    # the gradient of the causal forward, Nq < Nk (bottom-right alignment matters), dv > d
    rng = np.random.default_rng(61)
    B, H, Nq, Nk, d, dv = 1, 2, 3, 5, 3, 4
    q, k = rng.normal(size=(B, H, Nq, d)), rng.normal(size=(B, H, Nk, d))
    v, dout = rng.normal(size=(B, H, Nk, dv)), rng.normal(size=(B, H, Nq, dv))
    scale = 0.9
    grads = dict(zip("qkv", orc.attention_bwd(q, k, v, dout, scale, causal=True)))
    h = 1e-6
    for name in "qkv":
        base = {"q": q, "k": k, "v": v}
        x, g = base[name], grads[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            hi, lo = dict(base), dict(base)
            hi[name] = x.copy()
            hi[name][idx] += h
            lo[name] = x.copy()
            lo[name][idx] -= h
            l_hi = np.sum(orc.attention_dense(hi["q"], hi["k"], hi["v"], scale, causal=True)[0] * dout)
            l_lo = np.sum(orc.attention_dense(lo["q"], lo["k"], lo["v"], scale, causal=True)[0] * dout)
            fd[idx] = (l_hi - l_lo) / (2 * h)
        assert np.max(np.abs(fd - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), name


def pin_causal_bwd_single_query_equals_the_full_gradient(orc):
    # one query row at the end of the sequence sees every key
    q, k, v = make_qkv(1, 2, 1, 6, d=8, seed=62)
    dout = np.random.default_rng(63).normal(size=(1, 2, 1, 8))
    for gc, gf in zip(orc.attention_bwd(q, k, v, dout, 0.7, causal=True), orc.attention_bwd(q, k, v, dout, 0.7)):
        assert np.array_equal(gc, gf)


def pin_causal_bwd_keys_see_only_later_rows(orc):
    # Nq = Nk = 6 with dO zero on rows 3..5: keys 3..5 are seen only by those rows, so their
    # dK and dV are exactly zero, while keys 0..2 have gradients
    q, k, v = make_qkv(1, 1, 6, 6, d=8, seed=64)
    dout = np.random.default_rng(65).normal(size=(1, 1, 6, 8))
    dout[:, :, 3:] = 0.0
    _, dk, dv = orc.attention_bwd(q, k, v, dout, 0.8, causal=True)
    assert np.all(dk[0, 0, 3:] == 0.0) and np.all(dv[0, 0, 3:] == 0.0)
    assert np.min(np.abs(dv[0, 0, :3]).max(axis=-1)) > 1e-3


# ---- the backward of the biased forward (the bias held fixed) -------------------------------

def pin_bias_dense_forward_equals_the_bf16_bias_oracle(orc):
    # the double-input forward with a bias is the pinned BF16 bias oracle on the BF16 lattice,
    # for a bias per (batch, head, row, key) and one shared by every head and batch
    q, k, v = make_qkv(2, 3, 5, 7, d=8, seed=90)
    rng = np.random.default_rng(91)
    for shape in ((2, 3, 5, 7), (1, 1, 5, 7), (1, 3, 1, 7)):
        bias = f32_to_bf16_bits(rng.normal(0.0, 2.0, size=shape).astype(np.float32))
        o1, l1 = orc.attention_rows_bias(q, k, v, bias, 0.6)
        o2, l2 = orc.attention_dense(q, k, v, 0.6, bias=bias)
        assert np.max(np.abs(o1 - o2.reshape(-1, 8))) < 1e-15 and np.max(np.abs(l1 - l2.reshape(-1))) < 1e-13


def pin_bias_bwd_matches_central_differences(orc):
    # L = sum(dO * O) of the biased forward: dL/dx by central differences for every element of
    # q, k, v, with a bias that differs by head, row and key; dv > d
    rng = np.random.default_rng(92)
    B, H, Nq, Nk, d, dv = 1, 2, 3, 4, 3, 5
    q, k = rng.normal(size=(B, H, Nq, d)), rng.normal(size=(B, H, Nk, d))
    v, dout = rng.normal(size=(B, H, Nk, dv)), rng.normal(size=(B, H, Nq, dv))
    bias = rng.normal(0.0, 1.5, size=(B, H, Nq, Nk))
    scale = 0.8
    grads = dict(zip("qkv", orc.attention_bwd(q, k, v, dout, scale, bias=bias)))
    h = 1e-6
    for name in "qkv":
        base = {"q": q, "k": k, "v": v}
        x, g = base[name], grads[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            lo, hi = dict(base), dict(base)
            hi[name] = x.copy()
            hi[name][idx] += h
            lo[name] = x.copy()
            lo[name][idx] -= h
            l_hi = np.sum(orc.attention_dense(hi["q"], hi["k"], hi["v"], scale, bias=bias)[0] * dout)
            l_lo = np.sum(orc.attention_dense(lo["q"], lo["k"], lo["v"], scale, bias=bias)[0] * dout)
            fd[idx] = (l_hi - l_lo) / (2 * h)
        assert np.max(np.abs(fd - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), name


def pin_bias_bwd_causal_pattern_equals_the_causal_gradient(orc):
    # 0 on and left of the bottom-right diagonal, -inf right of it: the (pinned) causal gradient
    for Nq, Nk, seed in ((6, 6, 93), (4, 9, 94)):
        q, k, v = make_qkv(2, 2, Nq, Nk, d=8, seed=seed)
        dout = np.random.default_rng(seed + 100).normal(size=(2, 2, Nq, 8))
        mask = np.zeros((1, 1, Nq, Nk))
        for i in range(Nq):
            mask[0, 0, i, i + Nk - Nq + 1:] = -np.inf
        for gb, gc in zip(orc.attention_bwd(q, k, v, dout, 0.9, bias=mask),
                          orc.attention_bwd(q, k, v, dout, 0.9, causal=True)):
            assert np.max(np.abs(gb - gc)) < 1e-13


def pin_bias_bwd_constant_per_row_changes_no_gradient(orc):
    # adding c_i to every score of row i leaves every probability, hence every gradient, alone;
    # and the key gradients of each head still sum to zero under a general bias
    q, k, v = make_qkv(2, 2, 6, 9, d=8, seed=95, qk_mult=2.0)
    dout = np.random.default_rng(96).normal(size=(2, 2, 6, 8))
    c = np.broadcast_to(np.random.default_rng(97).normal(0.0, 3.0, size=(1, 1, 6, 1)), (1, 1, 6, 9)).copy()
    for gb, g0 in zip(orc.attention_bwd(q, k, v, dout, 0.5, bias=c), orc.attention_bwd(q, k, v, dout, 0.5)):
        assert np.max(np.abs(gb - g0)) < 1e-12 * max(1.0, np.max(np.abs(g0)))
    b = np.random.default_rng(98).normal(0.0, 2.0, size=(2, 2, 6, 9))
    _, dk, _ = orc.attention_bwd(q, k, v, dout, 0.5, bias=b)
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-12 * max(1.0, np.max(np.abs(dk))) and np.max(np.abs(dk)) > 1e-3


# ---- FP8 E4M3 scores ------------------------------------------------------------------------
# Q and K as E4M3 codes (the OCP 8-bit floating point format) with per-tensor descale factors.

def pin_e4m3_decoder_closed_forms_and_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_f64(codes)
    # values fixed by the format: bias 7, three mantissa bits, subnormals below 2^-6
    fixed = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0x3C: 1.5, 0x7E: 448.0, 0x77: 240.0, 0x08: 2.0 ** -6,
             0x0F: 1.875 * 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x04: 2.0 ** -7, 0xB8: -1.0,
             0xFE: -448.0, 0x00: 0.0}
    for c, val in fixed.items():
        assert got[c] == val, f"code {c:#04x}: {got[c]} != {val}"
    assert math.copysign(1.0, got[0x80]) == -1.0 and got[0x80] == 0.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and np.count_nonzero(np.isnan(got)) == 2
    assert np.all(np.diff(got[:127]) > 0), "positive codes must increase with their value"
    assert np.array_equal(got[128:255], -got[:127])
    torch = pytest.importorskip("torch")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~fin) and np.array_equal(got[fin], ref[fin])


def pin_e4m3_scores_equal_the_bf16_oracle_on_the_same_values(orc):
    # every E4M3 value is a BF16 value, so codes widened to BF16 bits give the pinned BF16
    # oracle the same real inputs once the descale factors move into its scale
    from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3
    q8, k8, v, dq, dk = make_qk_e4m3(1, 2, 9, 37, d=16, seed=70, qk_mult=2.0)
    qb, kb = bf16(orc.e4m3_to_f64(q8)), bf16(orc.e4m3_to_f64(k8))
    o8, l8 = orc.attention_rows_e4m3qk(q8, k8, v, 0.3, dq, dk)
    ob, lb = orc.attention_rows(qb, kb, v, 0.3 * dq * dk)
    assert np.max(np.abs(o8 - ob)) < 1e-12 and np.max(np.abs(l8 - lb)) < 1e-12 * np.max(np.abs(lb))
    # the descale factors act only through their product
    o2, l2 = orc.attention_rows_e4m3qk(q8, k8, v, 0.3, dq * 4.0, dk / 4.0)
    assert np.max(np.abs(o2 - o8)) < 1e-12 and np.max(np.abs(l2 - l8)) < 1e-12 * np.max(np.abs(l8))


def pin_e4m3_two_keys_logistic_closed_form(orc):
    # one query row over two keys: P_0 = 1 / (1 + exp(s_1 - s_0)), with s_j written out by hand
    q8 = np.zeros((1, 1, 1, 4), np.uint8)
    k8 = np.zeros((1, 1, 2, 4), np.uint8)
    q8[..., 0], q8[..., 1] = 0x38, 0x40                 # q = (1, 2, 0, 0)
    k8[0, 0, 0, 0], k8[0, 0, 1, 1] = 0x3C, 0xB0          # k_0 = (1.5, 0, ..), k_1 = (0, -0.5, ..)
    v = bf16(np.array([[[[1.0, 0.0], [0.0, 1.0]]]]))
    scale, dq, dk = 0.75, 0.5, 3.0
    s0, s1 = scale * dq * dk * 1.5, scale * dq * dk * (2 * -0.5)
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    o, lse = orc.attention_rows_e4m3qk(q8, k8, v, scale, dq, dk)
    assert abs(o[0, 0] - p0) < 1e-15 and abs(o[0, 1] - (1 - p0)) < 1e-15
    assert abs(lse[0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14


def pin_e4m3_values_equal_the_scores_only_oracle_times_the_value_descale(orc):
    # O is linear in V: with V as codes, O = v_descale * (the E4M3-score oracle on the codes'
    # values, which are BF16 values); the LSE does not involve V. dv != d catches a value
    # row read with the key stride.
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 2, 7, 29, d=16, seed=71, qk_mult=2.0)
    v8 = np.ascontiguousarray(v8[..., :8])
    o8, l8 = orc.attention_rows_e4m3(q8, k8, v8, 0.4, dq, dk, dv)
    ob, lb = orc.attention_rows_e4m3qk(q8, k8, bf16(orc.e4m3_to_f64(v8)), 0.4, dq, dk)
    assert np.max(np.abs(o8 - dv * ob)) < 1e-12 * max(1.0, np.max(np.abs(o8))) and np.array_equal(l8, lb)


def pin_e4m3_constant_values_are_returned(orc):
    # every value row equal to one code: O = v_descale * its value in every row and column
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, _ = make_qkv_e4m3(1, 1, 5, 40, d=16, seed=72)
    v8[:] = 0xC5   # -(1 + 5/8) * 2^(8 - 7) = -3.25
    o8, _ = orc.attention_rows_e4m3(q8, k8, v8, 0.25, dq, dk, 0.5)
    assert np.max(np.abs(o8 + 1.625)) < 1e-13


def pin_e4m3_causal_scores_equal_the_bf16_causal_oracle(orc):
    # under the causal mask too the E4M3-score oracle is the (pinned) BF16 causal oracle on
    # the codes' values, the descale factors moved into the scale; Nq < Nk puts the mask's
    # corner at key Nk - Nq
    from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3
    q8, k8, v, dq, dk = make_qk_e4m3(2, 1, 9, 23, d=16, seed=76, qk_mult=2.0)
    qb, kb = bf16(orc.e4m3_to_f64(q8)), bf16(orc.e4m3_to_f64(k8))
    o8, l8 = orc.attention_rows_e4m3qk(q8, k8, v, 0.3, dq, dk, causal=True)
    ob, lb = orc.attention_rows_causal(qb, kb, v, 0.3 * dq * dk)
    assert np.max(np.abs(o8 - ob)) < 1e-12 and np.max(np.abs(l8 - lb)) < 1e-12 * np.max(np.abs(lb))


def pin_e4m3_causal_rows_are_the_unmasked_rows_over_the_visible_prefix(orc):
    # row i of either FP8 oracle under the mask is its unmasked row over keys 0 .. i + Nk - Nq
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 2, 6, 13, d=16, seed=77, qk_mult=2.0)
    vb = bf16(orc.e4m3_to_f64(v8))
    oq, lq = orc.attention_rows_e4m3qk(q8, k8, vb, 0.4, dq, dk, causal=True)
    oa, la = orc.attention_rows_e4m3(q8, k8, v8, 0.4, dq, dk, dv, causal=True)
    oq, lq, oa, la = oq.reshape(2, 6, 16), lq.reshape(2, 6), oa.reshape(2, 6, 16), la.reshape(2, 6)
    for h in range(2):
        for i in range(6):
            n = i + 13 - 6 + 1
            sl = (slice(None), slice(h, h + 1))
            op, lp = orc.attention_rows_e4m3qk(q8[sl][:, :, i:i + 1], k8[sl][:, :, :n], vb[sl][:, :, :n], 0.4, dq, dk)
            assert np.array_equal(oq[h, i], op[0]) and lq[h, i] == lp[0]
            op, lp = orc.attention_rows_e4m3(q8[sl][:, :, i:i + 1], k8[sl][:, :, :n], v8[sl][:, :, :n], 0.4, dq, dk, dv)
            assert np.array_equal(oa[h, i], op[0]) and la[h, i] == lp[0]


def pin_e4m3_bias_equals_the_bf16_bias_oracle_on_the_same_values(orc):
    # with the optional B of the definition ("FlashAttention'ı Anlamak Bölüm 1", 0.2) the
    # E4M3-score oracle is still the (pinned) BF16 bias oracle on the codes' values: a bias
    # that differs by batch, head, row and key, and one shared by every head and batch
    from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3
    q8, k8, v, dq, dk = make_qk_e4m3(2, 3, 7, 19, d=16, seed=78, qk_mult=2.0)
    qb, kb = bf16(orc.e4m3_to_f64(q8)), bf16(orc.e4m3_to_f64(k8))
    rng = np.random.default_rng(79)
    for shape in ((2, 3, 7, 19), (1, 1, 7, 19), (2, 1, 1, 19)):
        bias = f32_to_bf16_bits(rng.normal(0.0, 2.0, size=shape).astype(np.float32))
        o8, l8 = orc.attention_rows_e4m3qk(q8, k8, v, 0.3, dq, dk, bias=bias)
        ob, lb = orc.attention_rows_bias(qb, kb, v, bias, 0.3 * dq * dk)
        assert np.max(np.abs(o8 - ob)) < 1e-12 and np.max(np.abs(l8 - lb)) < 1e-12 * np.max(np.abs(lb))


def pin_e4m3_bias_constant_per_row_moves_only_lse(orc):
    # adding c_i to every score of row i leaves the softmax alone and adds c_i to the LSE, for
    # both FP8 oracles (a bias row read from the wrong query fails the LSE)
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 2, 6, 11, d=16, seed=80)
    vb = bf16(orc.e4m3_to_f64(v8))
    c = np.array([0.5, -3.0, 2.25, 0.0, 7.5, -0.125], dtype=np.float32)
    bias = np.ascontiguousarray(np.broadcast_to(bf16(c)[None, None, :, None], (1, 1, 6, 11)))
    shift = np.tile(c.astype(np.float64), 2)
    o0, l0 = orc.attention_rows_e4m3qk(q8, k8, vb, 0.4, dq, dk)
    o1, l1 = orc.attention_rows_e4m3qk(q8, k8, vb, 0.4, dq, dk, bias=bias)
    assert np.max(np.abs(o1 - o0)) < 1e-13 and np.max(np.abs(l1 - (l0 + shift))) < 1e-12
    o0, l0 = orc.attention_rows_e4m3(q8, k8, v8, 0.4, dq, dk, dv)
    o1, l1 = orc.attention_rows_e4m3(q8, k8, v8, 0.4, dq, dk, dv, bias=bias)
    assert np.max(np.abs(o1 - o0)) < 1e-13 and np.max(np.abs(l1 - (l0 + shift))) < 1e-12


def pin_e4m3_values_with_bias_equal_the_scores_only_oracle_times_the_value_descale(orc):
    # as without a bias: with V as codes, O = v_descale * (the E4M3-score oracle on the codes'
    # values) under the same per-head bias, and the LSE does not involve V
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(2, 2, 5, 23, d=16, seed=81, qk_mult=2.0)
    v8 = np.ascontiguousarray(v8[..., :8])
    bias = f32_to_bf16_bits(np.random.default_rng(82).normal(size=(2, 2, 5, 23)).astype(np.float32))
    o8, l8 = orc.attention_rows_e4m3(q8, k8, v8, 0.4, dq, dk, dv, bias=bias)
    ob, lb = orc.attention_rows_e4m3qk(q8, k8, bf16(orc.e4m3_to_f64(v8)), 0.4, dq, dk, bias=bias)
    assert np.max(np.abs(o8 - dv * ob)) < 1e-12 * max(1.0, np.max(np.abs(o8))) and np.array_equal(l8, lb)


# ---- MXFP8: E4M3 elements with E8M0 scales per 32 elements along each contraction ----------

def pin_e8m0_decoder_closed_forms(orc):
    got = orc.e8m0_to_f64(np.array([127, 128, 126, 0, 254, 255, 137], dtype=np.uint8))
    assert list(got[:5]) == [1.0, 2.0, 0.5, 2.0 ** -127, 2.0 ** 127] and np.isnan(got[5]) and got[6] == 1024.0


def _mx_real(orc, codes, scales, axis):
    """Real values of MX codes, with the scales repeated over their 32-element blocks."""
    rep = np.repeat(orc.e8m0_to_f64(scales), 32, axis=axis)
    idx = [slice(None)] * codes.ndim
    idx[axis] = slice(0, codes.shape[axis])
    return orc.e4m3_to_f64(codes) * rep[tuple(idx)]


def pin_mxfp8_equals_the_bf16_oracle_on_the_scaled_values(orc):
    # E4M3 values times powers of two are BF16 values here, so the block-scaled inputs widen
    # exactly; random block scales, a partial last key block (Nk = 70) and dv != d catch a
    # scale applied to the wrong block, row or axis
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 2, 9, 70, d=64, seed=73, qk_mult=2.0)
    v8, sv = np.ascontiguousarray(v8[..., :8]), np.ascontiguousarray(sv[..., :8])
    rng = np.random.default_rng(74)
    sq, sk, sv = (np.ascontiguousarray(x + rng.integers(-3, 4, size=x.shape)).astype(np.uint8) for x in (sq, sk, sv))
    qb, kb, vb = (bf16(_mx_real(orc, c, sc, ax)) for c, sc, ax in ((q8, sq, 3), (k8, sk, 3), (v8, sv, 2)))
    om, lm = orc.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, 0.3)
    ob, lb = orc.attention_rows(qb, kb, vb, 0.3)
    assert np.max(np.abs(om - ob)) < 1e-12 * max(1.0, np.max(np.abs(ob)))
    assert np.max(np.abs(lm - lb)) < 1e-12 * np.max(np.abs(lb))


def pin_mxfp8_with_uniform_scales_is_per_tensor_fp8(orc):
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 1, 6, 45, d=32, seed=75)
    sq[:], sk[:], sv[:] = 126, 129, 125        # 2^-1, 2^2, 2^-2 everywhere
    om, lm = orc.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, 0.2)
    oe, le = orc.attention_rows_e4m3(q8, k8, v8, 0.2, 0.5, 4.0, 0.25)
    assert np.max(np.abs(om - oe)) < 1e-13 and np.max(np.abs(lm - le)) < 1e-13


def pin_mxfp8_causal_equals_the_bf16_causal_oracle_on_the_scaled_values(orc):
    # the MXFP8 oracle under the mask is the (pinned) BF16 causal oracle on the block-scaled
    # values; Nq < Nk and a partial last key block of V's scales
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 2, 9, 70, d=64, seed=78, qk_mult=2.0)
    rng = np.random.default_rng(79)
    sq, sk, sv = (np.ascontiguousarray(x + rng.integers(-3, 4, size=x.shape)).astype(np.uint8) for x in (sq, sk, sv))
    qb, kb, vb = (bf16(_mx_real(orc, c, sc, ax)) for c, sc, ax in ((q8, sq, 3), (k8, sk, 3), (v8, sv, 2)))
    om, lm = orc.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, 0.3, causal=True)
    ob, lb = orc.attention_rows_causal(qb, kb, vb, 0.3)
    assert np.max(np.abs(om - ob)) < 1e-12 * max(1.0, np.max(np.abs(ob)))
    assert np.max(np.abs(lm - lb)) < 1e-12 * np.max(np.abs(lb))


def pin_mxfp8_causal_rows_are_the_unmasked_rows_over_the_visible_prefix(orc):
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 1, 5, 64, d=32, seed=80)
    om, lm = orc.attention_rows_mxfp8(q8, sq, k8, sk, v8, sv, 0.25, causal=True)
    for i in range(5):
        n = i + 64 - 5 + 1   # a prefix of whole 32-key blocks plus part of the next: V's scales still apply
        op, lp = orc.attention_rows_mxfp8(q8[:, :, i:i + 1], sq[:, :, i:i + 1], k8[:, :, :n], sk[:, :, :n],
                                          v8[:, :, :n], np.ascontiguousarray(sv[:, :, :(n + 31) // 32]), 0.25)
        assert np.array_equal(om[i], op[0]) and lm[i] == lp[0]


PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__[4:])
def test_oracle_pin(pin):
    pin(oracle.default())

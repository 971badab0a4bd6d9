"""The seeded input generators: BF16 rounding, determinism and row sampling."""
import numpy as np
import pytest

from dense_attention_forward_fwd_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_qkv, sample_rows


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    x = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 1 + 2**-8 + 2**-20, 3.0e38], dtype=np.float32)
    got = bf16_bits_to_f32(f32_to_bf16_bits(x))
    want = np.array([1.0, 1.0, 1 + 2 * 2**-7, -1.0, 1 + 2**-7, 3.0e38], dtype=np.float32)
    assert np.allclose(got[:5], want[:5], rtol=0, atol=0)
    assert abs(got[5] - 3.0e38) / 3.0e38 < 2**-8


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.Generator(np.random.PCG64(1)).standard_normal(100000, dtype=np.float32) * 7
    ours = f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_make_qkv_is_deterministic_and_ordered():
    a = make_qkv(1, 2, 3, 5, d=8, seed=3)
    b = make_qkv(1, 2, 3, 5, d=8, seed=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert a[0].shape == (1, 2, 3, 8) and a[1].shape == (1, 2, 5, 8) and a[2].shape == (1, 2, 5, 8)
    c = make_qkv(1, 2, 3, 5, d=8, seed=3, qk_mult=3.0)
    assert np.array_equal(c[2], a[2])  # V is not scaled
    assert not np.array_equal(c[0], a[0])
    # Q drawn first: the Q block equals the first draws of the stream
    g = np.random.Generator(np.random.PCG64(3)).standard_normal((1, 2, 3, 8), dtype=np.float32)
    assert np.array_equal(a[0], f32_to_bf16_bits(g))


def test_sample_rows():
    r = sample_rows(1, 16, 16384, per_head=64)
    assert np.all(np.diff(r) > 0)
    assert {0, 127, 128, 16383}.issubset(set(r.tolist()))
    per_head = np.bincount(r // 16384, minlength=16)
    assert np.all(per_head >= 64)
    assert np.array_equal(r, sample_rows(1, 16, 16384, per_head=64))


def test_mxfp8_inputs_use_each_block_s_range_and_round_closely():
    # per block of 32 along the contraction axis: the shared exponent puts the block's largest
    # magnitude in [256, 512) before saturation to 448, and every element is the E4M3 rounding
    # of its normal clamped to +-448 block units (relative error <= 2^-4, or an absolute 2^-10
    # of the block scale below 2^-6)
    import numpy as np
    import oracle
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8
    q8, sq, k8, sk, v8, sv = make_qkv_mxfp8(1, 2, 40, 70, d=64, seed=9)
    rng = np.random.Generator(np.random.PCG64(9))
    q = rng.standard_normal((1, 2, 40, 64), dtype=np.float32)
    vals = oracle.e4m3_to_f64(q8)
    blocks = np.abs(vals).reshape(1, 2, 40, 2, 32).max(axis=-1)
    assert np.all((blocks >= 256) & (blocks <= 448))
    real = vals * np.repeat(oracle.e8m0_to_f64(sq), 32, axis=3)
    unit = np.repeat(oracle.e8m0_to_f64(sq), 32, axis=3)
    clamped = np.clip(q, -448.0 * unit, 448.0 * unit)
    assert np.all(np.abs(real - clamped) <= np.maximum(np.abs(clamped) * 2.0 ** -4, unit * 2.0 ** -10) * (1 + 1e-6))
    assert np.count_nonzero(clamped != q) < q.size // 50   # saturation is rare
    assert sv.shape == (1, 2, 3, 64) and sk.shape == (1, 2, 70, 2)


def test_e4m3_inputs_are_per_tensor_quantizations_of_the_bf16_draw():
    # descale = amax / 448 (so the largest code is 448), every code the E4M3 rounding of its
    # normal over the descale, and V of make_qkv_e4m3 the same draw as make_qkv's V
    import numpy as np
    import oracle
    from dense_attention_forward_fwd_gb300.inputs import make_qk_e4m3, make_qkv, make_qkv_e4m3
    q8, k8, v8, dq, dk, dv = make_qkv_e4m3(1, 2, 50, 70, d=32, seed=12, qk_mult=3.0)
    q8b, k8b, vb, dqb, dkb = make_qk_e4m3(1, 2, 50, 70, d=32, seed=12, qk_mult=3.0)
    assert np.array_equal(q8, q8b) and np.array_equal(k8, k8b) and (dq, dk) == (dqb, dkb)
    assert np.array_equal(vb, make_qkv(1, 2, 50, 70, d=32, seed=12)[2])
    rng = np.random.Generator(np.random.PCG64(12))
    q = rng.standard_normal((1, 2, 50, 32), dtype=np.float32) * np.float32(3.0)
    k = rng.standard_normal((1, 2, 70, 32), dtype=np.float32) * np.float32(3.0)
    v = rng.standard_normal((1, 2, 70, 32), dtype=np.float32)
    for codes, ds, x in ((q8, dq, q), (k8, dk, k), (v8, dv, v)):
        vals = oracle.e4m3_to_f64(codes)
        assert np.max(np.abs(vals)) == 448.0
        assert ds == float(np.float32(np.abs(x).max() / 448.0))
        t = x.astype(np.float64) / ds
        assert np.all(np.abs(vals - t) <= np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))


def test_mx_value_layout_transposes_and_pads():
    from dense_attention_forward_fwd_gb300.inputs import make_qkv_mxfp8, mx_value_layout
    for Nk in (33, 130, 640):
        _, _, _, _, v8, sv = make_qkv_mxfp8(1, 2, 4, Nk, seed=Nk)
        vt8, svt = mx_value_layout(v8, sv)
        ldv, ldsv = vt8.shape[3], svt.shape[3]
        assert ldv % 16 == 0 and ldv >= Nk
        assert ldsv % 16 == 0 and ldsv >= 4 * ((Nk + 127) // 128) and ldsv >= sv.shape[2]
        assert np.array_equal(vt8[..., :Nk], np.swapaxes(v8, 2, 3))
        assert np.array_equal(svt[..., :sv.shape[2]], np.swapaxes(sv, 2, 3))
        assert np.all(vt8[..., Nk:] == 0x7F) and np.all(svt[..., sv.shape[2]:] == 0xFF)   # NaN padding

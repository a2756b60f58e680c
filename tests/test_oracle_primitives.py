"""Pins for the oracle's primitives: closed forms, invariants, brute force and
textbook library routines (numpy / torch CPU, float64).  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle

FP16, BF16 = 0, 1


# ------------------------------------------------------------ 16-bit formats

def test_fp16_round_matches_numpy():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-5, 1000), rng.normal(0, 3e4, 500),
                         [65504.0, 65519.9, 65520.0, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8, -0.0, 1.0 + 2 ** -11]])
    for x in xs:
        ref = float(np.float16(x))
        got = oracle.act16_round(x, FP16)
        assert got == ref or (math.isinf(got) and math.isinf(ref)), (x, got, ref)
        assert oracle.act16_encode(x, FP16) == int(np.float16(x).view(np.uint16)), x


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-30, 300), rng.normal(0, 1e30, 300)]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16)
    ref_bits = ref.view(torch.int16).numpy().astype(np.uint16)
    ref_vals = ref.to(torch.float64).numpy()
    for x, rb, rv in zip(xs, ref_bits, ref_vals):
        assert oracle.act16_round(float(x), BF16) == rv
        assert oracle.act16_encode(float(x), BF16) == rb


def test_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    f16 = bits.view(np.float16).astype(np.float64)
    bf = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b in range(0, 65536, 7):
        for act, ref in ((FP16, f16[b]), (BF16, bf[b])):
            got = oracle.act16_decode(b, act)
            assert (math.isnan(got) and math.isnan(ref)) or got == ref


def test_sentinel_is_nan_in_both_types():
    assert math.isnan(oracle.act16_decode(oracle.KV_SENTINEL, FP16))
    assert math.isnan(oracle.act16_decode(oracle.KV_SENTINEL, BF16))


# ------------------------------------------------------------ cosine s(l)

def test_cosine_closed_forms():
    rng = np.random.default_rng(2)
    a = rng.normal(size=257)
    b = rng.normal(size=257)
    assert oracle.cosine(a, a) == pytest.approx(1.0, abs=1e-15)
    assert oracle.cosine(a, -a) == pytest.approx(-1.0, abs=1e-15)
    assert oracle.cosine(a, 7.5 * a) == pytest.approx(1.0, abs=1e-15)
    # scale invariance
    assert oracle.cosine(3.0 * a, 0.25 * b) == pytest.approx(oracle.cosine(a, b), abs=1e-14)
    # orthogonal vectors
    e0 = np.zeros(8); e0[0] = 2.0
    e3 = np.zeros(8); e3[3] = -5.0
    assert oracle.cosine(e0, e3) == 0.0
    # the 45-degree case
    assert oracle.cosine([1.0, 0.0], [1.0, 1.0]) == pytest.approx(1 / math.sqrt(2), abs=1e-15)
    # symmetric, bounded
    assert oracle.cosine(a, b) == pytest.approx(oracle.cosine(b, a), abs=1e-15)
    assert -1.0 <= oracle.cosine(a, b) <= 1.0
    # a zero vector gives 0 (floored denominator)
    assert oracle.cosine(np.zeros(4), np.ones(4)) == 0.0


def test_cosine_vs_angle_brute_force():
    # 2-D vectors at known angles: cos of the angle between them
    for th1, th2 in [(0.1, 1.3), (2.0, -1.0), (0.0, math.pi), (1.0, 1.0 + math.pi / 2)]:
        a = [3 * math.cos(th1), 3 * math.sin(th1)]
        b = [0.5 * math.cos(th2), 0.5 * math.sin(th2)]
        assert oracle.cosine(a, b) == pytest.approx(math.cos(th2 - th1), abs=1e-14)


# ------------------------------------------------------------ RMSNorm

def test_rmsnorm_closed_forms():
    one = np.full(64, 0x3C00, dtype=np.uint16)  # fp16 1.0
    # constant vector c: output = c / sqrt(c^2 + eps), rounded
    out = oracle.rmsnorm(np.full(64, 3.0), one, 1e-5, FP16)
    assert np.all(out == float(np.float16(3.0 / math.sqrt(9.0 + 1e-5))))
    # scale invariance (eps negligible)
    rng = np.random.default_rng(3)
    h = rng.normal(size=64) * 100
    assert np.array_equal(oracle.rmsnorm(h, one, 0.0, FP16), oracle.rmsnorm(h * 4.0, one, 0.0, FP16))
    # output has unit RMS before rounding
    o = oracle.rmsnorm(h, one, 0.0, FP16)
    assert math.sqrt(np.mean(o ** 2)) == pytest.approx(1.0, rel=2e-3)


def test_rmsnorm_vs_torch():
    rng = np.random.default_rng(4)
    h = rng.normal(size=256) * 3
    gam = rng.uniform(0.5, 1.5, 256).astype(np.float16)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h)[None], (256,), torch.from_numpy(gam.astype(np.float64)),
                                       eps=1e-5)[0].numpy()
    got = oracle.rmsnorm(h, gam.view(np.uint16), 1e-5, FP16)
    assert np.array_equal(got, ref.astype(np.float16).astype(np.float64)) or np.max(np.abs(got - ref)) < 2e-3


# ------------------------------------------------------------ RoPE

def test_rope_identity_at_zero_and_norm():
    rng = np.random.default_rng(5)
    v = rng.normal(size=64)
    assert np.array_equal(oracle.rope(v, 0, 10000.0), v)
    for p in (1, 17, 1000, 65535):
        r = oracle.rope(v, p, 500000.0)
        assert np.linalg.norm(r) == pytest.approx(np.linalg.norm(v), rel=1e-13)
        # each rotated pair keeps its own norm
        assert np.allclose(np.hypot(r[:32], r[32:]), np.hypot(v[:32], v[32:]), rtol=1e-13)


def test_rope_two_dims_is_rotation_by_position():
    # head_dim 2: one pair, frequency theta^0 = 1, angle = pos
    for p in (1, 2, 7):
        r = oracle.rope([1.0, 0.0], p, 10000.0)
        assert r[0] == pytest.approx(math.cos(p), abs=1e-15)
        assert r[1] == pytest.approx(math.sin(p), abs=1e-15)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(6)
    q = rng.normal(size=128)
    k = rng.normal(size=128)
    base = np.dot(oracle.rope(q, 10, 500000.0), oracle.rope(k, 3, 500000.0))
    for shift in (1, 100, 4000):
        d = np.dot(oracle.rope(q, 10 + shift, 500000.0), oracle.rope(k, 3 + shift, 500000.0))
        assert d == pytest.approx(base, rel=1e-9, abs=1e-9)


def test_rope_pairing_rotate_half():
    # a vector with one nonzero in slot i moves only into slot i + hd/2
    v = np.zeros(8); v[1] = 1.0
    r = oracle.rope(v, 5, 10000.0)
    ang = 5 * 10000.0 ** (-2 * 1 / 8)
    assert r[1] == pytest.approx(math.cos(ang)) and r[5] == pytest.approx(math.sin(ang))
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2


# ------------------------------------------------------------ attention

def _bits(x, act=FP16):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_attention_single_position_returns_value():
    rng = np.random.default_rng(7)
    K = _bits(rng.normal(size=(1, 64)))
    V = _bits(rng.normal(size=(1, 64)))
    out = oracle.attention(rng.normal(size=64), K, V, FP16)
    assert np.array_equal(out, V.view(np.float16).astype(np.float64)[0])


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(8)
    K = np.tile(_bits(rng.normal(size=(1, 32))), (5, 1))
    V = _bits(rng.normal(size=(5, 32)))
    out = oracle.attention(rng.normal(size=32), K, V, FP16)
    assert np.allclose(out, V.view(np.float16).astype(np.float64).mean(0), atol=1e-14)


def test_attention_vs_torch_sdpa():
    rng = np.random.default_rng(9)
    T, hd = 37, 64
    q = rng.normal(size=hd)
    K = _bits(rng.normal(size=(T, hd)))
    V = _bits(rng.normal(size=(T, hd)))
    Kf = torch.from_numpy(K.view(np.float16).astype(np.float64))
    Vf = torch.from_numpy(V.view(np.float16).astype(np.float64))
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[None, None, None], Kf[None, None],
                                                           Vf[None, None])[0, 0, 0].numpy()
    assert np.allclose(oracle.attention(q, K, V, FP16), ref, atol=1e-13, rtol=1e-12)


# ------------------------------------------------------------ argmax, silu

def test_argmax_lowest_index_on_ties():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([5.0, 5.0]) == 0
    rng = np.random.default_rng(10)
    v = rng.integers(0, 5, 1000).astype(np.float64)
    assert oracle.argmax(v) == int(np.argmax(v))  # numpy returns the first maximum


def test_silu_vs_torch():
    for g in (-30.0, -3.0, -0.5, 0.0, 0.7, 4.0, 40.0):
        assert oracle.silu(g) == pytest.approx(torch.nn.functional.silu(torch.tensor(g, dtype=torch.float64)).item(),
                                               rel=1e-15, abs=1e-300)

"""Pins of the oracle's small ops (RMSNorm, RoPE, softmax, SiLU, attention,
argmax) against closed forms, invariants and degenerate cases."""
import math

import numpy as np
import pytest

import oracle


def test_rmsnorm_closed_form_constant_vector():
    for c in (0.5, -3.0, 1e-3):
        out = oracle.rmsnorm(np.full(64, c), eps=1e-5)
        np.testing.assert_allclose(out, c / math.sqrt(c * c + 1e-5), rtol=1e-15)


def test_rmsnorm_output_rms_is_one_when_eps_negligible():
    x = np.random.default_rng(0).standard_normal(4096) * 3
    out = oracle.rmsnorm(x, eps=1e-5)
    ms = np.mean(x * x)
    assert abs(math.sqrt(np.mean(out * out)) - math.sqrt(ms / (ms + 1e-5))) < 1e-12
    assert abs(math.sqrt(np.mean(out * out)) - 1) < 1e-6


def test_rope_identity_at_position_zero():
    v = np.random.default_rng(1).standard_normal(4 * 64)
    np.testing.assert_array_equal(oracle.rope(v, 4, 64, 0), v)


def test_rope_closed_form_angles():
    hd, theta = 128, 500000.0
    v = np.zeros(hd)
    v[0::2] = 1.0                                   # every pair = (1, 0)
    out = oracle.rope(v, 1, hd, 3, theta)
    for i in (0, 1, 32, 63):
        ang = 3 * theta ** (-2 * i / hd)
        assert abs(out[2 * i] - math.cos(ang)) < 1e-15 and abs(out[2 * i + 1] - math.sin(ang)) < 1e-15
    # pair 0 turns by exactly the position (theta^0 = 1): a quarter turn at p = pi/2 is not an
    # integer, so check p = 1 -> (cos 1, sin 1)
    o1 = oracle.rope(v, 1, hd, 1, theta)
    assert abs(o1[0] - math.cos(1.0)) < 1e-15 and abs(o1[1] - math.sin(1.0)) < 1e-15


def test_rope_preserves_pair_norms_and_composes():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(8 * 64)
    a = oracle.rope(v, 8, 64, 37)
    np.testing.assert_allclose(np.hypot(a[0::2], a[1::2]), np.hypot(v[0::2], v[1::2]), rtol=1e-13)
    np.testing.assert_allclose(oracle.rope(oracle.rope(v, 8, 64, 37), 8, 64, 100), oracle.rope(v, 8, 64, 137),
                               atol=1e-12)
    # the rotation acts on adjacent pairs: swapping the halves of a pair and negating is a quarter turn
    w = np.zeros(64); w[10] = 1.0
    r = oracle.rope(w, 1, 64, 5)
    assert r[10] != 1.0 and r[11] != 0.0 and np.count_nonzero(r) == 2


def test_softmax_sums_to_one_shift_invariant_and_closed_form():
    s = np.random.default_rng(3).standard_normal(1000) * 5
    p = oracle.softmax(s)
    assert abs(p.sum() - 1) < 1e-12
    np.testing.assert_allclose(oracle.softmax(s + 123.0), p, rtol=1e-10)
    np.testing.assert_allclose(oracle.softmax(np.array([0.0, math.log(3.0)])), [0.25, 0.75], rtol=1e-15)
    # large scores do not overflow
    assert np.isfinite(oracle.softmax(np.array([1000.0, 999.0]))).all()


def test_silu_identities():
    assert oracle.silu(0.0) == 0.0
    for z in (0.1, 1.0, 2.5, 10.0):
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12


def _f16(a):
    return np.asarray(a, np.float16).view(np.uint16)


def test_attention_single_position_returns_v0():
    rng = np.random.default_rng(4)
    k = _f16(rng.standard_normal((1, 64)))
    v = _f16(rng.standard_normal((1, 64)))
    out = oracle.attend(rng.standard_normal(64), k, v)
    np.testing.assert_array_equal(out, v.view(np.float16).astype(np.float64)[0])


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(5)
    k = _f16(np.tile(rng.standard_normal(64), (7, 1)))
    vf = rng.standard_normal((7, 64))
    v = _f16(vf)
    out = oracle.attend(rng.standard_normal(64), k, v)
    np.testing.assert_allclose(out, v.view(np.float16).astype(np.float64).mean(0), rtol=1e-12, atol=1e-15)


def test_attention_two_positions_closed_form():
    # q.k_0 = 0 and q.k_1 = sqrt(64) ln 3 after scaling by 1/sqrt(64): weights 1/4, 3/4
    hd = 64
    q = np.zeros(hd); q[0] = 1.0
    k = np.zeros((2, hd)); k[1, 0] = 8 * math.log(3.0)
    kh = _f16(k)
    s1 = float(kh.view(np.float16)[1, 0]) / 8.0
    w1 = math.exp(s1) / (1 + math.exp(s1))
    v = np.zeros((2, hd)); v[0, :] = 1.0; v[1, :] = -1.0
    out = oracle.attend(q, kh, _f16(v))
    np.testing.assert_allclose(out, (1 - w1) - w1, rtol=1e-14)


def test_argmax_ties_lowest_index_and_margin():
    i, m = oracle.argmax(np.array([1.0, 3.0, 3.0, 2.0]))
    assert i == 1 and m == 0.0
    i, m = oracle.argmax(np.array([-5.0, -1.0, -2.5]))
    assert i == 1 and m == 1.5

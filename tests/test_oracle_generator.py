"""Pins of the oracle's counter-based generator and binary16 conversion."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GAMMA = 0x9E3779B97F4A7C15


def test_mix64_matches_published_splitmix64_sequence():
    for line in open(os.path.join(GOLDEN, "splitmix64_seed0.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, want = line.split()
        assert oracle.mix64((int(k) * GAMMA) % 2**64) == int(want, 16)


def test_normal_is_a_multiple_of_2_pow_minus16_and_bounded():
    z = oracle.gen_normal(0, 7, 0, 200_000, 1.0).astype(np.float64)
    assert np.all(np.abs(z) <= 6.0)
    assert np.all(z * 65536 == np.round(z * 65536))


def test_normal_moments_irwin_hall_12():
    # sum of 12 U(0,1) minus 6: mean 0, variance 1, kurtosis 3 - 6/(5*12) = 2.9
    z = oracle.gen_normal(0, 3, 0, 1_000_000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.var() - 1.0) < 5e-3
    kurt = np.mean(z**4) / z.var() ** 2
    assert abs(kurt - 2.9) < 0.03


def test_std_scaling_is_one_fp32_multiply():
    z = oracle.gen_normal(5, 11, 100, 4096, 1.0)
    w = oracle.gen_normal(5, 11, 100, 4096, 0.02)
    np.testing.assert_array_equal(w, (z * np.float32(0.02)).astype(np.float32))
    s = w.astype(np.float64)
    assert abs(s.std() / 0.02 - 1) < 0.05


def test_counter_keys_are_independent():
    a = oracle.gen_normal(0, 1, 0, 100_000, 1.0).astype(np.float64)
    b = oracle.gen_normal(0, 2, 0, 100_000, 1.0).astype(np.float64)
    c = oracle.gen_normal(1, 1, 0, 100_000, 1.0).astype(np.float64)
    for u, v in ((a, b), (a, c), (a[:-1], a[1:])):
        assert abs(np.corrcoef(u, v)[0, 1]) < 0.02
    # element i of the stream does not depend on where the draw starts
    np.testing.assert_array_equal(oracle.gen_normal(0, 1, 500, 10, 1.0), a[500:510].astype(np.float32))


def test_tokens_in_range_and_spread():
    t = np.array(oracle.tokens(3, 4000, 128256))
    assert t.min() >= 0 and t.max() < 128256
    assert len(set(t.tolist())) > 3900


def _all_f16_values():
    return np.arange(65536, dtype=np.uint16).view(np.float16)


def test_f16_decode_matches_ieee_binary16_for_every_code():
    vals = _all_f16_values().astype(np.float64)
    for code in range(0, 65536, 7):
        got = oracle.f16_to_double(code)
        want = vals[code]
        if np.isnan(want):
            assert np.isnan(got)
        else:
            assert got == want


def test_f16_encode_round_to_nearest_even_against_numpy():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        rng.standard_normal(5000).astype(np.float32) * np.float32(3e4),
        rng.standard_normal(5000).astype(np.float32) * np.float32(1e-6),
        np.float32([0.0, -0.0, 65504.0, 65519.996, 65520.0, 1e9, 2.0**-24, 2.0**-25, 3 * 2.0**-25,
                    2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11]),
    ])
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_from_double(float(x)) for x in xs], np.uint16)
    np.testing.assert_array_equal(got, want)


def test_f16_encode_hand_cases():
    assert oracle.f16_from_double(1.0) == 0x3C00
    assert oracle.f16_from_double(2.0**-10) == 0x1400
    assert oracle.f16_from_double(2.0**-24) == 0x0001
    assert oracle.f16_from_double(2.0**-25) == 0x0000          # tie -> even (zero)
    assert oracle.f16_from_double(3 * 2.0**-25) == 0x0002      # tie -> even (2 * 2^-24)
    assert oracle.f16_from_double(1.0 + 2.0**-11) == 0x3C00    # tie -> even
    assert oracle.f16_from_double(1.0 + 3 * 2.0**-11) == 0x3C02
    assert oracle.f16_from_double(65520.0) == 0x7C00           # rounds past the largest finite
    assert oracle.f16_from_double(-65504.0) == 0xFBFF

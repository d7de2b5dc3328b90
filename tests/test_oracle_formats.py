"""Pins of the oracle's block formats: hand-worked blocks, round-trip error
bounds, special cases and exact brute-force GEMV on dyadic data."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from blockspec import pack_q4_0, pack_q4_k, pack_q5_k, pack_q6_k, pack_q8_0

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FORMATS = ["q8_0", "q4_0", "q4_k", "q6_k", "q5_k"]


# ---------------------------------------------------------------- dequant --

def test_dequant_q8_0_hand_block():
    q = [k - 16 for k in range(32)]
    w = oracle.dequant_row("q8_0", np.frombuffer(pack_q8_0(0.5, q), np.uint8), 32)
    np.testing.assert_array_equal(w, np.array(q, np.float32) / 2)


def test_dequant_q4_0_hand_block():
    q = [k % 16 for k in range(32)]
    w = oracle.dequant_row("q4_0", np.frombuffer(pack_q4_0(0.25, q), np.uint8), 32)
    np.testing.assert_array_equal(w, (np.array(q, np.float32) - 8) / 4)   # -2 .. 1.75


def test_dequant_q4_k_hand_block():
    # d = 1, dmin = 0.5, sub-block j: sc = j+1, m = 2j  ->  w = (j+1) q - j
    sc = [j + 1 for j in range(8)]
    m = [2 * j for j in range(8)]
    q = [(k * 7) % 16 for k in range(256)]
    w = oracle.dequant_row("q4_k", np.frombuffer(pack_q4_k(1.0, 0.5, sc, m, q), np.uint8), 256)
    want = [(k // 32 + 1) * q[k] - k // 32 for k in range(256)]
    np.testing.assert_array_equal(w, np.array(want, np.float32))


def test_dequant_q4_k_uniform_scale_gives_3q_minus_1():
    q = [k % 16 for k in range(256)]
    w = oracle.dequant_row("q4_k", np.frombuffer(pack_q4_k(1.0, 0.5, [3] * 8, [2] * 8, q), np.uint8), 256)
    np.testing.assert_array_equal(w, 3 * np.array(q, np.float32) - 1)


def test_dequant_q5_k_hand_block():
    # d = 1, dmin = 0.5, sub-block j: sc = j+1, m = 2j  ->  w = (j+1) q - j, q in 0..31
    sc = [j + 1 for j in range(8)]
    m = [2 * j for j in range(8)]
    q = [(k * 7) % 32 for k in range(256)]
    w = oracle.dequant_row("q5_k", np.frombuffer(pack_q5_k(1.0, 0.5, sc, m, q), np.uint8), 256)
    want = [(k // 32 + 1) * q[k] - k // 32 for k in range(256)]
    np.testing.assert_array_equal(w, np.array(want, np.float32))
    # uniform sc = 3, m = 2: 3q - 1 for q = 0..31 (the fifth bit carries 16)
    q2 = [k % 32 for k in range(256)]
    w2 = oracle.dequant_row("q5_k", np.frombuffer(pack_q5_k(1.0, 0.5, [3] * 8, [2] * 8, q2), np.uint8), 256)
    np.testing.assert_array_equal(w2, 3 * np.array(q2, np.float32) - 1)


def test_dequant_q6_k_hand_block():
    # d = 0.125, sub-block j: sc = j - 8 (int8, may be negative) -> w = 0.125 (j-8)(q-32)
    sc = [j - 8 for j in range(16)]
    q = [(k * 5 + 3) % 64 for k in range(256)]
    w = oracle.dequant_row("q6_k", np.frombuffer(pack_q6_k(0.125, sc, q), np.uint8), 256)
    want = [0.125 * (k // 16 - 8) * (q[k] - 32) for k in range(256)]
    np.testing.assert_array_equal(w, np.array(want, np.float32))
    w8 = oracle.dequant_row("q6_k", np.frombuffer(pack_q6_k(0.125, [8] * 16, q), np.uint8), 256)
    np.testing.assert_array_equal(w8, np.array(q, np.float32) - 32)


# --------------------------------------------------------------- quantize --

def _golden_blocks():
    for line in open(os.path.join(GOLDEN, "quant_blocks.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, fmt, spec, hexs = [p.strip() for p in line.split("|")]
        w = np.zeros(oracle.BLOCK_ELEMS[fmt], np.float32)
        for i, item in enumerate(filter(None, spec.split(","))):
            mant, exp = item.split("@")
            w[i] = float(mant) * 2.0 ** int(exp)
        yield name, fmt, w, bytes.fromhex(hexs)


@pytest.mark.parametrize("case", list(_golden_blocks()), ids=lambda c: c[0])
def test_quantize_hand_worked_golden(case):
    _, fmt, w, want = case
    assert oracle.quantize_row(fmt, w).tobytes() == want


def test_quantize_q4_k_exact_grid_roundtrip():
    # Sub-block j holds w = -m_j 2^-9 + q sc_j 2^-8 with q = 0..15 present, so
    # lo = -m_j 2^-9, s_j = sc_j 2^-8, and max s = 63 * 2^-8 -> d = 2^-8,
    # max m* = 63 * 2^-9 -> dmin = 2^-9: every step is exact and the block
    # must come back as exactly these (d, dmin, sc, m, q).
    sc = [63 - 7 * j for j in range(8)]
    m = [9 * j for j in range(8)]
    q = [(k * 11 + j) % 16 for j in range(8) for k in range(32)]
    w = np.array([-m[k // 32] * 2.0**-9 + q[k] * sc[k // 32] * 2.0**-8 for k in range(256)], np.float32)
    got = oracle.quantize_row("q4_k", w).tobytes()
    assert got == pack_q4_k(2.0**-8, 2.0**-9, sc, m, q)
    np.testing.assert_array_equal(oracle.dequant_row("q4_k", np.frombuffer(got, np.uint8), 256), w)


def test_quantize_q5_k_exact_grid_roundtrip():
    # as the Q4_K case with q = 0..31 present in every sub-block: lo = -m_j 2^-9,
    # s_j = 31 sc_j 2^-8 / 31 = sc_j 2^-8, d = 2^-8, dmin = 2^-9
    sc = [63 - 7 * j for j in range(8)]
    m = [9 * j for j in range(8)]
    q = [(k * 13 + j) % 32 for j in range(8) for k in range(32)]
    w = np.array([-m[k // 32] * 2.0**-9 + q[k] * sc[k // 32] * 2.0**-8 for k in range(256)], np.float32)
    got = oracle.quantize_row("q5_k", w).tobytes()
    assert got == pack_q5_k(2.0**-8, 2.0**-9, sc, m, q)
    np.testing.assert_array_equal(oracle.dequant_row("q5_k", np.frombuffer(got, np.uint8), 256), w)


def test_quantize_q6_k_exact_grid_roundtrip():
    # amax_j = 31 sc_j 2^-10 -> s_j = sc_j 2^-10; max sc = 127 -> d = 2^-10.
    sc = [127 - 8 * j for j in range(16)]
    pattern = [1, 63, 32, 33, 31, 17, 47, 2, 62, 40, 24, 5, 59, 10, 54, 36]
    q = [pattern[(k + j) % 16] for j in range(16) for k in range(16)]
    w = np.array([(q[k] - 32) * sc[k // 16] * 2.0**-10 for k in range(256)], np.float32)
    got = oracle.quantize_row("q6_k", w).tobytes()
    assert got == pack_q6_k(2.0**-10, sc, q)
    np.testing.assert_array_equal(oracle.dequant_row("q6_k", np.frombuffer(got, np.uint8), 256), w)


@pytest.mark.parametrize("fmt", FORMATS)
def test_zero_block_dequantizes_to_zero(fmt):
    n = oracle.BLOCK_ELEMS[fmt]
    b = oracle.quantize_row(fmt, np.zeros(n, np.float32))
    np.testing.assert_array_equal(oracle.dequant_row(fmt, b, n), np.zeros(n, np.float32))


def _f16(x):
    return np.float32(np.float16(x))


def _block_bound(fmt, wb):
    """Per-element error bound of quantize->dequantize for one block (from the rules)."""
    wb = wb.astype(np.float32)
    if fmt == "q8_0":
        d32 = np.float32(np.abs(wb).max() / np.float32(127))
        return d32 / 2 + 127 * abs(d32 - _f16(d32))
    if fmt == "q4_0":
        d32 = np.float32(np.abs(wb).max() / np.float32(7))
        return d32 / 2 + 7 * abs(d32 - _f16(d32))
    if fmt == "q4_k":
        sub = wb.reshape(8, 32)
        lo = np.minimum(0, sub.min(1))
        s = (sub.max(1) - lo) / 15
        d, dmin = _f16(s.max() / 63), _f16((-lo).max() / 63)
        # half a step plus the shift of the grid from rounding sc and m
        return (s + d / 2).max() / 2 + 15 * d / 2 + dmin / 2
    if fmt == "q5_k":
        sub = wb.reshape(8, 32)
        lo = np.minimum(0, sub.min(1))
        s = (sub.max(1) - lo) / 31
        d, dmin = _f16(s.max() / 63), _f16((-lo).max() / 63)
        return (s + d / 2).max() / 2 + 31 * d / 2 + dmin / 2
    if fmt == "q6_k":
        sub = wb.reshape(16, 16)
        s = np.abs(sub).max(1) / 31
        d = _f16(s.max() / 127)
        return (s + d / 2).max() / 2 + 31 * d / 2
    raise ValueError(fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_roundtrip_error_within_rule_bound(fmt):
    n_blocks = 400
    qk = oracle.BLOCK_ELEMS[fmt]
    w = oracle.gen_normal(0, 99, 0, n_blocks * qk, 0.02)
    b = oracle.quantize_row(fmt, w)
    wh = oracle.dequant_row(fmt, b, w.size)
    err = np.abs(w.astype(np.float64) - wh)
    for i in range(n_blocks):
        sl = slice(i * qk, (i + 1) * qk)
        bound = float(_block_bound(fmt, w[sl])) * (1 + 1e-5) + 1e-12
        assert err[sl].max() <= bound, (fmt, i, err[sl].max(), bound)
    # and the typical error is a fraction of one step (uniform rounding error)
    rel = np.sqrt(np.mean(err**2)) / np.sqrt(np.mean(w.astype(np.float64) ** 2))
    assert rel < {"q8_0": 0.012, "q4_0": 0.2, "q4_k": 0.12, "q6_k": 0.05, "q5_k": 0.06}[fmt], rel


def test_q8_0_absmax_element_maps_to_127():
    w = oracle.gen_normal(1, 5, 0, 32 * 100, 0.02).reshape(100, 32)
    b = oracle.quantize_row("q8_0", w.ravel()).reshape(100, 34)
    for i in range(100):
        k = int(np.argmax(np.abs(w[i])))
        q = np.int8(b[i, 2 + k])
        assert q == (127 if w[i, k] > 0 else -127)


def test_q4_k_all_positive_sub_block_has_zero_min():
    w = np.abs(oracle.gen_normal(2, 5, 0, 256, 0.02))
    b = oracle.quantize_row("q4_k", w)
    bits = int.from_bytes(bytes(b[4:16]), "little")
    assert all(((bits >> (6 * (8 + j))) & 63) == 0 for j in range(8))
    assert b[2] == 0 and b[3] == 0            # dmin = f16(0)


def test_q5_k_fifth_bit_and_all_positive_min():
    # an all-positive sub-block has m = 0 (dmin = 0); its largest element takes code 31
    w = np.abs(oracle.gen_normal(2, 6, 0, 256, 0.02))
    b = oracle.quantize_row("q5_k", w)
    bits = int.from_bytes(bytes(b[4:16]), "little")
    assert all(((bits >> (6 * (8 + j))) & 63) == 0 for j in range(8))
    assert b[2] == 0 and b[3] == 0
    qh, qs = bytes(b[16:48]), bytes(b[48:176])
    code = [((qs[k // 2] >> (4 * (k % 2))) & 15) | (((qh[k // 8] >> (k % 8)) & 1) << 4) for k in range(256)]
    for j in range(8):
        sub = w[32 * j:32 * j + 32]
        assert code[32 * j + int(np.argmax(sub))] >= 30      # top of the 0..31 grid (sc is rounded)
    # every code uses 0..31 and both halves of the grid occur (the fifth bit is used)
    assert max(code) <= 31 and any(c >= 16 for c in code) and any(c < 16 for c in code)


def test_qtensor_rows_is_rowwise_generate_then_quantize():
    rows, cols = 6, 512
    full = oracle.qtensor_rows("q4_k", rows, cols, 3, 77, 0.02)
    part = oracle.qtensor_rows("q4_k", rows, cols, 3, 77, 0.02, row0=2, nrows=3, nthreads=3)
    np.testing.assert_array_equal(full[2:5], part)
    w = oracle.gen_normal(3, 77, 4 * cols, cols, 0.02)
    np.testing.assert_array_equal(full[4], oracle.quantize_row("q4_k", w))


# ------------------------------------------------------------------- GEMV --

def _rand_dyadic_block(fmt, rng):
    """A block with power-of-two scales and its exact dequantized values (Fractions)."""
    if fmt == "q8_0":
        e = int(rng.integers(-6, 0)); q = rng.integers(-127, 128, 32).tolist()
        return pack_q8_0(2.0**e, q), [Fraction(v) * Fraction(2) ** e for v in q]
    if fmt == "q4_0":
        e = int(rng.integers(-6, 0)); q = rng.integers(0, 16, 32).tolist()
        return pack_q4_0(2.0**e, q), [Fraction(v - 8) * Fraction(2) ** e for v in q]
    if fmt == "q4_k":
        e, em = int(rng.integers(-8, -2)), int(rng.integers(-8, -2))
        sc = rng.integers(0, 64, 8).tolist(); m = rng.integers(0, 64, 8).tolist()
        q = rng.integers(0, 16, 256).tolist()
        vals = [Fraction(sc[k // 32] * q[k]) * Fraction(2) ** e - Fraction(m[k // 32]) * Fraction(2) ** em
                for k in range(256)]
        return pack_q4_k(2.0**e, 2.0**em, sc, m, q), vals
    if fmt == "q5_k":
        e, em = int(rng.integers(-8, -2)), int(rng.integers(-8, -2))
        sc = rng.integers(0, 64, 8).tolist(); m = rng.integers(0, 64, 8).tolist()
        q = rng.integers(0, 32, 256).tolist()
        vals = [Fraction(sc[k // 32] * q[k]) * Fraction(2) ** e - Fraction(m[k // 32]) * Fraction(2) ** em
                for k in range(256)]
        return pack_q5_k(2.0**e, 2.0**em, sc, m, q), vals
    e = int(rng.integers(-10, -4)); sc = rng.integers(-128, 128, 16).tolist(); q = rng.integers(0, 64, 256).tolist()
    return pack_q6_k(2.0**e, sc, q), [Fraction(sc[k // 16] * (q[k] - 32)) * Fraction(2) ** e for k in range(256)]


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_brute_force_exact_on_dyadic_data(fmt):
    rng = np.random.default_rng(42)
    qk = oracle.BLOCK_ELEMS[fmt]
    rows, nb = 5, 3
    cols = nb * qk
    blob, vals = bytearray(), []
    for r in range(rows):
        row_vals = []
        for b in range(nb):
            by, v = _rand_dyadic_block(fmt, rng)
            blob += by
            row_vals += v
        vals.append(row_vals)
    x = (rng.integers(-16, 17, cols) / 8).astype(np.float32)
    y = oracle.gemv(fmt, np.frombuffer(bytes(blob), np.uint8), rows, cols, x)
    for r in range(rows):
        exact = sum(vals[r][c] * Fraction(float(x[c])) for c in range(cols))
        assert y[r] == float(exact)     # all terms are dyadic with few bits: the fp64 sum is exact


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_one_hot_reads_a_column(fmt):
    rows, cols = 7, 512
    b = oracle.qtensor_rows(fmt, rows, cols, 0, 5, 0.02)
    W = oracle.dequant_rows(fmt, b, cols)
    for c in (0, 1, 255, 256, 511):
        e = np.zeros(cols, np.float32); e[c] = 1
        np.testing.assert_array_equal(oracle.gemv(fmt, b, rows, cols, e), W[:, c].astype(np.float64))


def test_gemv_threads_do_not_change_results():
    rows, cols = 33, 1024
    b = oracle.qtensor_rows("q6_k", rows, cols, 0, 6, 0.02)
    x = np.random.default_rng(1).standard_normal(cols).astype(np.float32)
    np.testing.assert_array_equal(oracle.gemv("q6_k", b, rows, cols, x, nthreads=1),
                                  oracle.gemv("q6_k", b, rows, cols, x, nthreads=4))

"""Pins for the oracle's dequantised skinny GEMM and argmax (CPU only).

Closed forms and brute force: integer special cases checked with Python
integers / exact rationals, one-hot activations returning a dequantised
column, S-row windows against S single-row calls, and a brute-force argmax.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant, verify


def _half(v):
    return np.asarray(v, dtype=np.float16)


def test_integer_gemm_unit_scales_is_exact():
    rng = np.random.default_rng(0)
    s, n, h = 5, 37, 96
    x = rng.integers(-8, 9, (s, h))
    q = rng.integers(-127, 128, (n, h))
    scales = _half(np.ones((n, h // 32)))
    y = verify.dequant_gemm(_half(x), q.astype(np.int8), scales)
    ref = [[sum(int(x[i, k]) * int(q[j, k]) for k in range(h)) for j in range(n)] for i in range(s)]
    np.testing.assert_array_equal(y, np.array(ref, dtype=np.float32))


def test_power_of_two_block_scales_pin_the_block_index():
    # scales differ per block, so using the wrong block (h//32) changes the result
    rng = np.random.default_rng(1)
    s, n, h = 3, 11, 128
    x = rng.integers(-8, 9, (s, h))
    q = rng.integers(-127, 128, (n, h))
    e = rng.integers(0, 5, (n, h // 32))
    scales = _half(2.0 ** -e)
    y = verify.dequant_gemm(_half(x), q.astype(np.int8), scales)
    for i in range(s):
        for j in range(n):
            exact = sum(Fraction(int(x[i, k]) * int(q[j, k])) / (2 ** int(e[j, k // 32])) for k in range(h))
            assert y[i, j] == np.float32(float(exact))   # exact: fits in 24 bits


def test_one_hot_returns_dequantised_column():
    rng = np.random.default_rng(2)
    n, h = 50, 64
    w = (rng.standard_normal((n, h)) * 0.02).astype(np.float32)
    q, sc = quant.quantize_block32(w, 8)
    for col in (0, 31, 32, 63):
        x = np.zeros((1, h), np.float16)
        x[0, col] = 1.0
        y = verify.dequant_gemm(x, q, sc)
        expect = (q[:, col].astype(np.float64) * sc[:, col // 32].astype(np.float64)).astype(np.float32)
        np.testing.assert_array_equal(y[0], expect)


def test_operands_not_transposed():
    # distinct S, N, H and an asymmetric pattern: x row i hits only weight row i's column i
    s, n, h = 2, 3, 32
    x = np.zeros((s, h), np.float16)
    x[0, 0] = 1.0
    x[1, 5] = 2.0
    q = np.zeros((n, h), np.int8)
    q[2, 0] = 3
    q[1, 5] = -4
    sc = _half(np.ones((n, 1)))
    y = verify.dequant_gemm(x, q, sc)
    np.testing.assert_array_equal(y, np.array([[0, 0, 3], [0, -8, 0]], np.float32))


def test_random_against_exact_rationals():
    rng = np.random.default_rng(3)
    s, n, h = 4, 9, 64
    x = _half(rng.standard_normal((s, h)))
    w = (rng.standard_normal((n, h)) * 0.02).astype(np.float32)
    q, sc = quant.quantize_block32(w, 8)
    y = verify.dequant_gemm(x, q, sc)
    for i in range(s):
        for j in range(n):
            exact = sum(Fraction(float(x[i, k])) * int(q[j, k]) * Fraction(float(sc[j, k // 32]))
                        for k in range(h))
            ref = np.float32(float(exact))
            # float64 accumulation, then one rounding: at most 1 ulp of float32 apart
            assert abs(float(y[i, j]) - float(ref)) <= float(np.spacing(np.abs(ref)))


def test_window_equals_single_rows():
    rng = np.random.default_rng(4)
    s, n, h = 9, 300, 256
    x = _half(rng.standard_normal((s, h)))
    w = (rng.standard_normal((n, h)) * 0.02).astype(np.float32)
    q, sc = quant.quantize_block32(w, 8)
    y = verify.dequant_gemm(x, q, sc)
    for i in range(s):
        yi = verify.dequant_gemm(x[i:i + 1], q, sc)
        d = np.abs(yi[0].astype(np.float64) - y[i].astype(np.float64))
        assert np.all(d <= np.spacing(np.abs(y[i])).astype(np.float64))


def test_int4_dequant_uses_unpacked_codes():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((16, 64)) * 0.02).astype(np.float32)
    q, sc = quant.quantize_block32(w, 4)
    packed = quant.pack_int4(q)
    x = _half(rng.standard_normal((2, 64)))
    a = verify.dequant_gemm(x, q, sc)
    b = verify.dequant_gemm(x, quant.unpack_int4(packed), sc)
    np.testing.assert_array_equal(a, b)


# --- argmax -----------------------------------------------------------------------

def _brute_argmax(row):
    best = 0
    for i in range(1, len(row)):
        if row[i] > row[best]:
            best = i
    return best


def test_argmax_brute_force_and_ties():
    rng = np.random.default_rng(6)
    l = rng.standard_normal((7, 1000)).astype(np.float32)
    l[1, 10] = l[1, 900] = 50.0           # duplicated maximum -> lower index
    l[2, 999] = 50.0                      # maximum in the ragged tail
    l[3, :] = 0.0
    l[3, 5] = -0.0                        # +0 == -0: first index wins
    l[4, :] = -1.0
    l[4, 0] = -0.5
    am = verify.argmax_rows(l)
    for i in range(7):
        assert am[i] == _brute_argmax(list(l[i]))
    assert am[1] == 10 and am[2] == 999 and am[3] == 0 and am[4] == 0


def test_top2_gap():
    l = np.array([[1.0, 3.0, 2.5], [4.0, 4.0, 0.0]])
    np.testing.assert_allclose(verify.top2_gap(l), [0.5, 0.0])

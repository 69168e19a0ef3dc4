"""Pins of the C++ oracle's own building blocks (CPU only).

* binary16 conversions against numpy's (an independent library routine): all
  65536 half patterns widened, and doubles across the range -- ties, the
  subnormal range, the overflow boundary -- rounded once to half;
* the dequantised GEMM sums term by term in reduction order: on small cases it
  equals, bit for bit, a pure-Python loop of IEEE double operations in that
  order (Python floats: one rounding per multiply and per add, no fused
  multiply-add), for fp16 and for float64 activations; and it stays within the
  classical error bound of the exact (rational) sum on random data;
* E2M1 codes and their decoded values give the same GEMM;
* results do not depend on the OpenMP thread count.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import _native as N
from oracle import mlp, quant, verify


def test_half_to_double_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = np.empty(65536, np.float64)
    N.lib().orc_half_to_double(N.ptr(bits), 65536, N.ptr(got))
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _to_half(d):
    d = np.ascontiguousarray(d, dtype=np.float64)
    out = np.empty(d.shape, np.uint16)
    N.lib().orc_double_to_half(N.ptr(d), d.size, N.ptr(out))
    return out


def test_double_to_half_matches_numpy():
    rng = np.random.default_rng(3)
    vals = [rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000)]
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = (h[:-1] + h[1:]) / 2                      # exact ties between neighbours
    vals += [h, mid, -mid, np.nextafter(mid, 0), np.nextafter(mid, 1e9)]
    vals += [np.array([65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
                       3 * 2.0 ** -26, 0.0, -0.0, np.inf, -np.inf])]
    d = np.concatenate(vals)
    got = _to_half(d)
    with np.errstate(over="ignore"):
        ref = d.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def _python_sequential_gemm(x64, w64):
    """y[s][n] = (((0 + x0 w0) + x1 w1) + ...) in Python floats (IEEE doubles)."""
    S, k = x64.shape
    n = w64.shape[0]
    y = np.empty((S, n))
    for s in range(S):
        for r in range(n):
            acc = 0.0
            for h in range(k):
                acc = acc + float(x64[s, h]) * float(w64[r, h])
            y[s, r] = acc
    return y


@pytest.mark.parametrize("bits", [8, 4])
def test_gemm_is_the_sequential_sum(bits):
    rng = np.random.default_rng(bits)
    n, k, S = 7, 96, 3
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    codes, scales = quant.quantize_block32(w, bits)
    x = rng.standard_normal((S, k)).astype(np.float16)
    wq = codes.astype(np.float64) * np.repeat(scales.astype(np.float64), 32, axis=1)   # exact products
    ref = _python_sequential_gemm(x.astype(np.float64), wq)
    assert np.array_equal(verify.dequant_gemm64(x, codes, scales), ref)


def test_gemm_of_float64_activations_is_the_sequential_sum():
    # the MoE's down projection takes float64 h: products are rounded, the
    # order of the sum still decides every bit
    rng = np.random.default_rng(11)
    n, k, S = 5, 64, 2
    codes, scales = quant.quantize_block32((rng.standard_normal((n, k)) * 0.02).astype(np.float32), 8)
    h = rng.standard_normal((S, k)) * 1e-3
    wq = codes.astype(np.float64) * np.repeat(scales.astype(np.float64), 32, axis=1)
    assert np.array_equal(verify.dequant_gemm64(h, codes, scales), _python_sequential_gemm(h, wq))


def test_gemm_within_the_summation_bound_of_the_exact_sum():
    rng = np.random.default_rng(5)
    n, k, S = 6, 2560, 2
    codes, scales = quant.quantize_block32((rng.standard_normal((n, k)) * 0.02).astype(np.float32), 8)
    x = rng.standard_normal((S, k)).astype(np.float16)
    y = verify.dequant_gemm64(x, codes, scales)
    eps = 2.0 ** -53
    for s in range(S):
        for r in range(n):
            terms = [Fraction(float(x[s, h])) * int(codes[r, h]) * Fraction(float(scales[r, h // 32]))
                     for h in range(k)]
            exact = sum(terms)
            bound = (k - 1) * eps * float(sum(abs(t) for t in terms)) * 1.01
            assert abs(Fraction(y[s, r]) - exact) <= Fraction(bound)


def test_e2m1_codes_and_values_give_the_same_gemm():
    rng = np.random.default_rng(8)
    w = (rng.standard_normal((40, 256)) * 0.02).astype(np.float32)
    c4, scales = quant.quantize_fp4_block32(w)
    x = rng.standard_normal((4, 256)).astype(np.float16)
    a = verify.dequant_gemm64(x, c4, scales)
    b = verify.dequant_gemm64(x, quant.decode_e2m1(c4), scales)
    assert np.array_equal(a, b)


def test_uint8_codes_must_be_e2m1():
    with pytest.raises(ValueError):
        verify.dequant_gemm64(np.zeros((1, 32), np.float16), np.full((1, 32), 200, np.uint8),
                              np.ones((1, 1), np.float16))


def test_results_do_not_depend_on_the_thread_count():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((1000, 512)) * 0.02).astype(np.float32)
    x = rng.standard_normal((9, 512)).astype(np.float16)
    prev = oracle.set_threads(1)
    try:
        c1, s1 = quant.quantize_block32(w, 4)
        y1 = verify.dequant_gemm64(x, c1, s1)
        h1 = mlp.swiglu64(x, c1, s1, c1[::-1].copy(), s1[::-1].copy())
        oracle.set_threads(max(4, prev))
        c2, s2 = quant.quantize_block32(w, 4)
        y2 = verify.dequant_gemm64(x, c2, s2)
        h2 = mlp.swiglu64(x, c2, s2, c2[::-1].copy(), s2[::-1].copy())
    finally:
        oracle.set_threads(prev)
    assert np.array_equal(c1, c2) and np.array_equal(s1.view(np.uint16), s2.view(np.uint16))
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)

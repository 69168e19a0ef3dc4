"""Pins for the oracle's SwiGLU and gathered-expert MoE (CPU only)."""
import mpmath
import numpy as np
import pytest

from oracle import mlp, quant, verify


def test_silu_closed_forms():
    assert mlp.silu(0.0) == 0.0
    # sigmoid(ln 3) = 3/4 exactly in the reals
    t = float(mpmath.log(3))
    assert abs(float(mlp.silu(t)) - 0.75 * t) < 1e-15
    for v in (-30.0, -3.7, -0.1, 0.2, 1.0, 5.5, 40.0):
        ref = mpmath.mpf(v) / (1 + mpmath.e ** (-mpmath.mpf(v)))
        assert abs(float(mlp.silu(v)) - float(ref)) <= 1e-15 * max(1.0, abs(v))


def test_silu_reflection_identity():
    # SiLU(-t) = SiLU(t) - t catches a sign error in the exponent
    t = np.linspace(-20, 20, 401)
    np.testing.assert_allclose(mlp.silu(-t), mlp.silu(t) - t, rtol=0, atol=1e-12)


def _quantized(rng, n, h, bits):
    w = (rng.standard_normal((n, h)) * 0.02).astype(np.float32)
    return quant.quantize_block32(w, bits)


def test_swiglu_one_hot_closed_form():
    rng = np.random.default_rng(0)
    n, h = 40, 64
    gq, gs = _quantized(rng, n, h, 8)
    uq, us = _quantized(rng, n, h, 8)
    x = np.zeros((1, h), np.float16)
    x[0, 37] = 1.0
    hh = mlp.swiglu64(x, gq, gs, uq, us)
    g = gq[:, 37].astype(np.float64) * gs[:, 1].astype(np.float64)
    u = uq[:, 37].astype(np.float64) * us[:, 1].astype(np.float64)
    np.testing.assert_allclose(hh[0], g / (1 + np.exp(-g)) * u, rtol=1e-15, atol=0)
    # zero input -> SiLU(0) * 0 = 0
    assert np.all(mlp.swiglu64(np.zeros((2, h), np.float16), gq, gs, uq, us) == 0)


def test_swiglu_fp16_output_is_one_rounding():
    rng = np.random.default_rng(1)
    gq, gs = _quantized(rng, 64, 128, 8)
    uq, us = _quantized(rng, 64, 128, 8)
    x = rng.standard_normal((3, 128)).astype(np.float16)
    h64 = mlp.swiglu64(x, gq, gs, uq, us)
    h16 = mlp.qlinear_swiglu(x, gq, gs, uq, us)
    assert h16.dtype == np.float16
    np.testing.assert_array_equal(h16, h64.astype(np.float16))


def _brute_topk(row, k):
    idx = list(range(len(row)))
    chosen = []
    for _ in range(k):
        best = None
        for i in idx:
            if i in chosen:
                continue
            if best is None or row[i] > row[best]:
                best = i
        chosen.append(best)
    return chosen


def test_route_topk_brute_force_and_ties():
    rng = np.random.default_rng(2)
    r = rng.standard_normal((17, 256)).astype(np.float32)
    r[3, [5, 9, 200]] = 9.0            # ties -> lower id first
    ids, w = mlp.route_topk(r, 8)
    for s in range(17):
        assert list(ids[s]) == _brute_topk(list(r[s]), 8)
    assert list(ids[3][:3]) == [5, 9, 200]
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(w[3][:3], w[3][0])
    # equal logits -> uniform weights
    ids, w = mlp.route_topk(np.zeros((2, 16), np.float32), 8)
    assert list(ids[0]) == list(range(8))
    np.testing.assert_allclose(w, 1 / 8, rtol=0, atol=1e-15)


def test_group_by_expert():
    ids = np.array([[3, 1], [1, 0], [2, 3]])
    off, rows, slots = mlp.group_by_expert(ids, 5)
    assert list(off) == [0, 1, 3, 4, 6, 6]
    assert list(rows) == [1, 0, 1, 2, 0, 2]
    assert list(slots) == [1, 1, 0, 0, 0, 1]


def _moe_weights(rng, e, inter, hidden, bits):
    g = _quantized(rng, e * inter, hidden, bits)
    u = _quantized(rng, e * inter, hidden, bits)
    d = _quantized(rng, e * hidden, inter, bits)
    return g, u, d


def test_moe_top1_dominant_expert_equals_that_expert():
    rng = np.random.default_rng(3)
    e, inter, hidden = 8, 32, 64
    g, u, d = _moe_weights(rng, e, inter, hidden, 4)
    x = rng.standard_normal((3, hidden)).astype(np.float16)
    router = rng.standard_normal((3, e)).astype(np.float32)
    router[:, 5] = 50.0
    out, ids, w = mlp.moe_forward(x, router, g, u, d, e, inter, hidden, 1)
    assert np.all(ids[:, 0] == 5) and np.all(w == 1.0)
    # the same expert as a dense SwiGLU + down projection (separate code path)
    gs = slice(5 * inter, 6 * inter)
    ds = slice(5 * hidden, 6 * hidden)
    hh = mlp.swiglu64(x, g[0][gs], g[1][gs], u[0][gs], u[1][gs])
    y = hh @ quant.dequantize(d[0][ds], d[1][ds]).T
    np.testing.assert_allclose(out, y.astype(np.float32), rtol=1e-6, atol=1e-7)


def test_moe_identical_experts_equal_one_expert():
    rng = np.random.default_rng(4)
    e, inter, hidden = 16, 32, 64
    g1, u1, d1 = _moe_weights(rng, 1, inter, hidden, 4)
    tile = lambda t: (np.tile(t[0], (e, 1)), np.tile(t[1], (e, 1)))
    g, u, d = tile(g1), tile(u1), tile(d1)
    x = rng.standard_normal((5, hidden)).astype(np.float16)
    router = rng.standard_normal((5, e)).astype(np.float32)
    out, _, _ = mlp.moe_forward(x, router, g, u, d, e, inter, hidden, 8)
    hh = mlp.swiglu64(x, g1[0], g1[1], u1[0], u1[1])
    y = hh @ quant.dequantize(d1[0], d1[1]).T
    np.testing.assert_allclose(out, y.astype(np.float32), rtol=1e-5, atol=1e-6)


def test_moe_is_weighted_sum_of_expert_outputs():
    rng = np.random.default_rng(5)
    e, inter, hidden, k = 8, 32, 64, 3
    g, u, d = _moe_weights(rng, e, inter, hidden, 8)
    x = rng.standard_normal((2, hidden)).astype(np.float16)
    router = rng.standard_normal((2, e)).astype(np.float32)
    out, ids, w = mlp.moe_forward(x, router, g, u, d, e, inter, hidden, k)
    for s in range(2):
        acc = np.zeros(hidden)
        for j in range(k):
            ex = int(ids[s, j])
            gs = slice(ex * inter, (ex + 1) * inter)
            ds = slice(ex * hidden, (ex + 1) * hidden)
            hh = mlp.swiglu64(x[s:s + 1], g[0][gs], g[1][gs], u[0][gs], u[1][gs])
            acc += w[s, j] * (hh @ quant.dequantize(d[0][ds], d[1][ds]).T)[0]
        np.testing.assert_allclose(out[s], acc.astype(np.float32), rtol=1e-6, atol=1e-7)

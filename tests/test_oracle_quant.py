"""Pins for the oracle's per-block-32 quantiser (CPU only).

The quantiser is pinned by (1) hand-worked blocks whose codes and fp16 scale
bits were derived by hand (tests/golden/quant_block32_worked.txt), (2) the
round-trip bound and the absmax invariants that the rule implies, and (3) an
exact-rational re-derivation of random tiny blocks that rounds with integer
arithmetic and with CPython's own fp16 packing instead of numpy's casts.
"""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_block32_worked.txt")


def _half_value(bits: int) -> float:
    return struct.unpack("<e", struct.pack("<H", bits))[0]


def _load_golden():
    blocks, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("block "):
            _, name, bits = line.split()
            cur = {"name": name, "bits": int(bits.split("=")[1])}
            blocks.append(cur)
            continue
        key, val = line.split(":", 1)
        cur[key] = val.split()
    for b in blocks:
        s = _half_value(int(b["scale"][0], 16))
        b["scale_bits"] = int(b["scale"][0], 16)
        b["w"] = np.array([eval(t, {"S": s}) for t in b["w"]], dtype=np.float64).astype(np.float32)
        b["codes"] = np.array([int(t) for t in b["codes"]], dtype=np.int8)
        if "packed" in b:
            b["packed"] = np.array([int(t, 16) for t in b["packed"]], dtype=np.uint8)
    return blocks


@pytest.mark.parametrize("blk", _load_golden(), ids=lambda b: b["name"])
def test_worked_blocks(blk):
    assert blk["w"].shape == (32,)
    codes, scales = quant.quantize_block32(blk["w"][None, :], blk["bits"])
    assert int(scales.view(np.uint16)[0, 0]) == blk["scale_bits"]
    np.testing.assert_array_equal(codes[0], blk["codes"])
    if "packed" in blk:
        np.testing.assert_array_equal(quant.pack_int4(codes)[0], blk["packed"])
        np.testing.assert_array_equal(quant.unpack_int4(blk["packed"][None, :])[0], blk["codes"])


# --- exact re-derivation -------------------------------------------------------

def fp32_rne(x: Fraction) -> float:
    """Round a rational to the nearest float32, ties to even (integer arithmetic)."""
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                     # below: fixed subnormal quantum
    quantum = Fraction(2) ** (e - 23)
    q = a / quantum
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(n * quantum)


def half_bits_of(v: float) -> int:
    return struct.unpack("<H", struct.pack("<e", v))[0]


def round_half_even(v: float) -> int:
    return round(v)  # Python's round() on a float is round-half-to-even


def exact_quantize_block(w32, qmax):
    m = max(abs(Fraction(float(v))) for v in w32)
    s32 = fp32_rne(m / qmax)
    sbits = half_bits_of(s32)
    s16 = _half_value(sbits)
    if s16 == 0:
        return sbits, [0] * len(w32)
    codes = []
    for v in w32:
        r = fp32_rne(Fraction(float(v)) / Fraction(s16))
        codes.append(max(-qmax, min(qmax, round_half_even(r))))
    return sbits, codes


@pytest.mark.parametrize("bits", [8, 4])
def test_exact_rederivation_random_blocks(bits):
    rng = np.random.default_rng(1234 + bits)
    qmax = quant.QMAX[bits]
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-6, 1)
        w = (rng.standard_normal(32) * scale).astype(np.float32)
        if trial % 7 == 0:   # plant exact ties relative to a power-of-two scale
            w = (rng.integers(-2 * qmax, 2 * qmax + 1, 32) / 2.0 * 2.0 ** -5).astype(np.float32)
        codes, scales = quant.quantize_block32(w[None, :], bits)
        sbits, ref = exact_quantize_block(w, qmax)
        assert int(scales.view(np.uint16)[0, 0]) == sbits
        np.testing.assert_array_equal(codes[0], np.array(ref, dtype=np.int8))


# --- invariants -----------------------------------------------------------------

@pytest.mark.parametrize("bits", [8, 4])
def test_roundtrip_bound_and_absmax(bits):
    rng = np.random.default_rng(7 + bits)
    qmax = quant.QMAX[bits]
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    codes, scales = quant.quantize_block32(w, bits)
    assert codes.min() >= -qmax and codes.max() <= qmax
    s = np.repeat(scales.astype(np.float64), 32, axis=1)
    err = np.abs(w.astype(np.float64) - codes.astype(np.float64) * s)
    # |w - q s16| <= s16/2 up to the float32 rounding of w / s16 (<= Q * 2^-24 relative)
    assert np.all(err <= s * (0.5 + qmax * 2.0 ** -23))
    # every nonzero block holds a code of magnitude exactly Q
    blk = np.abs(codes.reshape(64, 8, 32)).max(axis=2)
    assert np.all(blk == qmax)
    # re-quantising the dequantised block reproduces the codes and the scale
    deq = (codes.astype(np.float64) * s).astype(np.float32)
    codes2, scales2 = quant.quantize_block32(deq, bits)
    np.testing.assert_array_equal(codes2, codes)
    np.testing.assert_array_equal(scales2.view(np.uint16), scales.view(np.uint16))


def test_scale_is_absmax_over_q_rounded_to_fp16():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((8, 64)) * 0.02).astype(np.float32)
    _, scales = quant.quantize_block32(w, 8)
    m = np.abs(w.reshape(8, 2, 32)).max(axis=2)
    for i in range(8):
        for b in range(2):
            s32 = fp32_rne(Fraction(float(m[i, b])) / 127)
            assert int(scales.view(np.uint16)[i, b]) == half_bits_of(s32)


def test_block_boundaries_are_along_the_row():
    # one large weight per block: only that block's scale grows
    w = np.full((2, 96), 1e-3, dtype=np.float32)
    w[0, 40] = 0.5
    w[1, 95] = -0.25
    codes, scales = quant.quantize_block32(w, 8)
    s = scales.astype(np.float32)
    assert s[0, 1] > 10 * s[0, 0] and s[0, 1] > 10 * s[0, 2]
    assert s[1, 2] > 10 * s[1, 0] and s[1, 0] == s[1, 1]
    assert codes[0, 40] == 127 and codes[1, 95] == -127


def test_int4_pack_roundtrip_and_nibble_order():
    c = np.array([[1, -1, -8, 7, 0, -3]], dtype=np.int8)
    p = quant.pack_int4(c)
    assert list(p[0]) == [0xF1, 0x78, 0xD0]
    np.testing.assert_array_equal(quant.unpack_int4(p), c)
    rng = np.random.default_rng(5)
    c = rng.integers(-8, 8, (17, 64)).astype(np.int8)
    np.testing.assert_array_equal(quant.unpack_int4(quant.pack_int4(c)), c)


def test_rejects_ragged_block():
    with pytest.raises(ValueError):
        quant.quantize_block32(np.zeros((2, 40), np.float32), 8)

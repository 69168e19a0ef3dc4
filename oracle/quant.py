"""Per-block-32 absmax symmetric weight quantisation (oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product path; it shares no code with it.

Follows "Riding Apple's pipelined GPU engine -- 3.5x over a hand-rolled loop,
zero custom kernels", section "Quantization on the GPU delegate": the ship
configuration is *int8 linear per-block-32 (no LUT)*, the int4 class is
*linear per-block-32*, *q4_0 is per-block-32 absmax symmetric int4*, and big
vocabulary heads are quantised *absmax symmetric, never with clipping*.

Readings taken where the page is silent (all arithmetic float32 unless said):

* block = 32 consecutive weights of one output row along the reduction
  (hidden) axis; Q = 127 for int8, Q = 7 for int4;
* m = max |w| over the block; s32 = m / Q (IEEE float32 division);
  s16 = s32 rounded to fp16 (round-to-nearest-even); the stored scale is s16;
* q = clamp(rint(w / float32(s16)), -Q, Q), rint = round half to even, the
  division again IEEE float32;  codes are taken against the *rounded* scale so
  that dequantisation (q * s16) is self-consistent;
* s16 == 0 (an all-zero block, or a scale that underflows fp16) gives all
  codes 0;
* int4 storage: two's-complement nibbles, two per byte, the even element of
  each pair in the low nibble (byte i of a row holds elements 2i and 2i+1).
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
QMAX = {8: 127, 4: 7}


def quantize_block32(w: np.ndarray, bits: int):
    """Quantise fp32 ``w[N, H]`` (H % 32 == 0) per block of 32 along H.

    Returns ``(codes int8 [N, H], scales fp16 [N, H/32])``.  For ``bits == 4``
    the codes are still returned unpacked (one int8 per weight, in [-7, 7]);
    ``pack_int4`` produces the two-per-byte storage.
    """
    w = np.asarray(w, dtype=np.float32)
    n, h = w.shape
    if h % BLOCK:
        raise ValueError("reduction length must be a multiple of 32")
    q_max = QMAX[bits]
    blocks = w.reshape(n, h // BLOCK, BLOCK)
    m = np.max(np.abs(blocks), axis=2)                       # float32, exact
    s32 = m / np.float32(q_max)                              # IEEE fp32 divide
    s16 = s32.astype(np.float16)                             # RNE to fp16
    sf = s16.astype(np.float32)[:, :, None]                  # exact widening
    with np.errstate(divide="ignore", invalid="ignore"):
        r = blocks / sf                                      # IEEE fp32 divide
    q = np.rint(r)                                           # half to even
    q = np.clip(q, -q_max, q_max)
    q = np.where(sf == 0, np.float32(0), q)
    return q.astype(np.int8).reshape(n, h), s16


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Pack int4 codes ``[N, H]`` (values in [-8, 7]) into bytes ``[N, H/2]``.

    Byte i of a row = (c[2i] & 0xF) | ((c[2i+1] & 0xF) << 4).
    """
    c = np.asarray(codes, dtype=np.int16)
    if c.shape[1] % 2:
        raise ValueError("row length must be even to pack int4")
    lo = c[:, 0::2] & 0xF
    hi = c[:, 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Inverse of ``pack_int4``: bytes ``[N, H/2]`` -> int8 codes ``[N, H]``."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    lo = b & 0xF
    hi = (b >> 4) & 0xF
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    n, half = b.shape
    out = np.empty((n, 2 * half), dtype=np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantised weights in float64: w[n, h] = q[n, h] * s16[n, h // 32].

    Each product is exact in float64 (8 + 11 significant bits).
    """
    q = np.asarray(codes).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    return q * np.repeat(s, BLOCK, axis=1)


# ---------------------------------------------------------------------------
# FP4 (E2M1) weights: the pages' "quality-safe 4-bit" lever ("Flagship
# dramatic-speedup plan -- the full stackable tuning set", section "Axis 1 --
# per-forward BYTE reduction", lever 1c: FP4 (E2M1) at near-FP8 quality).
#
# E2M1 as in the OCP Microscaling Formats specification v1.0: sign, 2 exponent
# bits (bias 1), 1 mantissa bit; magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3,
# 4, 6; no infinities or NaNs.  Code = (sign << 3) | magnitude index.
#
# Readings (the page names the format only): the same per-block-32 absmax
# layout as the integer types with an fp16 scale -- s32 = max|w| / 6 (fp32
# division), s16 = fp16 RNE of s32, r = w / s16 (fp32 division); the code is
# r rounded to the nearest E2M1 magnitude with ties to the even mantissa bit
# (IEEE round-half-even on the E2M1 grid), saturating above 6; zero is always
# the +0 code; s16 == 0 gives all codes 0.  Storage: two codes per byte, the
# even element in the low nibble, like int4.
# ---------------------------------------------------------------------------

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
FP4_MAX = 6.0
# magnitude index = number of thresholds passed; ">" at a tie that rounds down
# (to an even mantissa), ">=" where the tie rounds up
_FP4_UP = ((0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False), (3.5, True), (5.0, False))


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """float64 values of E2M1 codes (0..15)."""
    c = np.asarray(codes, dtype=np.int64)
    mag = E2M1[c & 7]
    return np.where(c & 8, -mag, mag)


def encode_e2m1(r: np.ndarray) -> np.ndarray:
    """E2M1 codes (uint8) of float32 ratios r, round-half-even, saturating."""
    r = np.asarray(r, dtype=np.float32)
    a = np.abs(r)
    idx = np.zeros(r.shape, dtype=np.int64)
    for t, inclusive in _FP4_UP:
        idx += (a >= np.float32(t)) if inclusive else (a > np.float32(t))
    sign = (r < 0) & (idx > 0)
    return (idx | np.where(sign, 8, 0)).astype(np.uint8)


def quantize_fp4_block32(w: np.ndarray):
    """Quantise fp32 ``w[N, H]`` to E2M1 per block of 32 along H.

    Returns ``(codes uint8 [N, H] (0..15, unpacked), scales fp16 [N, H/32])``.
    """
    w = np.asarray(w, dtype=np.float32)
    n, h = w.shape
    if h % BLOCK:
        raise ValueError("reduction length must be a multiple of 32")
    blocks = w.reshape(n, h // BLOCK, BLOCK)
    m = np.max(np.abs(blocks), axis=2)
    s16 = (m / np.float32(FP4_MAX)).astype(np.float16)
    sf = s16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = blocks / sf
    codes = encode_e2m1(r)
    codes = np.where(sf == 0, np.uint8(0), codes)
    return codes.reshape(n, h), s16


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Two 4-bit codes (0..15) per byte, the even element in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[1] % 2:
        raise ValueError("row length must be even")
    return ((c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)).astype(np.uint8)

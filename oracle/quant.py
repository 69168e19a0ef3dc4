"""Per-block-32 absmax symmetric weight quantisation (oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product path; it shares no code with it.
The arithmetic is in the plain C++ oracle (``oracle/src/oracle.cpp``); this
module only marshals arrays.

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

FP4 (E2M1) weights: the pages' "quality-safe 4-bit" lever ("Flagship
dramatic-speedup plan -- the full stackable tuning set", section "Axis 1 --
per-forward BYTE reduction", lever 1c: FP4 (E2M1) at near-FP8 quality).  E2M1
as in the OCP Microscaling Formats specification v1.0: sign, 2 exponent bits
(bias 1), 1 mantissa bit; magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6; no
infinities or NaNs.  Code = (sign << 3) | magnitude index.  Readings: the same
per-block-32 absmax layout with an fp16 scale -- s32 = max|w| / 6, s16 = fp16
RNE of s32, r = w / s16 (fp32 division); the code is r rounded to the nearest
E2M1 magnitude with ties to the even mantissa bit, saturating above 6; zero is
always the +0 code; s16 == 0 gives all codes 0.  Storage as int4.
"""
from __future__ import annotations

import numpy as np

from . import _native as N

BLOCK = 32
QMAX = {8: 127, 4: 7}
FP4_MAX = 6.0


def quantize_block32(w: np.ndarray, bits: int):
    """Quantise fp32 ``w[N, H]`` (H % 32 == 0) per block of 32 along H.

    Returns ``(codes int8 [N, H], scales fp16 [N, H/32])``.  For ``bits == 4``
    the codes are still returned unpacked (one int8 per weight, in [-7, 7]);
    ``pack_int4`` produces the two-per-byte storage.
    """
    w = N.as_c(w, np.float32)
    n, h = w.shape
    if h % BLOCK or bits not in QMAX:
        raise ValueError("reduction length must be a multiple of 32; bits 8 or 4")
    codes = np.empty((n, h), dtype=np.int8)
    scales = np.empty((n, h // BLOCK), dtype=np.uint16)
    N.check(N.lib().orc_quantize_block32(N.ptr(w), n, h, bits, N.ptr(codes), N.ptr(scales), N.threads()),
            "quantize_block32")
    return codes, scales.view(np.float16)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Two 4-bit codes per byte, the even element in the low nibble."""
    c = np.ascontiguousarray(np.asarray(codes)).view(np.uint8) if np.asarray(codes).dtype == np.int8 \
        else N.as_c(codes, np.uint8)
    n, k = c.shape
    if k % 2:
        raise ValueError("row length must be even")
    out = np.empty((n, k // 2), dtype=np.uint8)
    N.check(N.lib().orc_pack_nibbles(N.ptr(c), n, k, N.ptr(out)), "pack_nibbles")
    return out


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Pack int4 codes ``[N, H]`` (values in [-8, 7]) into bytes ``[N, H/2]``:
    byte i of a row = (c[2i] & 0xF) | ((c[2i+1] & 0xF) << 4)."""
    return pack_nibbles(N.as_c(codes, np.int8))


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Inverse of ``pack_int4``: bytes ``[N, H/2]`` -> int8 codes ``[N, H]``."""
    p = N.as_c(packed, np.uint8)
    n, half = p.shape
    out = np.empty((n, 2 * half), dtype=np.int8)
    N.lib().orc_unpack_int4(N.ptr(p), n, 2 * half, N.ptr(out))
    return out


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantised weights in float64: w[n, h] = q[n, h] * s16[n, h // 32]
    (codes: int8 integer codes, uint8 E2M1 codes or float64 values)."""
    kind, c = N.code_kind(codes)
    s = N.half_bits(scales)
    n, k = c.shape
    out = np.empty((n, k), dtype=np.float64)
    N.lib().orc_dequantize(kind, N.ptr(c), N.ptr(s), n, k, N.ptr(out))
    return out


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """float64 values of E2M1 codes (0..15)."""
    c = N.as_c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    N.lib().orc_e2m1_values(N.ptr(c), c.size, N.ptr(out))
    return out


E2M1 = decode_e2m1(np.arange(8))


def encode_e2m1(r: np.ndarray) -> np.ndarray:
    """E2M1 codes (uint8) of float32 ratios r, round-half-even, saturating."""
    r = N.as_c(r, np.float32)
    out = np.empty(r.shape, dtype=np.uint8)
    N.lib().orc_e2m1_encode(N.ptr(r), r.size, N.ptr(out))
    return out


def quantize_fp4_block32(w: np.ndarray):
    """Quantise fp32 ``w[N, H]`` to E2M1 per block of 32 along H.

    Returns ``(codes uint8 [N, H] (0..15, unpacked), scales fp16 [N, H/32])``.
    """
    w = N.as_c(w, np.float32)
    n, h = w.shape
    if h % BLOCK:
        raise ValueError("reduction length must be a multiple of 32")
    codes = np.empty((n, h), dtype=np.uint8)
    scales = np.empty((n, h // BLOCK), dtype=np.uint16)
    N.check(N.lib().orc_quantize_fp4_block32(N.ptr(w), n, h, N.ptr(codes), N.ptr(scales), N.threads()),
            "quantize_fp4_block32")
    return codes, scales.view(np.float16)

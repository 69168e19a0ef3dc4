"""Per-block-32 absmax symmetric weight quantisation (oracle).

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

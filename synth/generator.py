"""Seeded, counter-based synthetic input generator.

This module is the only code shared by the CPU oracle side (tests) and the
GPU side (tests, bench).  It draws random numbers and nothing else: no
quantisation, no matmul, no argmax, no accept rule lives here.

Generator
---------
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; constants as published by Vigna) used as a
counter-based hash: element ``i`` of a stream with seed ``k`` is
``mix(k + (i + 1) * GOLDEN)``.  Normals come from the Box-Muller transform
(Box & Muller, 1958) on pairs of uniforms: pair ``p`` uses counters ``2p``
(radius) and ``2p + 1`` (angle).  Every element is a pure function of
(seed, index), so any slice can be produced independently and in chunks.

All integer arithmetic is uint64 modulo 2**64; float arithmetic is float64
(numpy), rounded once to the requested storage type.
"""
from __future__ import annotations

import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30 = np.uint64(30)
_S27 = np.uint64(27)
_S31 = np.uint64(31)
_S11 = np.uint64(11)
_S32 = np.uint64(32)
_TWO_M53 = float(2.0 ** -53)

_CHUNK = 1 << 22  # elements per vectorised chunk (keeps temporaries cache sized)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, in place on a uint64 array."""
    z ^= z >> _S30
    z *= _M1
    z ^= z >> _S27
    z *= _M2
    z ^= z >> _S31
    return z


def mix_scalar(v: int) -> int:
    """SplitMix64 finaliser on one Python int (mod 2**64)."""
    m = (1 << 64) - 1
    z = v & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_seed(*key: int) -> int:
    """Derive a 64-bit stream seed from a tuple of small integers."""
    h = 0x243F6A8885A308D3
    for v in key:
        h = mix_scalar(h ^ (int(v) & ((1 << 64) - 1)))
    return h


class _Scratch:
    """Reusable chunk buffers (fresh allocations are page-fault bound)."""

    def __init__(self, n: int):
        self.idx = np.empty(n, dtype=np.uint64)
        self.z = np.empty(n, dtype=np.uint64)
        self.t = np.empty(n, dtype=np.uint64)
        self.f = np.empty(n, dtype=np.float64)
        self.g = np.empty(n, dtype=np.float64)
        self.h = np.empty(n, dtype=np.float64)
        self.base = np.arange(1, n + 1, dtype=np.uint64)


_tls = threading.local()


def _get_scratch(n: int) -> _Scratch:
    sc = getattr(_tls, "scratch", None)
    if sc is None or sc.idx.size < n:
        size = 1024
        while size < n:
            size *= 2
        sc = _Scratch(min(max(size, n), max(n, _CHUNK)))
        _tls.scratch = sc
    return sc


def _workers() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _u64_into(seed: int, start: int, count: int, sc: _Scratch) -> np.ndarray:
    """Counters ``start .. start+count-1`` of stream ``seed``, into scratch."""
    idx = sc.idx[:count]
    z = sc.z[:count]
    t = sc.t[:count]
    with np.errstate(over="ignore"):
        np.add(sc.base[:count], np.uint64(start), out=idx)   # i + 1
        np.multiply(idx, GOLDEN, out=z)
        np.add(z, np.uint64(seed), out=z)
        np.right_shift(z, _S30, out=t)
        np.bitwise_xor(z, t, out=z)
        np.multiply(z, _M1, out=z)
        np.right_shift(z, _S27, out=t)
        np.bitwise_xor(z, t, out=z)
        np.multiply(z, _M2, out=z)
        np.right_shift(z, _S31, out=t)
        np.bitwise_xor(z, t, out=z)
    return z


def raw_u64(seed: int, start: int, count: int) -> np.ndarray:
    """Counters ``start .. start+count-1`` of stream ``seed`` as uint64."""
    out = np.empty(count, dtype=np.uint64)
    p = 0
    while p < count:
        m = min(_CHUNK, count - p)
        out[p:p + m] = _u64_into(seed, start + p, m, _get_scratch(m))
        p += m
    return out


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Uniforms in [0, 1) with 53 random bits (float64)."""
    return (raw_u64(seed, start, count) >> _S11).astype(np.float64) * _TWO_M53


def _normal_chunk(seed: int, p0: int, npairs: int, sigma: float, out: np.ndarray) -> None:
    """Box-Muller normals for pairs ``p0 .. p0+npairs-1`` times ``sigma``.

    With r = sigma * sqrt(-2 ln u1) and t = 2 pi u2 (all float64), the pair is
    (r cos t, r sin t).

    Writes ``out[0::2]`` (cosine branch) and ``out[1::2]`` (sine branch);
    ``out`` has 2*npairs elements, or 2*npairs-1 for a ragged final pair.
    """
    sc = _get_scratch(2 * npairs)
    z = _u64_into(seed, 2 * p0, 2 * npairs, sc).reshape(npairs, 2)
    t = sc.t[: 2 * npairs].reshape(npairs, 2)
    f = sc.f[:npairs]
    g = sc.g[:npairs]
    # radius: u1 in (0, 1]
    np.right_shift(z[:, 0], _S11, out=t[:, 0])
    np.add(t[:, 0], np.uint64(1), out=t[:, 0])
    np.multiply(t[:, 0], _TWO_M53, out=f, casting="unsafe")
    np.log(f, out=f)
    np.multiply(f, -2.0, out=f)
    np.sqrt(f, out=f)
    np.multiply(f, sigma, out=f)
    # angle: u2 in [0, 1)
    np.right_shift(z[:, 1], _S11, out=t[:, 1])
    np.multiply(t[:, 1], _TWO_M53 * 2.0 * np.pi, out=g, casting="unsafe")
    n = out.size
    c = sc.h[:npairs]
    np.cos(g, out=c)
    np.multiply(c, f, out=c)
    out[0::2] = c[: (n + 1) // 2]
    np.sin(g, out=g)
    np.multiply(g, f, out=g)
    out[1::2] = g[: n // 2]


def normal(seed: int, shape, sigma: float = 1.0, dtype=np.float32) -> np.ndarray:
    """i.i.d. N(0, sigma^2) values, computed in float64, rounded once to ``dtype``."""
    if not isinstance(shape, tuple):
        shape = tuple(int(s) for s in np.atleast_1d(shape))
    n = int(np.prod(shape, dtype=np.int64)) if len(shape) else 1
    out = np.empty(n, dtype=dtype)
    npairs_total = (n + 1) // 2
    step = _CHUNK // 2
    starts = list(range(0, npairs_total, step))

    def run(p: int) -> None:
        m = min(step, npairs_total - p)
        lo = 2 * p
        hi = min(n, lo + 2 * m)
        _normal_chunk(seed, p, m, float(sigma), out[lo:hi])

    # Chunks are independent functions of (seed, counter); numpy ufuncs drop
    # the GIL, so threads give a parallel fill with identical values.
    if len(starts) > 1 and _workers() > 1:
        with ThreadPoolExecutor(max_workers=_workers()) as ex:
            list(ex.map(run, starts))
    else:
        for p in starts:
            run(p)
    return out.reshape(shape)


def randint(seed: int, count: int, high: int, start: int = 0) -> np.ndarray:
    """Integers uniform on {0 .. high-1} (multiply-high of the top 32 bits), int64."""
    assert 0 < high < (1 << 32)
    z = raw_u64(seed, start, count) >> _S32
    with np.errstate(over="ignore"):
        return ((z * np.uint64(high)) >> _S32).astype(np.int64)

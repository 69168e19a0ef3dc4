"""Sampling (temperature > 0) verify of speculative decoding -- TEST
INFRASTRUCTURE ONLY (imported by tests/, __graft_entry__.smoke() and the CPU
baseline of bench.py; never by the product path).

The pages defer it: "Stream C -- Speculative decoding: feasibility verdict +
implementation plan", section "Deferred / harder": a lossless sampling verify
needs the probabilities and a resample from the residual distribution, not the
argmax.  The method is speculative sampling (Leviathan, Kalman & Matias, "Fast
Inference from Transformers via Speculative Decoding", ICML 2023; Chen et al.,
"Accelerating Large Language Model Decoding with Speculative Sampling", 2023):
draft token d drawn from q is kept with probability min(1, p(d) / q(d)); at the
first rejection the token is drawn from norm(max(0, p - q)); when every draft
is kept the bonus token is drawn from the last row's p.  The n-gram drafter of
the pages proposes one token deterministically, q = the point mass on d, so:

* keep d_i iff u_i < p_i(d_i)            (u_i uniform on (0, 1));
* at the first rejection, row j: draw from p_j restricted to v != d_j,
  renormalised (norm(max(0, p - q)) for a point-mass q);
* all kept: draw from p_{n_valid};

with p_i = softmax(L_i / T) over the vocabulary, L_i the logits of window row i.
Draws use the Gumbel-max trick (Gumbel 1954; Maddison, Tarlow & Minka 2014):
argmax_v (L_i(v) / T + g_i(v)) with g i.i.d. standard Gumbel is a draw from
p_i, and the same argmax over v != d is a draw from the residual.

Random numbers come from a counter-based generator implemented here from its
published definition (the kernel implements its own copy; the two share no
code): SplitMix64 (Steele, Lea & Flood, OOPSLA 2014; finaliser constants as
published by Vigna) keyed by (seed, counter):

    key    = mix(seed + (counter + 1) * G)          (mod 2**64, G = 0x9E3779B97F4A7C15)
    w(c)   = mix(key + (c + 1) * G)                  one output per pair of elements
    h(e)   = the low 32 bits of w(e >> 1) for even e, the high 32 bits for odd e
    u(e)   = (2 * (h(e) >> 9) + 1) * 2**-24         in (0, 1), exact in fp32
    Gumbel for row i, entry v:   e = 32 * v + i,  g = -log(-log(u))
    acceptance uniform, row i:   e = 32 * V + i

-log(u) is taken as -log1p(-(1 - u)) (1 - u is exact), which keeps the large-g
tail (u near 1) accurate.  Everything here is fp64.  The arithmetic is in the
plain C++ oracle (``oracle/src/oracle.cpp``); this module only marshals arrays.
"""
from __future__ import annotations

import numpy as np

from . import _native as N

G = np.uint64(0x9E3779B97F4A7C15)
MAX_ROWS = 32


def mix(z):
    """SplitMix64 finaliser on uint64 (array or scalar), mod 2**64."""
    a = np.asarray(z, dtype=np.uint64)
    c = np.ascontiguousarray(a.reshape(-1))
    out = np.empty(c.shape, dtype=np.uint64)
    N.lib().orc_mix_array(N.ptr(c), c.size, N.ptr(out))
    return out.reshape(a.shape)


def rng_key(seed: int, counter: int) -> np.uint64:
    return np.uint64(N.lib().orc_rng_key(seed % 2**64, counter % 2**64))


def uniforms(key, idx) -> np.ndarray:
    """u(e) for the element indices ``idx`` (float64 values exact in fp32)."""
    a = np.asarray(idx, dtype=np.uint64)
    c = np.ascontiguousarray(a.reshape(-1))
    out = np.empty(c.shape, dtype=np.float64)
    N.lib().orc_uniforms(int(key), N.ptr(c), c.size, N.ptr(out))
    return out.reshape(a.shape)


def gumbel(key, S: int, V: int) -> np.ndarray:
    """Standard Gumbel noise ``[S, V]``: row i, entry v uses element 32 * v + i."""
    out = np.empty((S, V), dtype=np.float64)
    N.lib().orc_gumbel(int(key), S, V, N.ptr(out))
    return out


def accept_uniforms(key, S: int, V: int) -> np.ndarray:
    return uniforms(key, np.uint64(MAX_ROWS) * np.uint64(V) + np.arange(S, dtype=np.uint64))


def verify_sample(logits: np.ndarray, drafts, n_valid: int, temperature: float, seed: int, counter: int):
    """Speculative-sampling verify of one window.

    ``logits`` [S, V] (fp64 from ``verify.dequant_gemm64``), drafts [S-1].
    Returns a dict: ``accepted`` (kept drafts), ``token`` (the draw at the first
    rejection or the bonus draw), ``samples`` [S] (each row's full-distribution
    draw), ``p_draft`` [n_valid] (p_i(d_i)), ``u`` [S] and, for tolerance
    decisions, ``z_gap`` [S] (top-2 gap of L/T + g per row), ``z_gap_res``
    [S] (the same gap with the row's draft excluded) and ``u_margin`` (the
    smallest |u_i - p_i(d_i)| over the rows the accept scan read).
    """
    if not temperature > 0.0:
        raise ValueError("temperature must be > 0")
    L = N.as_c(logits, np.float64)
    S, V = L.shape
    if not 1 <= S <= MAX_ROWS or not 0 <= n_valid <= S - 1:
        raise ValueError("bad window")
    d = N.as_c(drafts if drafts is not None and len(drafts) else np.zeros(1, np.int32), np.int32)
    acc, tok = np.zeros(1, np.int32), np.zeros(1, np.int32)
    samples = np.empty(S, dtype=np.int32)
    p_draft = np.empty(max(n_valid, 1), dtype=np.float64)
    u = np.empty(S, dtype=np.float64)
    z_gap, z_gap_res = np.empty(S, dtype=np.float64), np.empty(S, dtype=np.float64)
    margin = np.zeros(1, dtype=np.float64)
    probs = np.empty((S, V), dtype=np.float64)
    N.check(N.lib().orc_verify_sample(N.ptr(L), S, V, N.ptr(d), n_valid, float(temperature), seed % 2**64,
                                      counter % 2**64, N.ptr(acc), N.ptr(tok), N.ptr(samples), N.ptr(p_draft),
                                      N.ptr(u), N.ptr(z_gap), N.ptr(z_gap_res), N.ptr(margin), N.ptr(probs)),
            "verify_sample")
    return {"accepted": int(acc[0]), "token": int(tok[0]), "samples": samples, "p_draft": p_draft[:n_valid],
            "u": u, "z_gap": z_gap, "z_gap_res": z_gap_res, "u_margin": float(margin[0]), "probs": probs}

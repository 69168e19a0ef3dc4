"""Verify forward over a static window of S = K+1 rows (oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product path; it shares no code with it.

Pages followed:

* "Spec-decode on GDN hybrids (Qwen3.5/3.6 family) -- static-S verify
  design", section "Verify graph = STATIC S=K+1 + chunked GDN scan": one
  forward over a fixed window of S rows returns logits for every position;
  section "Hybrid state discipline": the window is ``[a0] + drafts (+pad)``,
  a0 is committed first, the longest draft prefix is accepted and the row
  after the last accepted token is the next round's a0.
* "Stream C -- Speculative decoding: feasibility verdict + implementation
  plan", section "The delta -- new ENGINE work for greedy n-gram
  spec-decode": a batched argmax ``[K, vocab] -> [K]`` and the accept/reject
  rule (accept d_i iff d_i == a_i and every earlier draft was accepted; the
  first miss at j emits the correction a_j, all-accept emits the bonus a_K);
  section "Control-logic proof": the indexing a_i = argmax(prefix +
  draft[:i]).
* "Flagship dramatic-speedup plan -- the full stackable tuning set",
  section "Baseline byte model": the lm_head is a quantised matvec over the
  whole vocabulary (the single biggest one).

The arithmetic is in the plain C++ oracle (``oracle/src/oracle.cpp``); this
module only marshals arrays.

Readings: the dequantised GEMM accumulates in float64, term by term in
reduction order (every product x * q * s is exact in float64), and is rounded
once to float32, the dtype of the logits.  The argmax is taken on those float32 logits, the precision the
GPU decides in; ties go to the lowest index.  The top-2 gap that decides
which rows are compared exactly is taken from the float64 values.
"""
from __future__ import annotations

import numpy as np

from . import _native as N

BLOCK = 32


def dequant_gemm64(x: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Y[s, n] = sum_h x[s, h] * q[n, h] * s16[n, h // 32], in float64, h in order.

    ``x`` fp16 ``[S, H]`` (or float64 values, e.g. inside the MoE); ``codes``
    ``[N, H]`` unpacked: int8 integer codes, uint8 E2M1 codes (0..15) or float64
    values; ``scales`` fp16 ``[N, H/32]``.
    """
    kind, c = N.code_kind(codes)
    n, h = c.shape
    s = N.half_bits(scales)
    if s.shape != (n, h // BLOCK) or h % BLOCK:
        raise ValueError("shape mismatch")
    xa = np.asarray(x)
    if xa.ndim != 2 or xa.shape[1] != h:
        raise ValueError("shape mismatch")
    y = np.empty((xa.shape[0], n), dtype=np.float64)
    if xa.dtype == np.float16:
        xb = N.half_bits(xa)
        N.check(N.lib().orc_dequant_gemm64(kind, N.ptr(c), N.ptr(s), n, h, N.ptr(xb), xa.shape[0], N.ptr(y),
                                           N.threads()), "dequant_gemm64")
    else:
        xd = N.as_c(xa, np.float64)
        N.check(N.lib().orc_dequant_gemm64_x64(kind, N.ptr(c), N.ptr(s), n, h, N.ptr(xd), xa.shape[0], N.ptr(y),
                                               N.threads()), "dequant_gemm64")
    return y


def dequant_gemm(x: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """``dequant_gemm64`` rounded to float32 (the dtype of logits / Y)."""
    return dequant_gemm64(x, codes, scales).astype(np.float32)


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """Per-row argmax, lowest index among equal maxima (int32 ``[S]``)."""
    a = np.asarray(logits)
    if a.ndim != 2:
        raise ValueError("expected [S, N]")
    out = np.empty(a.shape[0], dtype=np.int32)
    if a.dtype == np.float64:
        a = N.as_c(a, np.float64)
        N.lib().orc_argmax_rows_f64(N.ptr(a), a.shape[0], a.shape[1], N.ptr(out))
    else:
        a = N.as_c(a, np.float32)
        N.lib().orc_argmax_rows_f32(N.ptr(a), a.shape[0], a.shape[1], N.ptr(out))
    return out


def top2_gap(logits64: np.ndarray) -> np.ndarray:
    """Per-row gap between the largest and the second largest value.

    The second largest is taken over the other indices, so a duplicated
    maximum gives a gap of 0.
    """
    a = N.as_c(logits64, np.float64)
    out = np.empty(a.shape[0], dtype=np.float64)
    N.lib().orc_top2_gap(N.ptr(a), a.shape[0], a.shape[1], N.ptr(out))
    return out


def greedy_accept(argmax: np.ndarray, drafts: np.ndarray, n_valid: int):
    """Greedy longest-prefix accept over one verify window.

    ``argmax[i]`` is the target's prediction after window position i (row 0
    is the row of a0); ``drafts[i]`` is the token at window position i+1.
    Draft i is accepted iff every draft before it was accepted and
    ``drafts[i] == argmax[i]``; only the first ``n_valid`` drafts are real
    (the rest are pad and never accepted).  Returns ``(accepted, next_a0)``
    with ``next_a0 = argmax[accepted]``: the correction on a miss, the bonus
    token when every real draft was accepted.
    """
    am = N.as_c(argmax, np.int32)
    s = am.shape[0]
    if not (0 <= n_valid <= s - 1):
        raise ValueError("n_valid must lie in [0, S-1]")
    d = N.as_c(drafts if drafts is not None and len(drafts) else np.zeros(1, np.int32), np.int32)
    if d.shape[0] < n_valid:
        raise ValueError("fewer drafts than n_valid")
    acc, nxt = np.zeros(1, np.int32), np.zeros(1, np.int32)
    N.check(N.lib().orc_greedy_accept(N.ptr(am), s, N.ptr(d), n_valid, N.ptr(acc), N.ptr(nxt)), "greedy_accept")
    return int(acc[0]), int(nxt[0])


def verify_head(x, codes, scales, drafts, n_valid):
    """Whole verify step: logits, argmax, accept, next a0, and the top-2 gaps.

    Returns a dict with ``logits`` (float32 ``[S, N]``), ``argmax`` (int32
    ``[S]``), ``accepted``, ``next_a0`` and ``gap`` (float64 ``[S]``).
    """
    kind, c = N.code_kind(codes)
    n, h = c.shape
    s = N.half_bits(scales)
    xb = N.half_bits(x)
    S = xb.shape[0]
    if xb.shape[1] != h or s.shape != (n, h // BLOCK):
        raise ValueError("shape mismatch")
    if not (0 <= n_valid <= S - 1):
        raise ValueError("n_valid must lie in [0, S-1]")
    d = N.as_c(drafts if drafts is not None and len(drafts) else np.zeros(1, np.int32), np.int32)
    logits = np.empty((S, n), dtype=np.float32)
    am = np.empty(S, dtype=np.int32)
    gap = np.empty(S, dtype=np.float64)
    acc, nxt = np.zeros(1, np.int32), np.zeros(1, np.int32)
    N.check(N.lib().orc_verify_head(kind, N.ptr(c), N.ptr(s), n, h, N.ptr(xb), S, N.ptr(d), n_valid,
                                    N.ptr(logits), N.ptr(am), N.ptr(gap), N.ptr(acc), N.ptr(nxt), N.threads()),
            "verify_head")
    return {"logits": logits, "argmax": am, "accepted": int(acc[0]), "next_a0": int(nxt[0]), "gap": gap}


def tree_accept(argmax: np.ndarray, tokens: np.ndarray, parent: np.ndarray):
    """Tree verify accept (the tree variant the pages defer: "Stream C -- ...",
    section "Deferred / harder", EAGLE-3 tree verify; "Spec-decode on GDN
    hybrids ...", section "S/K SWEEP").

    The window's S rows are the nodes of a draft tree: node 0 is the root (the
    row of a0); node i > 0 carries the draft ``tokens[i]`` and hangs below
    ``parent[i]`` (< i), or is absent (pad) when ``parent[i]`` is not in
    [0, i).  ``argmax[i]`` is the target's prediction after the path root ->
    i.  Node i is accepted iff its parent is accepted and
    ``tokens[i] == argmax[parent[i]]`` (the root always is).  The commit is the
    path to the deepest accepted node, the lowest index among equally deep
    ones.  Returns ``(path, next_a0)``: the accepted nodes from the root's
    child down, and ``argmax`` of the deepest one.  A chain (parent[i] = i-1
    for the n_valid real drafts) gives ``greedy_accept``.
    """
    am = N.as_c(argmax, np.int32)
    s = am.shape[0]
    tok = N.as_c(tokens, np.int32) if s > 1 else np.zeros(1, np.int32)
    par = N.as_c(parent, np.int32) if s > 1 else np.zeros(1, np.int32)
    path = np.zeros(max(s, 1), dtype=np.int32)
    depth, nxt = np.zeros(1, np.int32), np.zeros(1, np.int32)
    N.check(N.lib().orc_tree_accept(N.ptr(am), s, N.ptr(tok), N.ptr(par), N.ptr(path), N.ptr(depth), N.ptr(nxt)),
            "tree_accept")
    return [int(v) for v in path[: int(depth[0])]], int(nxt[0])

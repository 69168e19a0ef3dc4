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

Readings: the dequantised GEMM accumulates in float64 (every product
x * q * s is exact in float64) and is rounded once to float32, the dtype of
the logits.  The argmax is taken on those float32 logits, the precision the
GPU decides in; ties go to the lowest index.  The top-2 gap that decides
which rows are compared exactly is taken from the float64 values.
"""
from __future__ import annotations

import numpy as np

from .quant import BLOCK

_ROW_CHUNK = 8192  # output rows per float64 matmul (bounds memory only)


def dequant_gemm64(x: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Y[s, n] = sum_h x[s, h] * q[n, h] * s16[n, h // 32], in float64.

    ``x`` fp16 ``[S, H]``; ``codes`` int8 ``[N, H]`` (unpacked); ``scales``
    fp16 ``[N, H/32]``.  The matmul is a library float64 product; output rows
    are processed in chunks only to bound memory (no element's arithmetic
    depends on the chunking).
    """
    x64 = np.asarray(x, dtype=np.float16).astype(np.float64)
    n, h = codes.shape
    if x64.shape[1] != h or scales.shape != (n, h // BLOCK):
        raise ValueError("shape mismatch")
    s64 = np.asarray(scales, dtype=np.float16).astype(np.float64)
    y = np.empty((x64.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, _ROW_CHUNK):
        r1 = min(n, r0 + _ROW_CHUNK)
        w = codes[r0:r1].astype(np.float64) * np.repeat(s64[r0:r1], BLOCK, axis=1)
        y[:, r0:r1] = x64 @ w.T
    return y


def dequant_gemm(x: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """``dequant_gemm64`` rounded to float32 (the dtype of logits / Y)."""
    return dequant_gemm64(x, codes, scales).astype(np.float32)


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """Per-row argmax, lowest index among equal maxima (int32 ``[S]``)."""
    return np.argmax(np.asarray(logits), axis=1).astype(np.int32)


def top2_gap(logits64: np.ndarray) -> np.ndarray:
    """Per-row gap between the largest and the second largest value.

    The second largest is taken over the other indices, so a duplicated
    maximum gives a gap of 0.
    """
    l = np.asarray(logits64, dtype=np.float64)
    if l.shape[1] < 2:
        return np.full(l.shape[0], np.inf)
    part = -np.partition(-l, 1, axis=1)[:, :2]
    return part[:, 0] - part[:, 1]


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
    s = len(argmax)
    if not (0 <= n_valid <= s - 1):
        raise ValueError("n_valid must lie in [0, S-1]")
    j = 0
    while j < n_valid and int(drafts[j]) == int(argmax[j]):
        j += 1
    return j, int(argmax[j])


def verify_head(x, codes, scales, drafts, n_valid):
    """Whole verify step: logits, argmax, accept, next a0, and the top-2 gaps.

    Returns a dict with ``logits`` (float32 ``[S, N]``), ``argmax`` (int32
    ``[S]``), ``accepted``, ``next_a0`` and ``gap`` (float64 ``[S]``).
    """
    y64 = dequant_gemm64(x, codes, scales)
    logits = y64.astype(np.float32)
    am = argmax_rows(logits)
    acc, nxt = greedy_accept(am, drafts, n_valid)
    return {"logits": logits, "argmax": am, "accepted": acc, "next_a0": nxt,
            "gap": top2_gap(y64)}


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
    s = len(argmax)
    acc = [True] + [False] * (s - 1)
    depth = [0] * s
    for i in range(1, s):
        p = int(parent[i])
        if 0 <= p < i and acc[p] and int(tokens[i]) == int(argmax[p]):
            acc[i] = True
            depth[i] = depth[p] + 1
    best = 0
    for i in range(1, s):
        if acc[i] and depth[i] > depth[best]:
            best = i
    path = []
    i = best
    while i != 0:
        path.append(i)
        i = int(parent[i])
    return path[::-1], int(argmax[best])

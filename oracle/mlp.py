"""SwiGLU projections and the top-k gathered-expert MoE (oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product path; it shares no code with it.

Pages followed:

* "Flagship dramatic-speedup plan -- the full stackable tuning set",
  section "Axis 4 -- kernel micro-opts" (the fused SwiGLU MLP) and section
  "Baseline byte model" (routed experts on gather_qmm, top-8 of 256, the
  biggest byte bucket; an fp16 router that stays).
* "Riding Apple's pipelined GPU engine", section "Quantization on the GPU
  delegate" (per-block-32 linear int4 / int8 weights).

Readings where the pages are silent:

* SwiGLU: h = SiLU(g) * u with g = x G^T, u = x U^T and
  SiLU(t) = t / (1 + exp(-t)); float64 throughout.  When h is an API output
  (the dense gate/up projection) it is rounded once to fp16 (RNE); inside the
  MoE it stays float64.
* Routing: per row, the k experts with the largest router logits, ties to
  the lower expert id; weights = softmax over the k selected logits
  (identical to renormalising the full softmax over those k).
* Grouping: the (row, expert) pairs ordered by expert, and by row within an
  expert (each row picks an expert at most once, so the order is total).
* Combine: out[s] = sum over the row's k selections, in selection order, of
  w * (h_e(x[s]) D_e^T), float64, rounded once to float32.
"""
from __future__ import annotations

import numpy as np

from .quant import dequantize
from .verify import dequant_gemm64


def silu(t):
    """SiLU(t) = t / (1 + exp(-t)) in float64."""
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def swiglu64(x, gate_codes, gate_scales, up_codes, up_scales):
    """h = SiLU(x G^T) * (x U^T), float64 ``[S, N]``."""
    g = dequant_gemm64(x, gate_codes, gate_scales)
    u = dequant_gemm64(x, up_codes, up_scales)
    return silu(g) * u


def qlinear_swiglu(x, gate_codes, gate_scales, up_codes, up_scales):
    """The fused gate/up projection's API output: ``swiglu64`` rounded to fp16."""
    return swiglu64(x, gate_codes, gate_scales, up_codes, up_scales).astype(np.float16)


def route_topk(router_logits, k: int):
    """Top-k experts per row (ties to the lower id) and their softmax weights.

    Returns ``(ids int32 [S, k], weights float64 [S, k])``; ids are listed in
    selection order (largest logit first).
    """
    r = np.asarray(router_logits, dtype=np.float32)
    s_rows, e = r.shape
    if not (1 <= k <= e):
        raise ValueError("top_k must lie in [1, E]")
    ids = np.empty((s_rows, k), dtype=np.int32)
    w = np.empty((s_rows, k), dtype=np.float64)
    for s in range(s_rows):
        order = sorted(range(e), key=lambda j: (-float(r[s, j]), j))[:k]
        ids[s] = order
        l = r[s, order].astype(np.float64)
        p = np.exp(l - l.max())
        w[s] = p / p.sum()
    return ids, w


def group_by_expert(ids, n_experts: int):
    """Counting-sort the (row, slot) selections by expert.

    Returns ``(offsets int32 [E+1], rows int32 [S*k], slots int32 [S*k])``:
    expert e's selections are entries ``offsets[e] .. offsets[e+1]-1``, in
    increasing row order.
    """
    ids = np.asarray(ids)
    s_rows, k = ids.shape
    counts = np.zeros(n_experts, dtype=np.int64)
    for s in range(s_rows):
        for j in range(k):
            counts[ids[s, j]] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].astype(np.int64).copy()
    rows = np.empty(s_rows * k, dtype=np.int32)
    slots = np.empty(s_rows * k, dtype=np.int32)
    for s in range(s_rows):
        for j in range(k):
            e = ids[s, j]
            rows[fill[e]] = s
            slots[fill[e]] = j
            fill[e] += 1
    return offsets, rows, slots


def expert_swiglu64(x_rows, e, inter, hidden, gate, up, down):
    """One expert's SwiGLU MLP on rows ``x_rows`` (fp16 ``[R, H]``), float64.

    ``gate``/``up``/``down`` are ``(codes, scales)`` of the stacked tensors:
    gate/up ``[E*I, H]``, down ``[E*H, I]``; expert e owns rows
    ``e*I .. (e+1)*I-1`` of gate/up and ``e*H .. (e+1)*H-1`` of down.
    """
    gs = slice(e * inter, (e + 1) * inter)
    ds = slice(e * hidden, (e + 1) * hidden)
    g = dequant_gemm64(x_rows, gate[0][gs], gate[1][gs])
    u = dequant_gemm64(x_rows, up[0][gs], up[1][gs])
    h = silu(g) * u
    return h @ dequantize(down[0][ds], down[1][ds]).T


def moe_forward(x, router_logits, gate, up, down, n_experts, inter, hidden, top_k):
    """Gathered-expert SwiGLU MoE over the window: returns
    ``(out float32 [S, H], ids int32 [S, k], weights float64 [S, k])``."""
    x = np.asarray(x, dtype=np.float16)
    ids, w = route_topk(router_logits, top_k)
    s_rows = x.shape[0]
    out = np.zeros((s_rows, hidden), dtype=np.float64)
    for s in range(s_rows):
        for j in range(top_k):
            y = expert_swiglu64(x[s:s + 1], int(ids[s, j]), inter, hidden, gate, up, down)
            out[s] += w[s, j] * y[0]
    return out.astype(np.float32), ids, w

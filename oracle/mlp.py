"""SwiGLU projections and the top-k gathered-expert MoE (oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product path; it shares no code with it.
The arithmetic is in the plain C++ oracle (``oracle/src/oracle.cpp``); this
module only marshals arrays.

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
  (identical to renormalising the full softmax over those k), the sum taken
  over the selection in selection order.
* Grouping: the (row, expert) pairs ordered by expert, and by row within an
  expert (each row picks an expert at most once, so the order is total).
* Combine: out[s] = sum over the row's k selections, in selection order, of
  w * (h_e(x[s]) D_e^T), float64, rounded once to float32.
"""
from __future__ import annotations

import numpy as np

from . import _native as N

BLOCK = 32


def silu(t):
    """SiLU(t) = t / (1 + exp(-t)) in float64."""
    shape = np.shape(t)
    a = N.as_c(np.reshape(t, -1), np.float64)
    out = np.empty(a.shape, dtype=np.float64)
    N.lib().orc_silu(N.ptr(a), a.size, N.ptr(out))
    return out.reshape(shape) if shape else float(out[0])


def _swiglu(x, gate_codes, gate_scales, up_codes, up_scales, want16: bool):
    kg, gc = N.code_kind(gate_codes)
    ku, uc = N.code_kind(up_codes)
    if kg != ku or gc.shape != uc.shape:
        raise ValueError("gate and up must have the same shape and code type")
    n, k = gc.shape
    xb = N.half_bits(x)
    S = xb.shape[0]
    h = np.empty((S, n), dtype=np.float64)
    h16 = np.empty((S, n), dtype=np.uint16) if want16 else None
    N.check(N.lib().orc_swiglu64(kg, N.ptr(gc), N.ptr(N.half_bits(gate_scales)), N.ptr(uc),
                                 N.ptr(N.half_bits(up_scales)), n, k, N.ptr(xb), S, N.ptr(h), N.ptr(h16),
                                 N.threads()), "swiglu64")
    return h, h16


def swiglu64(x, gate_codes, gate_scales, up_codes, up_scales):
    """h = SiLU(x G^T) * (x U^T), float64 ``[S, N]``."""
    return _swiglu(x, gate_codes, gate_scales, up_codes, up_scales, False)[0]


def qlinear_swiglu(x, gate_codes, gate_scales, up_codes, up_scales):
    """The fused gate/up projection's API output: ``swiglu64`` rounded once to fp16."""
    return _swiglu(x, gate_codes, gate_scales, up_codes, up_scales, True)[1].view(np.float16)


def route_topk(router_logits, k: int):
    """Top-k experts per row (ties to the lower id) and their softmax weights.

    Returns ``(ids int32 [S, k], weights float64 [S, k])``; ids are listed in
    selection order (largest logit first).
    """
    r = N.as_c(router_logits, np.float32)
    s_rows, e = r.shape
    if not (1 <= k <= e):
        raise ValueError("top_k must lie in [1, E]")
    ids = np.empty((s_rows, k), dtype=np.int32)
    w = np.empty((s_rows, k), dtype=np.float64)
    N.check(N.lib().orc_route_topk(N.ptr(r), s_rows, e, k, N.ptr(ids), N.ptr(w)), "route_topk")
    return ids, w


def group_by_expert(ids, n_experts: int):
    """Counting-sort the (row, slot) selections by expert.

    Returns ``(offsets int32 [E+1], rows int32 [S*k], slots int32 [S*k])``:
    expert e's selections are entries ``offsets[e] .. offsets[e+1]-1``, in
    increasing row order.
    """
    a = N.as_c(ids, np.int32)
    s_rows, k = a.shape
    offsets = np.empty(n_experts + 1, dtype=np.int32)
    rows = np.empty(s_rows * k, dtype=np.int32)
    slots = np.empty(s_rows * k, dtype=np.int32)
    N.check(N.lib().orc_group_by_expert(N.ptr(a), s_rows, k, n_experts, N.ptr(offsets), N.ptr(rows),
                                        N.ptr(slots)), "group_by_expert")
    return offsets, rows, slots


def _stacked(gate, up, down):
    kinds = [N.code_kind(t[0]) for t in (gate, up, down)]
    if len({k for k, _ in kinds}) != 1:
        raise ValueError("gate, up and down must share a code type")
    return kinds[0][0], [c for _, c in kinds], [N.half_bits(t[1]) for t in (gate, up, down)]


def expert_swiglu64(x_rows, e, inter, hidden, gate, up, down):
    """One expert's SwiGLU MLP on rows ``x_rows`` (fp16 ``[R, H]``), float64.

    ``gate``/``up``/``down`` are ``(codes, scales)`` of the stacked tensors:
    gate/up ``[E*I, H]``, down ``[E*H, I]``; expert e owns rows
    ``e*I .. (e+1)*I-1`` of gate/up and ``e*H .. (e+1)*H-1`` of down.
    """
    kind, c, s = _stacked(gate, up, down)
    xb = N.half_bits(x_rows)
    R = xb.shape[0]
    y = np.empty((R, hidden), dtype=np.float64)
    N.check(N.lib().orc_expert_swiglu64(kind, N.ptr(c[0]), N.ptr(s[0]), N.ptr(c[1]), N.ptr(s[1]), N.ptr(c[2]),
                                        N.ptr(s[2]), int(e), inter, hidden, N.ptr(xb), R, N.ptr(y), N.threads()),
            "expert_swiglu64")
    return y


def moe_forward(x, router_logits, gate, up, down, n_experts, inter, hidden, top_k):
    """Gathered-expert SwiGLU MoE over the window: returns
    ``(out float32 [S, H], ids int32 [S, k], weights float64 [S, k])``."""
    kind, c, s = _stacked(gate, up, down)
    xb = N.half_bits(x)
    S = xb.shape[0]
    r = N.as_c(router_logits, np.float32)
    out = np.empty((S, hidden), dtype=np.float32)
    ids = np.empty((S, top_k), dtype=np.int32)
    w = np.empty((S, top_k), dtype=np.float64)
    N.check(N.lib().orc_moe_forward(kind, N.ptr(c[0]), N.ptr(s[0]), N.ptr(c[1]), N.ptr(s[1]), N.ptr(c[2]),
                                    N.ptr(s[2]), n_experts, inter, hidden, top_k, N.ptr(xb), N.ptr(r), S, N.ptr(out),
                                    N.ptr(ids), N.ptr(w), N.threads()), "moe_forward")
    return out, ids, w

"""The five seeded synthetic workloads and their input recipes.

Shapes follow the models the pages discuss (no weights or prompts exist here,
so every tensor is drawn from the generator in ``synth.generator``):

=====  ======================  =====================================================
name   shape                   recipe
=====  ======================  =====================================================
tiny   head 4096 x 256, int8   S = 9, 1000 windows
q4b    head 151936 x 2560 int8 S = 9, 200 windows (Qwen3-4B-shaped lm_head)
a3b    head 248320 x 2048 int4 S in {1, 2, 9, 17}, 200 windows (35B-A3B lm_head)
mlp27  5120 -> 17408 -> 5120   gate/up/down int8, S in {1, 9, 17}, 200 windows
moe    256 experts, 2048/512   top-8, int4, S = 17, 200 windows
=====  ======================  =====================================================

Distributions: weights i.i.d. N(0, 0.02) float32 (quantised afterwards by
whichever side is under test), activations i.i.d. N(0, 1) rounded to fp16,
router logits i.i.d. N(0, 1) float32.

Draft rule (verify heads): for window w pick j ~ U{0..S-1}; the first j
drafts copy a supplied argmax chain (the oracle's, in the parity tests), the
rest are uniform token ids; n_valid = S - 1.  This module only draws the
random numbers; the chain comes from the caller.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .generator import normal, randint, stream_seed

W_SIGMA = 0.02

# tensor ids inside a workload's seed key
T_HEAD, T_X, T_DRAFT_J, T_DRAFT_TOK, T_GATE, T_UP, T_DOWN, T_ROUTER = range(1, 9)


@dataclass(frozen=True)
class Workload:
    key: int            # seed namespace
    name: str
    kind: str           # "head", "mlp" or "moe"
    bits: int           # 8 or 4
    n: int = 0          # head: vocab rows
    h: int = 0          # head / mlp / moe: hidden (reduction length of the head, gate, up)
    inter: int = 0      # mlp / moe: intermediate size
    experts: int = 0    # moe
    top_k: int = 0      # moe
    s_list: tuple = ()  # window sizes this workload is run at
    windows: int = 0
    s_default: int = 0
    notes: dict = field(default_factory=dict)


TINY = Workload(0, "tiny", "head", 8, n=4096, h=256, s_list=(9,), windows=1000, s_default=9)
Q4B = Workload(1, "q4b", "head", 8, n=151936, h=2560, s_list=(9,), windows=200, s_default=9)
A3B = Workload(2, "a3b", "head", 4, n=248320, h=2048, s_list=(1, 2, 9, 17), windows=200, s_default=17)
MLP27 = Workload(3, "mlp27", "mlp", 8, h=5120, inter=17408, s_list=(1, 9, 17), windows=200, s_default=17)
MOE = Workload(4, "moe", "moe", 4, h=2048, inter=512, experts=256, top_k=8, s_list=(17,),
               windows=200, s_default=17)

ALL = (TINY, Q4B, A3B, MLP27, MOE)
BY_NAME = {w.name: w for w in ALL}


def head_weights(wl: Workload, rows: slice | None = None) -> np.ndarray:
    """fp32 head weights ``[n, h]`` (or a row slice of them)."""
    seed = stream_seed(wl.key, T_HEAD)
    if rows is None:
        return normal(seed, (wl.n, wl.h), W_SIGMA)
    full = _rows_of(seed, wl.h, rows)
    return full


def _rows_of(seed: int, width: int, rows: slice) -> np.ndarray:
    """Rows ``rows`` of a row-major ``[*, width]`` normal tensor, without
    generating the rest (element index = row * width + col)."""
    from .generator import _normal_chunk
    r0, r1 = rows.start, rows.stop
    start, count = r0 * width, (r1 - r0) * width
    # Box-Muller pairs are (2p, 2p+1); align to a pair boundary.
    p0 = start // 2
    lo = 2 * p0
    npairs = (start + count - lo + 1) // 2
    buf = np.empty(2 * npairs, dtype=np.float32)
    _normal_chunk(seed, p0, npairs, W_SIGMA, buf)
    off = start - lo
    return buf[off:off + count].reshape(r1 - r0, width)


def mlp_weights(wl: Workload, which: str) -> np.ndarray:
    """fp32 dense MLP weights: gate/up ``[inter, h]``, down ``[h, inter]``."""
    tid = {"gate": T_GATE, "up": T_UP, "down": T_DOWN}[which]
    shape = (wl.h, wl.inter) if which == "down" else (wl.inter, wl.h)
    return normal(stream_seed(wl.key, tid), shape, W_SIGMA)


def moe_weights(wl: Workload, which: str) -> np.ndarray:
    """fp32 stacked expert weights: gate/up ``[E*I, H]``, down ``[E*H, I]``."""
    tid = {"gate": T_GATE, "up": T_UP, "down": T_DOWN}[which]
    e = wl.experts
    shape = (e * wl.h, wl.inter) if which == "down" else (e * wl.inter, wl.h)
    return normal(stream_seed(wl.key, tid), shape, W_SIGMA)


def activations(wl: Workload, window: int, s: int) -> np.ndarray:
    """fp16 activations ``[s, h]`` for one window (N(0, 1) rounded to fp16)."""
    return normal(stream_seed(wl.key, T_X, window, s), (s, wl.h), 1.0, dtype=np.float64).astype(np.float16)


def router_logits(wl: Workload, window: int, s: int) -> np.ndarray:
    """fp32 router logits ``[s, E]`` for one window."""
    return normal(stream_seed(wl.key, T_ROUTER, window, s), (s, wl.experts), 1.0, dtype=np.float32)


def drafts(wl: Workload, window: int, s: int, chain, vocab: int | None = None):
    """Drafts ``int32 [s-1]`` and ``n_valid`` for one window.

    j ~ U{0..s-1}; drafts[:j] = chain[:j]; drafts[j:] uniform on the vocab.
    """
    vocab = vocab if vocab is not None else wl.n
    k = s - 1
    j = int(randint(stream_seed(wl.key, T_DRAFT_J, window, s), 1, s)[0])
    d = randint(stream_seed(wl.key, T_DRAFT_TOK, window, s), max(k, 1), vocab)[:k].astype(np.int32)
    d[:j] = np.asarray(chain[:j], dtype=np.int32)
    return d, k

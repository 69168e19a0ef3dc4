"""Greedy n-gram speculative decoding driven through the GPU verify head.

The host loop of "Stream C -- Speculative decoding: feasibility verdict +
implementation plan":

* section "The delta -- new ENGINE work for greedy n-gram spec-decode": the
  drafter is a pure host hashtable over the prompt + generated stream (the last
  m tokens map to their most recent continuation); accept/reject is greedy on
  the per-position argmax of one verify forward;
* section "Implementation status -- WORKS ON DEVICE": the fused round -- a0
  (the always-correct next token) is committed first, then [a0] + drafts is
  verified in one forward, the accepted drafts are committed and the argmax at
  the first miss (or the bonus) becomes the next a0;
* section "C-value -- speedup model": E(alpha, K) = (1 - alpha^(K+1)) / (1 - alpha)
  new tokens per round, against which the measured tokens per round are set.

"Spec-decode on GDN hybrids -- static-S verify design", section "Two
hard-won harness lessons": the drafter proposes past a0, and the window is
padded to exactly S = K + 1 (pads are never accepted).

Every step of a round's arithmetic -- the head GEMM, the per-row argmax, the
accept -- runs in libsdv (``sdv_verify_head``), and so does the drafter's table
(``sdv_ngram_*``, host C++); this module keeps the token stream and pinned
staging buffers.
"""
from __future__ import annotations

from typing import Callable, Sequence

import numpy as np
import torch

from . import sdv

PAD = 0


class NgramDrafter:
    """Prompt-lookup drafter with an incremental table, held by libsdv
    (``sdv_ngram_*``: host C++, no GPU).

    The table maps each m-gram to the position right after its latest
    occurrence that has a continuation in the stream, i.e. that ends before the
    last token.  ``propose(k)`` looks up the stream's last m tokens and returns
    up to ``k`` tokens from that position on (none when the m-gram is new).
    """

    def __init__(self, m: int):
        self.m = m
        self._h = None
        self._destroy = sdv.sdv_ngram_destroy  # held so that teardown at exit still finds it
        self._h = sdv.sdv_ngram_create(m)

    def close(self) -> None:
        """Free the native table (also done when the drafter is collected)."""
        if self._h is not None:
            h, self._h = self._h, None
            self._destroy(h)

    def __del__(self):
        self.close()

    def append(self, tokens: Sequence[int]) -> None:
        if len(tokens):
            sdv.sdv_ngram_append(self._h, tokens)

    def propose(self, k: int) -> list[int]:
        return sdv.sdv_ngram_propose(self._h, k) if k > 0 else []


def expected_tokens_per_round(alpha: float, k: int) -> float:
    """E(alpha, K): committed tokens per verify round (accepted drafts + 1)."""
    if alpha >= 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


class HeadVerifier:
    """One verify forward through ``sdv_verify_head`` from host rows.

    ``verifier(x, drafts, n_valid)`` stages the window's fp16 hidden rows
    ``x [S, k]`` and the drafts through pinned host buffers, runs the fused
    head GEMM + argmax + accept on ``stream`` and returns
    ``(argmax int32 [S], accepted, next_a0)`` once the stream has finished.

    With ``graph`` (the default) a round's GPU work -- the two host-to-device
    copies, the verify launch, the copy of the results back -- is captured once
    per window size as a CUDA graph and replayed: a round then costs the host
    one replay and one stream synchronisation instead of the per-call work of
    the copies and the library call.  The graph bakes in n_valid = S - 1: the
    drafts past the real n_valid are -1, which no argmax equals, so the accept
    stops at the same place.
    """

    def __init__(self, head: sdv.QWeight, s_max: int, device="cuda", stream: torch.cuda.Stream | None = None,
                 graph: bool = True):
        self.head, self.s_max, self.graph = head, s_max, graph
        self.stream = stream if stream is not None else torch.cuda.Stream(device)
        self.ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, head.n, head.k, s_max, device=device)
        self.x_d = torch.empty((s_max, head.k), dtype=torch.float16, device=device)
        self.dr_d = torch.zeros(max(s_max - 1, 1), dtype=torch.int32, device=device)
        self.out_d = torch.empty(s_max + 2, dtype=torch.int32, device=device)  # argmax[S], accepted, next_a0
        self.x_h = torch.empty((s_max, head.k), dtype=torch.float16).pin_memory()
        self.dr_h = torch.zeros(max(s_max - 1, 1), dtype=torch.int32).pin_memory()
        self.out_h = torch.empty(s_max + 2, dtype=torch.int32).pin_memory()
        self.graphs: dict[int, torch.cuda.CUDAGraph] = {}
        self.calls = 0

    def _round(self, S: int, n_valid: int) -> None:
        """The GPU work of one round, on the current stream."""
        self.x_d[:S].copy_(self.x_h[:S], non_blocking=True)
        if S > 1:
            self.dr_d[:S - 1].copy_(self.dr_h[:S - 1], non_blocking=True)
        am, acc, nxt = self.out_d[:S], self.out_d[self.s_max:self.s_max + 1], self.out_d[self.s_max + 1:]
        sdv.sdv_verify_head(self.head, self.x_d[:S], S, self.dr_d, n_valid, None, am, acc, nxt, self.ws)
        self.out_h.copy_(self.out_d, non_blocking=True)

    def __call__(self, x: np.ndarray, drafts: Sequence[int], n_valid: int):
        S = x.shape[0]
        if not 1 <= S <= self.s_max:
            raise ValueError(f"window of {S} rows, at most {self.s_max}")
        self.x_h[:S].numpy()[...] = np.asarray(x, dtype=np.float16)
        if S > 1:
            d = self.dr_h[:S - 1].numpy()
            d[...] = np.asarray(drafts, dtype=np.int32)[:S - 1]
            if self.graph:
                d[n_valid:] = -1
        with torch.cuda.stream(self.stream):
            if not self.graph:
                self._round(S, n_valid)
            else:
                g = self.graphs.get(S)
                if g is None:
                    self._round(S, S - 1)  # outside the capture first: plans, tensor maps, attributes
                    self.stream.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=self.stream):
                        self._round(S, S - 1)
                    self.graphs[S] = g
                g.replay()
        self.stream.synchronize()
        self.calls += 1
        o = self.out_h.numpy()
        return o[:S].copy(), int(o[self.s_max]), int(o[self.s_max + 1])

    def status(self) -> int:
        """The device status of the verify calls since the last read: SDV_OK, or
        SDV_ERR_TIMEOUT where a bounded device wait gave up (the results of that
        call are then not to be trusted).  Read and cleared once the verifier's
        stream has finished; a caller checks it after a decode, or as often as
        it wants to pay a read-back for."""
        return sdv.sdv_last_device_status(self.ws, self.stream)


def greedy_decode(verify: Callable, hidden: Callable, prompt: Sequence[int], gen: int) -> list[int]:
    """Plain greedy decoding: one S = 1 forward per token."""
    toks = [int(t) for t in prompt]
    for _ in range(gen):
        am, _, _ = verify(hidden(toks)[None, :], [], 0)
        toks.append(int(am[0]))
    return toks[len(prompt):]


def spec_decode(verify: Callable, hidden: Callable, prompt: Sequence[int], gen: int, k: int, m: int,
                stats: dict | None = None) -> list[int]:
    """Greedy n-gram speculative decoding, fused-a0 rounds of S = k + 1 rows.

    Row i of a round's window holds the hidden state after the committed prefix
    (which ends with a0) followed by drafts[:i]; ``verify`` returns the row
    argmaxes, the number of accepted drafts and the next a0.
    """
    committed = [int(t) for t in prompt]
    target = len(committed) + gen
    drafter = NgramDrafter(m)
    drafter.append(committed)
    am, _, _ = verify(hidden(committed)[None, :], [], 0)
    a0 = int(am[0])
    rounds = accepted = trials = 0
    while True:
        committed.append(a0)
        drafter.append([a0])
        if len(committed) >= target:
            break
        drafts = drafter.propose(k)
        n_valid = len(drafts)
        window = drafts + [PAD] * (k - n_valid)
        x = hidden_rows(hidden, committed, drafts, k + 1)
        _, j, a0 = verify(x, window, n_valid)
        committed.extend(drafts[:j])
        drafter.append(drafts[:j])
        rounds += 1
        accepted += j
        trials += j + (1 if j < n_valid else 0)  # draft positions compared up to the first miss
    if stats is not None:
        stats.update(rounds=rounds, accepted=accepted, trials=trials, forwards=rounds + 1,
                     tokens=target - len(prompt))
    return committed[len(prompt):target]


def hidden_rows(hidden: Callable, committed: list[int], drafts: list[int], S: int) -> np.ndarray:
    """The S rows of a round: after ``committed`` (ending with a0), after each
    further draft, then zero rows for the pads -- a pad row's argmax is never
    read (the next a0 is the argmax of the row after the last accepted draft,
    at most the last real row)."""
    first = hidden(committed)
    x = np.zeros((S, first.shape[0]), dtype=np.float16)
    x[0] = first
    prefix = list(committed)
    for i, t in enumerate(drafts):
        prefix.append(t)
        x[i + 1] = hidden(prefix)
    return x


def alpha_estimate(stats: dict) -> float:
    """Per-position acceptance: accepted drafts / draft positions compared."""
    return stats["accepted"] / stats["trials"] if stats.get("trials") else 0.0

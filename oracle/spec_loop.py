"""Toy greedy speculative-decoding loop (oracle-side test machinery).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product path; it shares no code with it.

Follows "Stream C -- Speculative decoding: feasibility verdict +
implementation plan":

* section "The delta -- new ENGINE work for greedy n-gram spec-decode": the
  n-gram drafter is a host lookup over the prompt + generated stream (the last
  m tokens map to the continuation after their most recent earlier
  occurrence), and the accept/reject rule;
* section "Control-logic proof + empirical alpha": the spec-decode output must
  be token-identical to plain greedy decoding on random cases (random vocab,
  prompt and length, hash and Markov next-token oracles, K in {1,2,3,4,8},
  n-gram order in {1,2,3}); the fused scheme commits a0 first and verifies
  [a0] + drafts in one forward;

and "Spec-decode on GDN hybrids -- static-S verify design", section "Two
hard-won harness lessons": drafters propose past a0, and the window is
padded to exactly S = K+1 when the drafter has fewer than K tokens (pads are
never accepted).

The toy "models" map a token prefix to a float32 logits vector; the greedy
token is its argmax.  Everything is a pure function of the seed and prefix.
"""
from __future__ import annotations

from functools import lru_cache

import numpy as np

from .verify import argmax_rows, greedy_accept

PAD = 0


class HashModel:
    """Logits = a seeded random vector keyed by the last ``ctx`` tokens."""

    def __init__(self, vocab: int, seed: int, ctx: int = 2):
        self.vocab, self.seed, self.ctx = vocab, seed, ctx
        self._cached = lru_cache(maxsize=None)(self._logits_tail)

    def _logits_tail(self, tail):
        rng = np.random.default_rng([self.seed, len(tail), *tail])
        return rng.standard_normal(self.vocab).astype(np.float32)

    def logits(self, prefix):
        return self._cached(tuple(prefix[-self.ctx:]))


class MarkovModel:
    """Logits = a seeded random table row selected by the last token."""

    def __init__(self, vocab: int, seed: int):
        self.vocab = vocab
        rng = np.random.default_rng([seed, 7])
        self.table = rng.standard_normal((vocab, vocab)).astype(np.float32)
        self.start = rng.standard_normal(vocab).astype(np.float32)

    def logits(self, prefix):
        return self.table[prefix[-1]] if prefix else self.start


class CyclicModel:
    """Echoes the token ``period`` positions back (an n-gram drafter's best case)."""

    def __init__(self, vocab: int, seed: int, period: int):
        self.vocab, self.period = vocab, period
        rng = np.random.default_rng([seed, 11])
        self.noise = rng.standard_normal(vocab).astype(np.float32) * np.float32(0.1)

    def logits(self, prefix):
        l = self.noise.copy()
        tok = prefix[-self.period] if len(prefix) >= self.period else (len(prefix) % self.vocab)
        l[tok] += np.float32(10.0)
        return l


def greedy_token(model, prefix) -> int:
    return int(argmax_rows(model.logits(prefix)[None, :])[0])


def plain_greedy(model, prompt, gen: int):
    """Plain greedy decoding: one forward per token."""
    toks = list(prompt)
    for _ in range(gen):
        toks.append(greedy_token(model, toks))
    return toks[len(prompt):]


def ngram_propose(ctx, k: int, m: int):
    """Prompt-lookup drafter: continuation after the latest earlier match of
    the last ``m`` tokens of ``ctx`` (at most ``k`` tokens, possibly none)."""
    if k <= 0 or len(ctx) <= m:
        return []
    key = ctx[-m:]
    for start in range(len(ctx) - m - 1, -1, -1):
        if ctx[start:start + m] == key:
            return list(ctx[start + m:start + m + k])
    return []


def spec_decode(model, prompt, gen: int, k: int, m: int, accept=greedy_accept,
                argmax=argmax_rows, stats=None):
    """Greedy n-gram speculative decoding with the fused a0 scheme.

    Each round commits the pending token a0, drafts up to K tokens past it,
    runs one verify "forward" over the S = K+1 window [a0] + drafts (+pad)
    (row i holds the logits after committed-prefix + window[:i+1]), takes the
    per-row argmax, accepts the longest matching draft prefix and carries
    ``argmax[accepted]`` as the next a0.
    """
    committed = list(prompt)
    target = len(prompt) + gen
    a0 = greedy_token(model, committed)
    rounds = accepted_total = 0
    while len(committed) < target:
        committed.append(a0)
        if len(committed) >= target:
            break
        drafts = ngram_propose(committed, k, m)
        n_valid = len(drafts)
        window = [a0] + drafts + [PAD] * (k - n_valid)
        base = committed[:-1]
        rows = np.stack([model.logits(base + window[:i + 1]) for i in range(k + 1)])
        am = argmax(rows)
        j, a0 = accept(am, np.asarray(window[1:], dtype=np.int32), n_valid)
        committed.extend(drafts[:j])
        rounds += 1
        accepted_total += j
    if stats is not None:
        stats["rounds"] = rounds
        stats["accepted"] = accepted_total
    return committed[len(prompt):target]

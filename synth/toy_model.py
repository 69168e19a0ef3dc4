"""Toy model body for the end-to-end speculative-decoding loop.

A deterministic stand-in for everything in front of the head: the hidden row
that predicts the token after a prefix is a pure function of the seed and the
last ``period`` tokens of the prefix.  A seeded coin per context picks one of
two kinds of row:

* echo: the head's own fp32 weight row of the token ``period`` positions back,
  divided by the weights' standard deviation -- its logit (about h * sigma)
  stands far above every other (about N(0, sqrt(h) * sigma)), so greedy
  decoding repeats the stream with that period, the case an n-gram drafter
  predicts;
* novel: N(0, 1) -- greedy decoding picks an unrelated token.

Random numbers and the generator's own head rows only: no quantisation,
matmul or argmax lives here (the verify kernel takes the argmax).  Shared by
the GPU loop and the oracle's loop in the tests, like every generator.
"""
from __future__ import annotations

from typing import Callable

import numpy as np

from .generator import normal, stream_seed, uniform01

T_COIN, T_NOVEL = 1, 2


class ToyHidden:
    """``hidden(prefix) -> fp16 [h]`` for a prefix of token ids.

    ``head_row(t)`` returns the fp32 weight row of vocabulary entry ``t`` (the
    same numbers the head was quantised from) and ``sigma`` their standard
    deviation.  Rows are cached per context.
    """

    def __init__(self, h: int, seed: int, head_row: Callable[[int], np.ndarray], sigma: float,
                 p_echo: float = 0.7, period: int = 5):
        self.h, self.seed, self.head_row, self.sigma = h, seed, head_row, sigma
        self.p_echo, self.period = p_echo, period
        self._cache: dict[tuple, np.ndarray] = {}

    def __call__(self, prefix) -> np.ndarray:
        key = tuple(int(t) for t in prefix[-self.period:])
        row = self._cache.get(key)
        if row is not None:
            return row
        sk = stream_seed(self.seed, len(key), *key)
        coin = float(uniform01(stream_seed(sk, T_COIN), 0, 1)[0])
        if coin < self.p_echo and len(key) == self.period:
            v = np.asarray(self.head_row(key[0]), dtype=np.float64) / self.sigma
            row = v.astype(np.float16)
        else:
            row = normal(stream_seed(sk, T_NOVEL), (self.h,), 1.0, dtype=np.float64).astype(np.float16)
        self._cache[key] = row
        return row

    def rows(self, prefixes) -> np.ndarray:
        """fp16 ``[len(prefixes), h]``."""
        return np.stack([self(p) for p in prefixes])

"""Host logic of the end-to-end speculative-decoding loop (CPU only).

* the incremental n-gram drafter against the oracle's prompt-lookup search
  ("Stream C -- Speculative decoding: feasibility verdict + implementation
  plan", section "The delta": last m tokens -> most recent continuation);
* E(alpha, K) against the speedup table the same page prints (section
  "C-value -- speedup model");
* the product loop against the oracle's loop and plain greedy decoding, with a
  CPU stand-in for the verify call built from the oracle (lossless: token for
  token), on the toy model body of ``synth.toy_model``.
"""
import os

import numpy as np
import pytest

from oracle import quant, spec_loop, verify
from speculative_decode_verify_sdv_gb300 import specdec
from synth import generator as G
from synth.toy_model import ToyHidden

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ngram_speedup_table.txt")

# the drafter's table lives in libsdv (host C++): build and load it first
pytestmark = pytest.mark.usefixtures("libsdv")


@pytest.mark.parametrize("m", [1, 2, 3])
def test_drafter_matches_oracle_search(m):
    rng = np.random.default_rng(m)
    for case in range(40):
        vocab = int(rng.integers(2, 6))
        stream = [int(t) for t in rng.integers(0, vocab, int(rng.integers(1, 60)))]
        d = specdec.NgramDrafter(m)
        for i, t in enumerate(stream):
            d.append([t])
            for k in (1, 3, 8):
                assert d.propose(k) == spec_loop.ngram_propose(stream[:i + 1], k, m), (case, i, k)


def test_drafter_examples():
    d = specdec.NgramDrafter(2)
    d.append([1, 2, 3, 1, 2])
    assert d.propose(4) == [3, 1, 2]          # continuation of the earlier (1, 2), up to the end
    d.append([9])
    assert d.propose(4) == []                 # (2, 9) never seen before
    d.append([1, 2])
    assert d.propose(2) == [9, 1]             # the LATEST earlier (1, 2) wins
    assert specdec.NgramDrafter(3).propose(5) == []


def test_drafter_full_int32_range_and_long_stream():
    # token ids are opaque 32-bit keys; a long stream with a large n-gram order
    rng = np.random.default_rng(7)
    base = [int(t) for t in rng.integers(-2**31, 2**31 - 1, 64)]
    stream = base * 40 + [int(t) for t in rng.integers(-2**31, 2**31 - 1, 50)] + base[:20]
    for m in (4, 64):
        d = specdec.NgramDrafter(m)
        d.append(stream)
        for k in (1, 17, 100):
            assert d.propose(k) == spec_loop.ngram_propose(stream, k, m)


def test_drafter_close_is_idempotent():
    d = specdec.NgramDrafter(2)
    d.append([1, 2, 1])
    d.close()
    d.close()
    del d


def test_drafters_are_independent():
    a, b = specdec.NgramDrafter(1), specdec.NgramDrafter(1)
    a.append([5, 6, 5])
    b.append([5, 7, 5])
    assert a.propose(3) == [6, 5] and b.propose(3) == [7, 5]


def test_drafter_rejects_bad_arguments(libsdv):
    from speculative_decode_verify_sdv_gb300 import sdv
    for m in (0, -1, 65):
        with pytest.raises(sdv.SdvError):
            specdec.NgramDrafter(m)
    import ctypes
    h = sdv.sdv_ngram_create(2)
    try:
        cnt = ctypes.c_int32(0)
        assert libsdv.sdv_ngram_propose(ctypes.c_void_p(h), 3, None, ctypes.byref(cnt)) == sdv.SDV_ERR_INVALID_ARG
        assert libsdv.sdv_ngram_propose(ctypes.c_void_p(h), -1, None, ctypes.byref(cnt)) == sdv.SDV_ERR_INVALID_ARG
        assert libsdv.sdv_ngram_append(ctypes.c_void_p(h), None, 2) == sdv.SDV_ERR_INVALID_ARG
        assert libsdv.sdv_ngram_append(ctypes.c_void_p(h), None, 0) == sdv.SDV_OK
        assert libsdv.sdv_ngram_append(None, None, 0) == sdv.SDV_ERR_INVALID_ARG
        assert libsdv.sdv_ngram_create(2, None) == sdv.SDV_ERR_INVALID_ARG
    finally:
        sdv.sdv_ngram_destroy(h)
    assert libsdv.sdv_ngram_destroy(None) == sdv.SDV_OK


def test_expected_tokens_match_page_table():
    rows = [list(map(float, line.split())) for line in open(GOLDEN) if line.strip() and not line.startswith("#")]
    assert len(rows) == 5
    for alpha, s10, s13 in rows:
        best = max(specdec.expected_tokens_per_round(alpha, k) for k in range(1, 9))
        assert round(best / 1.0, 2) == pytest.approx(s10, abs=1e-9)
        assert round(best / 1.3, 2) == pytest.approx(s13, abs=1e-9)
    assert specdec.expected_tokens_per_round(1.0, 8) == 9.0
    assert specdec.expected_tokens_per_round(0.0, 8) == 1.0


class _OracleHead:
    """CPU stand-in for the verify call: oracle dequant GEMM, argmax, accept."""

    def __init__(self, n, k, seed, bits=8):
        self.w = G.normal(G.stream_seed(950, n, k, seed), (n, k), 0.02)
        self.codes, self.scales = quant.quantize_block32(self.w, bits)
        self.calls = 0

    def row(self, t):
        return self.w[t]

    def logits(self, x):
        return verify.dequant_gemm64(np.asarray(x, dtype=np.float16), self.codes, self.scales)

    def __call__(self, x, drafts, n_valid):
        self.calls += 1
        am = verify.argmax_rows(self.logits(x).astype(np.float32))
        j, nxt = verify.greedy_accept(am, np.asarray(drafts, dtype=np.int64), n_valid)
        return am, int(j), int(nxt)


class _OracleModel:
    """The oracle loop's model interface over the same head and hidden rows."""

    def __init__(self, head, hidden):
        self.head, self.hidden = head, hidden

    def logits(self, prefix):
        return self.head.logits(self.hidden(prefix)[None, :])[0].astype(np.float32)


@pytest.mark.parametrize("k,m,p_echo", [(1, 1, 0.7), (4, 2, 0.7), (8, 3, 0.7), (8, 2, 0.0), (8, 1, 1.0)])
def test_loop_is_lossless_on_cpu(k, m, p_echo):
    n, h = 512, 64
    head = _OracleHead(n, h, seed=k * 10 + m)
    hidden = ToyHidden(h, 77 + k, head.row, 0.02, p_echo=p_echo, period=4)
    prompt = [int(t) for t in G.randint(G.stream_seed(951, k, m), 12, n)]
    gen = 120
    stats = {}
    spec = specdec.spec_decode(head, hidden, prompt, gen, k, m, stats)
    greedy = specdec.greedy_decode(head, hidden, prompt, gen)
    assert spec == greedy
    model = _OracleModel(head, hidden)
    assert spec == spec_loop.plain_greedy(model, prompt, gen)
    ostats = {}
    assert spec == spec_loop.spec_decode(model, prompt, gen, k, m, stats=ostats)
    assert (stats["rounds"], stats["accepted"]) == (ostats["rounds"], ostats["accepted"])
    assert stats["forwards"] == stats["rounds"] + 1
    if p_echo == 1.0:   # a periodic stream: the drafter hits after the first period
        assert stats["accepted"] > gen // 2
    a = specdec.alpha_estimate(stats)
    assert 0.0 <= a <= 1.0

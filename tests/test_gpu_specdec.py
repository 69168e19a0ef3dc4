"""End-to-end greedy n-gram speculative decoding through sdv_verify_head.

Lossless: the loop's tokens equal plain greedy decoding (one S = 1 verify per
token) token for token, and equal the oracle's greedy decoding up to the first
step whose oracle top-2 logit gap is under 1e-2 (where fp32 accumulation may
legitimately flip the argmax).  Also: a window row's logits do not depend on
the window it sits in (the GPU side of losslessness).
"""
import numpy as np
import pytest
import torch

from oracle import verify
from speculative_decode_verify_sdv_gb300 import specdec
from synth import generator as G
from synth.toy_model import ToyHidden
from tests.helpers import device_weight, oracle_weight, run_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _head(n, k, bits, seed):
    w = G.normal(G.stream_seed(960, n, k, bits, seed), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, bits)
    return w, codes, scales, device_weight(stored, scales, bits, n, k)


def _oracle_greedy(codes, scales, hidden, prompt, gen):
    """Oracle greedy tokens and the number of leading steps whose top-2 gap is >= 1e-2."""
    toks, safe = list(prompt), None
    for step in range(gen):
        y = verify.dequant_gemm64(hidden(toks)[None, :], codes, scales)[0]
        top2 = np.sort(y)[-2:]
        if safe is None and top2[1] - top2[0] < 1e-2:
            safe = step
        toks.append(int(verify.argmax_rows(y[None, :].astype(np.float32))[0]))
    return toks[len(prompt):], gen if safe is None else safe


@pytest.mark.parametrize("bits,n,k", [(8, 4096, 256), (4, 8192, 512)])
@pytest.mark.parametrize("K,m", [(1, 1), (4, 2), (8, 3), (15, 2), (16, 3)])
def test_spec_loop_lossless(sdv, bits, n, k, K, m):
    w, codes, scales, qw = _head(n, k, bits, K * 7 + m)
    hidden = ToyHidden(k, G.stream_seed(961, K, m), lambda t: w[t], 0.02, p_echo=0.7, period=4)
    prompt = [int(t) for t in G.randint(G.stream_seed(962, K, m), 16, n)]
    gen = 160
    stats = {}
    ver_s, ver_1 = specdec.HeadVerifier(qw, K + 1), specdec.HeadVerifier(qw, 1)
    spec = specdec.spec_decode(ver_s, hidden, prompt, gen, K, m, stats)
    greedy = specdec.greedy_decode(ver_1, hidden, prompt, gen)
    assert ver_s.status() == sdv.SDV_OK and ver_1.status() == sdv.SDV_OK
    assert spec == greedy
    ref, safe = _oracle_greedy(codes, scales, hidden, prompt, gen)
    assert spec[:safe] == ref[:safe]
    assert stats["accepted"] > 0 and stats["rounds"] + stats["accepted"] >= gen - 1


@pytest.mark.parametrize("bits,k", [(8, 2560), (4, 2048)])
def test_row_logits_independent_of_window(sdv, bits, k):
    """Row i's logits are the same bits whether it is verified alone, in a
    window of 9 or of 16 (one MMA width); windows of 17..32 use the wider MMA
    and agree within the logits tolerance."""
    n = 3000
    _, codes, scales, qw = _head(n, k, bits, 5)
    x = G.normal(G.stream_seed(963, k), (32, k), 1.0, dtype=np.float64).astype(np.float16)
    alone = np.stack([run_head(qw, x[i:i + 1], np.zeros(0, np.int32), 0)[0][0] for i in range(17)])
    for S in (9, 16):
        got = run_head(qw, x[:S], np.zeros(S - 1, np.int32), 0)[0]
        assert np.array_equal(got.view(np.uint32), alone[:S].view(np.uint32)), S
    got = run_head(qw, x[:17], np.zeros(16, np.int32), 0)[0]
    ref = verify.dequant_gemm64(x[:17], codes, scales)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert float(np.max(np.abs(got - alone))) <= 2e-3 * np.sqrt(k / 256.0) * rms


@pytest.mark.parametrize("bits,k", [(8, 2560), (4, 2048)])
def test_graph_rounds_match_direct_calls(sdv, bits, k):
    """The verifier's replayed CUDA graph (n_valid baked in as S - 1, drafts past
    the real n_valid set to -1) returns what a direct call with the real n_valid
    returns, over windows whose drafts partly match the argmax chain."""
    n, S = 3000, 9
    _, codes, scales, qw = _head(n, k, bits, 11)
    direct = specdec.HeadVerifier(qw, S, graph=False)
    graphed = specdec.HeadVerifier(qw, S, graph=True)
    rng = np.random.default_rng(12)
    for case in range(24):
        x = G.normal(G.stream_seed(964, case, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
        chain = direct(x, [0] * (S - 1), 0)[0]
        drafts = list(chain[:S - 1])
        cut = int(rng.integers(0, S))
        if cut < S - 1:
            drafts[cut] = (drafts[cut] + 1) % n  # a miss at `cut`
        n_valid = int(rng.integers(0, S))
        a = direct(x, drafts, n_valid)
        b = graphed(x, drafts, n_valid)
        assert np.array_equal(a[0], b[0]) and a[1:] == b[1:], (case, n_valid, a[1:], b[1:])
    assert direct.status() == sdv.SDV_OK and graphed.status() == sdv.SDV_OK

"""The stored per-window oracle results (tests/golden/*_windows_*.jsonl) are the
oracle's: a few windows of every file are recomputed here with the oracle on
the same seeded inputs and must agree exactly (ids, accept, the drafts the
seeded draft rule builds from the argmax chain) or to the stored precision
(gaps, RMS).  CPU only; about half a minute (two full-size weight tensors are
generated and quantised)."""
import numpy as np
import pytest

from oracle import quant, verify
from synth import workloads as W
from tests.helpers import load_windows

WINDOWS = (0, 137)

_Q = {}


def _quantized(wl, which=None):
    key = (wl.name, which)
    if key not in _Q:
        _Q.clear()
        w = W.head_weights(wl) if which is None else W.mlp_weights(wl, which)
        _Q[key] = quant.quantize_block32(w, wl.bits)
    return _Q[key]


@pytest.mark.parametrize("name,S", [("q4b", 9), ("a3b", 1), ("a3b", 2), ("a3b", 9), ("a3b", 17)])
def test_head_windows_are_the_oracles(name, S):
    wl = W.BY_NAME[name]
    head, recs = load_windows("head_windows", name, S)
    assert len(recs) == wl.windows and "oracle_sha256" in head
    codes, scales = _quantized(wl)
    for win in WINDOWS:
        rec = recs[win]
        assert rec["window"] == win
        x = W.activations(wl, win, S)
        ref = verify.verify_head(x, codes, scales, np.zeros(max(S - 1, 0), np.int32), 0)
        np.testing.assert_array_equal(ref["argmax"], rec["argmax"])
        np.testing.assert_allclose(ref["gap"], rec["gap"], rtol=1e-8, atol=0)
        drafts, n_valid = W.drafts(wl, win, S, ref["argmax"])
        assert drafts.tolist() == rec["drafts"] and n_valid == rec["n_valid"]
        assert verify.greedy_accept(ref["argmax"], drafts, n_valid) == (rec["accepted"], rec["next_a0"])


def test_head_windows_exercise_the_accept():
    """Across the stored windows the accept sees every outcome: misses at 0,
    partial prefixes and full acceptance."""
    for name, S in (("q4b", 9), ("a3b", 9), ("a3b", 17)):
        _, recs = load_windows("head_windows", name, S)
        acc = np.array([r["accepted"] for r in recs])
        assert (acc == 0).any() and (acc == S - 1).any() and ((acc > 0) & (acc < S - 1)).any()


@pytest.mark.parametrize("S", [1, 9, 17])
def test_mlp_windows_are_the_oracles(S):
    wl = W.MLP27
    _, recs = load_windows("mlp_windows", "mlp27", S)
    assert len(recs) == wl.windows
    cg, sg = _quantized(wl, "gate")
    g = verify.dequant_gemm64(W.activations(wl, WINDOWS[-1], S), cg, sg)
    np.testing.assert_allclose(np.sqrt(np.mean(g * g)), recs[WINDOWS[-1]]["rms_g"], rtol=1e-12)
    cu, su = _quantized(wl, "up")
    u = verify.dequant_gemm64(W.activations(wl, 0, S), cu, su)
    np.testing.assert_allclose(np.sqrt(np.mean(u * u)), recs[0]["rms_u"], rtol=1e-12)

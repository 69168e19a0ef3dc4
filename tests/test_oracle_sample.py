"""Pins for the oracle's sampling verify (CPU only).

* the counter generator against SplitMix64's published output stream (seed 0:
  e220a8397b1dcdaf, 6e789e6aa1b965f4, 06c45d188009454f, ...);
* Gumbel-max draws follow softmax(L / T) (chi-square over many counters);
* the first emitted token after a0 -- the kept draft or the residual draw --
  follows p_0 exactly, whatever the draft (the losslessness of speculative
  sampling, Leviathan et al. 2023, Theorem 1), checked by chi-square;
* as T -> 0 with clear logit gaps the sampling verify reduces to the greedy
  accept (the pages' greedy rule, "Stream C", section "The delta").
"""
import numpy as np
import pytest
from scipy import stats

from oracle import sample, verify


def test_splitmix64_published_stream():
    # state x_k = k * G, output mix(x_k): Vigna's splitmix64.c seeded with 0
    with np.errstate(over="ignore"):
        got = [int(sample.mix(np.uint64(k) * sample.G)) for k in (1, 2, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniforms_in_open_interval_and_fp32_exact():
    key = sample.rng_key(123, 4)
    u = sample.uniforms(key, np.arange(100000, dtype=np.uint64))
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert abs(u.mean() - 0.5) < 0.01


def _chi2_ok(counts, probs, alpha=1e-4):
    exp = probs * counts.sum()
    keep = exp > 5
    obs, e = counts[keep], exp[keep]
    e = e * obs.sum() / e.sum()
    return stats.chisquare(obs, e).pvalue > alpha


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_gumbel_max_follows_softmax(T):
    V = 7
    L = np.array([[0.3, -1.0, 2.0, 0.0, 1.2, -0.4, 0.9]])
    p = np.exp(L[0] / T - (L[0] / T).max())
    p /= p.sum()
    counts = np.zeros(V)
    for c in range(6000):
        r = sample.verify_sample(L, [], 0, T, seed=7, counter=c)
        counts[r["samples"][0]] += 1
    assert _chi2_ok(counts, p)


@pytest.mark.parametrize("draft", [2, 5, 1])
def test_first_token_follows_target(draft):
    """Emitted token after a0 (draft kept, else residual draw) ~ p_0."""
    V = 6
    rng = np.random.default_rng(draft)
    L = rng.normal(0, 1.2, (3, V))
    T = 0.8
    p0 = np.exp(L[0] / T - (L[0] / T).max())
    p0 /= p0.sum()
    counts = np.zeros(V)
    for c in range(8000):
        r = sample.verify_sample(L, [draft, 0], 2, T, seed=11, counter=c)
        first = draft if r["accepted"] >= 1 else r["token"]
        counts[first] += 1
    assert _chi2_ok(counts, p0)
    assert abs(counts[draft] / counts.sum() - p0[draft]) < 4 * np.sqrt(p0[draft] * (1 - p0[draft]) / 8000)


def test_low_temperature_reduces_to_greedy():
    rng = np.random.default_rng(3)
    checked = 0
    for case in range(300):
        S, V = int(rng.integers(1, 9)), int(rng.integers(2, 40))
        L = rng.normal(0, 1, (S, V))
        srt = np.sort(L, axis=1)
        if np.any(srt[:, -1] - srt[:, -2] < 0.05):
            continue
        am = L.argmax(axis=1)
        n_valid = int(rng.integers(0, S))
        d = am[:S - 1].copy()
        if n_valid > 0:
            miss = int(rng.integers(0, n_valid + 1))
            if miss < n_valid:
                d[miss] = (d[miss] + 1) % V
        r = sample.verify_sample(L, d, n_valid, 1e-4, seed=case, counter=0)
        j, nxt = verify.greedy_accept(am, d.astype(np.int64), n_valid)
        assert (r["accepted"], r["token"]) == (j, nxt)
        assert np.array_equal(r["samples"], am)
        checked += 1
    assert checked > 100


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        sample.verify_sample(np.zeros((2, 4)), [0], 1, 0.0, 0, 0)
    with pytest.raises(ValueError):
        sample.verify_sample(np.zeros((2, 4)), [0], 2, 1.0, 0, 0)

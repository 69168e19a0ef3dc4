"""Pins for the oracle's greedy accept rule (CPU only).

* exhaustive brute force on tiny alphabets against an independent statement
  of the rule (the first mismatching draft bounds the accepted prefix);
* the fixed points the pages report: a perfect drafter accepts every draft
  and the bonus token is the last row's argmax; a drafter that re-proposes a0
  (off by one) accepts nothing; pad drafts are never accepted;
* 3000 random toy speculative-decoding runs whose output must equal plain
  greedy decoding token for token ("Stream C -- Speculative decoding:
  feasibility verdict + implementation plan", section "Control-logic proof").
"""
import itertools

import numpy as np
import pytest

from oracle import spec_loop, verify


def _independent_accept(am, drafts, n_valid):
    mism = [i for i in range(n_valid) if drafts[i] != am[i]]
    j = min(mism) if mism else n_valid
    return j, am[j]


@pytest.mark.parametrize("s", [1, 2, 3, 4, 5])
def test_accept_exhaustive_tiny(s):
    vocab = 3 if s <= 4 else 2
    count = 0
    for am in itertools.product(range(vocab), repeat=s):
        for dr in itertools.product(range(vocab), repeat=s - 1):
            for n_valid in range(s):
                got = verify.greedy_accept(np.array(am), np.array(dr, dtype=np.int64), n_valid)
                assert got == _independent_accept(am, dr, n_valid)
                count += 1
    assert count > 0


def test_all_drafts_match_gives_bonus():
    am = np.array([5, 6, 7, 8, 9, 10, 11, 12, 13])
    assert verify.greedy_accept(am, am[:8], 8) == (8, 13)


def test_first_mismatch_at_zero():
    am = np.array([5, 6, 7])
    assert verify.greedy_accept(am, np.array([4, 6]), 2) == (0, 5)


def test_single_row_window_is_a_decode_step():
    assert verify.greedy_accept(np.array([42]), np.array([], dtype=np.int32), 0) == (0, 42)


def test_pads_are_never_accepted():
    am = np.array([1, 2, 3, 4, 5])
    # pads happen to equal the argmax, but only the first n_valid drafts are real
    assert verify.greedy_accept(am, np.array([1, 2, 3, 4]), 2) == (2, 3)
    assert verify.greedy_accept(am, np.array([1, 2, 3, 4]), 0) == (0, 1)


def test_off_by_one_drafter_accepts_nothing():
    # a drafter that proposes a0 itself (continuation of C, not C + [a0]) shifts every draft
    am = np.array([10, 11, 12, 13, 14])
    shifted = np.array([9, 10, 11, 12])       # drafts[i] == am[i-1]
    assert verify.greedy_accept(am, shifted, 4) == (0, 10)


def test_rejects_bad_n_valid():
    with pytest.raises(ValueError):
        verify.greedy_accept(np.array([1, 2]), np.array([1]), 2)


def test_spec_loop_matches_plain_greedy_3000_cases():
    rng = np.random.default_rng(2026)
    stats_acc = []
    for case in range(3000):
        vocab = int(rng.integers(2, 40))
        kind = case % 3
        if kind == 0:
            model = spec_loop.HashModel(vocab, case, ctx=int(rng.integers(1, 4)))
        elif kind == 1:
            model = spec_loop.MarkovModel(vocab, case)
        else:
            model = spec_loop.CyclicModel(vocab, case, period=int(rng.integers(1, 6)))
        prompt = [int(t) for t in rng.integers(0, vocab, int(rng.integers(1, 20)))]
        gen = int(rng.integers(1, 40))
        k = int(rng.choice([1, 2, 3, 4, 8]))
        m = int(rng.integers(1, 4))
        ref = spec_loop.plain_greedy(model, prompt, gen)
        st = {}
        out = spec_loop.spec_decode(model, prompt, gen, k, m, stats=st)
        assert out == ref, f"case {case}: vocab={vocab} k={k} m={m}"
        stats_acc.append(st.get("accepted", 0))
    # the cyclic model must drive real acceptance, or the loop above tests little
    assert sum(stats_acc) > 3000


def test_spec_loop_perfect_drafter_fills_the_window():
    # echo model with a period longer than K: the drafter always has K tokens and
    # every round but the last accepts all of them
    model = spec_loop.CyclicModel(17, 1, period=10)
    prompt = list(range(10)) * 2
    st = {}
    out = spec_loop.spec_decode(model, prompt, 40, 8, 2, stats=st)
    assert out == spec_loop.plain_greedy(model, prompt, 40)
    assert st["accepted"] >= 8 * (st["rounds"] - 1)

"""Pins for the oracle's tree accept (CPU only).

* a chain tree equals the greedy accept on every case of a brute force;
* on random trees, each node's acceptance equals an independent statement:
  every edge (p -> c) on the root -> node path has tokens[c] == argmax[p];
  the committed path is the deepest such node (lowest index among equals);
* hand-made trees with a branch that wins deeper than a shallower sibling.
"""
import itertools

import numpy as np
import pytest

from oracle import verify


def _independent(argmax, tokens, parent):
    s = len(argmax)
    ok, depth = [True] + [False] * (s - 1), [0] * s
    for i in range(1, s):
        path, j, good = [], i, True
        while j != 0:
            p = int(parent[j])
            if not (0 <= p < j):
                good = False
                break
            path.append((p, j))
            j = p
        if good and all(int(tokens[c]) == int(argmax[p]) for p, c in path):
            ok[i], depth[i] = True, len(path)
    cand = [i for i in range(s) if ok[i]]
    best = min(cand, key=lambda i: (-depth[i], i))
    return best, depth[best]


@pytest.mark.parametrize("s", [1, 2, 3, 4, 5])
def test_chain_equals_greedy(s):
    vocab = 3
    for am in itertools.product(range(vocab), repeat=s):
        for dr in itertools.product(range(vocab), repeat=s - 1):
            for n_valid in range(s):
                parent = [-1] + [i - 1 if i <= n_valid else -1 for i in range(1, s)]
                tokens = [0] + list(dr)
                path, nxt = verify.tree_accept(np.array(am), np.array(tokens), np.array(parent))
                assert (len(path), nxt) == verify.greedy_accept(np.array(am), np.array(dr), n_valid)
                assert path == list(range(1, len(path) + 1))


def test_random_trees_match_independent_statement():
    rng = np.random.default_rng(0)
    for case in range(3000):
        s = int(rng.integers(1, 33))
        vocab = int(rng.integers(2, 5))
        am = rng.integers(0, vocab, s)
        tokens = rng.integers(0, vocab, s)
        parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, s)])
        path, nxt = verify.tree_accept(am, tokens, parent)
        best, depth = _independent(am, tokens, parent)
        assert len(path) == depth and nxt == int(am[best])
        assert (path[-1] if path else 0) == best
        for a, b in zip([0] + path[:-1], path):   # the path is a chain of parent links
            assert int(parent[b]) == a


def test_deeper_branch_wins():
    #        0
    #      /   \
    #     1     2        argmax[0] = 7: both children (tokens 7) accepted
    #     |     |
    #     3     4        argmax[1] = 5, argmax[2] = 6; tokens[3] = 9 (miss), tokens[4] = 6 (hit)
    am = np.array([7, 5, 6, 1, 2])
    tokens = np.array([0, 7, 7, 9, 6])
    parent = np.array([-1, 0, 0, 1, 2])
    path, nxt = verify.tree_accept(am, tokens, parent)
    assert path == [2, 4] and nxt == 2
    tokens[3] = 5                                       # now both depth-2 nodes hit: lowest index
    path, nxt = verify.tree_accept(am, tokens, parent)
    assert path == [1, 3] and nxt == 1

"""sdv_tree_accept on the GPU vs the oracle's tree accept: bit-exact on random
trees (absent nodes, duplicate sibling tokens, S = 1 .. 32) and on chains,
where it must equal the greedy accept; then on the argmax of a real verify
window whose rows are the nodes of a draft tree."""
import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from tests.helpers import device_weight, oracle_weight, run_head, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _gpu_tree(sdv, am, tokens, parent):
    S = len(am)
    i32 = torch.int32
    path = torch.full((max(S - 1, 1),), -7, dtype=i32, device="cuda")
    acc = torch.full((1,), -1, dtype=i32, device="cuda")
    nxt = torch.full((1,), -1, dtype=i32, device="cuda")
    sdv.sdv_tree_accept(to_dev(np.asarray(am, np.int32)), S, to_dev(np.asarray(tokens, np.int32)),
                        to_dev(np.asarray(parent, np.int32)), path, acc, nxt)
    a = int(acc.item())
    return path.cpu().numpy()[:a].tolist(), a, int(nxt.item())


def test_random_trees(sdv):
    rng = np.random.default_rng(1)
    for case in range(400):
        S = int(rng.integers(1, 33))
        vocab = int(rng.integers(2, 5))
        am = rng.integers(0, vocab, S)
        tokens = rng.integers(0, vocab, S)
        parent = np.array([-1] + [int(rng.integers(-2, i)) for i in range(1, S)])
        path, acc, nxt = _gpu_tree(sdv, am, tokens, parent)
        ref_path, ref_nxt = verify.tree_accept(am, tokens, parent)
        assert (path, acc, nxt) == (ref_path, len(ref_path), ref_nxt), case


def test_chains_equal_greedy(sdv):
    rng = np.random.default_rng(2)
    for case in range(100):
        S = int(rng.integers(1, 33))
        am = rng.integers(0, 3, S)
        drafts = rng.integers(0, 3, max(S - 1, 0))
        n_valid = int(rng.integers(0, S))
        parent = [-1] + [i - 1 if i <= n_valid else -1 for i in range(1, S)]
        path, acc, nxt = _gpu_tree(sdv, am, [0] + list(drafts), parent)
        assert (acc, nxt) == verify.greedy_accept(am, drafts, n_valid)


def test_tree_window_through_the_head(sdv):
    """Rows of a verify window as tree nodes: the head's argmax feeds the tree accept."""
    n, k, S = 4096, 256, 12
    w = G.normal(G.stream_seed(980, n, k), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, 8)
    qw = device_weight(stored, scales, 8, n, k)
    x = G.normal(G.stream_seed(981, S, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
    _, am, _, _ = run_head(qw, x, np.zeros(S - 1, np.int32), 0)
    eligible = ref["gap"] > 1e-2
    am_ref = ref["argmax"]
    # a tree whose first branch follows the head's predictions for three levels
    parent = np.array([-1, 0, 0, 1, 1, 3, 2, 5, 5, 6, 7, -1])
    tokens = np.zeros(S, np.int64)
    for i in range(1, S):
        if parent[i] >= 0:
            tokens[i] = am_ref[parent[i]] if i in (1, 3, 5, 7) else (am_ref[parent[i]] + 1) % n
    path, acc, nxt = _gpu_tree(sdv, am, tokens, parent)
    ref_path, ref_nxt = verify.tree_accept(am_ref, tokens, parent)
    if all(eligible[[0] + ref_path]):
        assert (path, nxt) == (ref_path, ref_nxt)
        assert ref_path == [1, 3, 5, 7]

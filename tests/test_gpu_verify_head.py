"""sdv_verify_head on the GPU vs the oracle, element by element.

Covers the tiny head over all 1000 seeded windows, window sizes S = 1 .. 32,
ragged vocabulary (not a multiple of the 16-row tile) and ragged reduction
length (not a multiple of the 256-element stage), int8 and int4, planted ties
and maxima in the last tile.  The two full-size heads run every seeded window
in test_gpu_windows.py.
"""
import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from synth import workloads as W
from tests.helpers import (GAP, assert_gemm_close, check_head_outputs, device_weight, gemm_path,
                           oracle_weight, run_head)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


_CURRENT = {"path": None}


@pytest.fixture(params=["mma", "tc"])
def path(request, sdv):
    """Run the test on each GEMM implementation (mma.sync and tcgen05)."""
    with gemm_path(request.param):
        _CURRENT["path"] = request.param
        yield request.param
        _CURRENT["path"] = None


def _synthetic_head(n, k, bits, seed):
    w = G.normal(G.stream_seed(900, n, k, bits, seed), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, bits)
    return codes, scales, stored


def _x(S, k, seed):
    return G.normal(G.stream_seed(901, S, k, seed), (S, k), 1.0, dtype=np.float64).astype(np.float16)


def _window(sdv, head, codes, scales, x, seed, k):
    S = x.shape[0]
    ref0 = verify.verify_head(x, codes, scales, np.zeros(max(S - 1, 0), np.int32), 0)
    rng = np.random.default_rng(seed)
    j = int(rng.integers(0, S))
    drafts = rng.integers(0, head.n, max(S - 1, 0)).astype(np.int32)
    drafts[:j] = ref0["argmax"][:j]
    n_valid = S - 1
    ref = verify.verify_head(x, codes, scales, drafts, n_valid)
    try:
        logits, am, acc, nxt = run_head(head, x, drafts, n_valid)
    except sdv.SdvError as e:
        if e.status == sdv.SDV_ERR_UNSUPPORTED and _CURRENT["path"] == "tc":
            pytest.skip("window rows x reduction length do not fit the tcgen05 plan")
        raise
    assert_gemm_close(logits, ref["logits"], k, "logits")
    check_head_outputs(ref, am, acc, nxt)
    return ref, am, acc, nxt


def test_tiny_head_all_windows(sdv, path):
    wl = W.TINY
    w = W.head_weights(wl)
    codes, scales, stored = oracle_weight(w, 8)
    head = device_weight(stored, scales, 8, wl.n, wl.h)
    eligible = total = accepted_checked = 0
    for win in range(wl.windows):
        x = W.activations(wl, win, 9)
        ref0 = verify.verify_head(x, codes, scales, np.zeros(8, np.int32), 0)
        drafts, n_valid = W.drafts(wl, win, 9, ref0["argmax"])
        ref = verify.verify_head(x, codes, scales, drafts, n_valid)
        logits, am, acc, nxt = run_head(head, x, drafts, n_valid, want_logits=(win % 50 == 0))
        if logits is not None:
            assert_gemm_close(logits, ref["logits"], wl.h, f"window {win} logits")
        eligible += check_head_outputs(ref, am, acc, nxt)
        total += 9
        accepted_checked += int((ref["gap"][: ref["accepted"] + 1] > GAP).all())
    # logit std 0.32 over 4096 rows: about one row in ten has a top-2 gap under 1e-2;
    # the exemption must stay that rare, or the comparison above checks little
    assert eligible >= 0.85 * total
    assert accepted_checked >= 0.5 * wl.windows


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("S", [1, 2, 3, 8, 9, 16, 17, 24, 25, 32])
def test_window_sizes(sdv, path, bits, S):
    n, k = 1000, 512
    codes, scales, stored = _synthetic_head(n, k, bits, S)
    head = device_weight(stored, scales, bits, n, k)
    _window(sdv, head, codes, scales, _x(S, k, S), S, k)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("n,k", [(1, 32), (17, 64), (4097, 96), (2000, 288), (3001, 800), (640, 2560)])
def test_ragged_shapes(sdv, path, bits, n, k):
    codes, scales, stored = _synthetic_head(n, k, bits, 1)
    head = device_weight(stored, scales, bits, n, k)
    for S in (1, 9, 17):
        _window(sdv, head, codes, scales, _x(S, k, n + S), n + S, k)


@pytest.mark.parametrize("S", [17, 25, 32])
def test_int4_long_reduction_wide_windows(sdv, path, S):
    """int4 at K = 2048 with window sizes whose staged rows fill most of the
    tensor-core path's shared memory (S = 32: ring depth 4)."""
    n, k = 3000, 2048
    codes, scales, stored = _synthetic_head(n, k, 4, 7)
    head = device_weight(stored, scales, 4, n, k)
    _window(sdv, head, codes, scales, _x(S, k, 70 + S), 70 + S, k)


@pytest.mark.parametrize("S", [17, 25, 32])
def test_int8_long_reduction_wide_windows(sdv, path, S):
    """int8 at K = 2560 (the q4b head's reduction): the widest windows exceed
    one launch's shared memory on either path and are verified in row chunks."""
    n, k = 3000, 2560
    codes, scales, stored = _synthetic_head(n, k, 8, 11)
    head = device_weight(stored, scales, 8, n, k)
    _window(sdv, head, codes, scales, _x(S, k, 90 + S), 90 + S, k)


@pytest.mark.parametrize("bits", [8, 4])
def test_large_block_scales(sdv, path, bits):
    """Some 32-blocks carry weights ~1e4 times larger (int4 block scales of about
    50 to 160), scattered so that some warps hold none, some a few; rows without
    them are checked against their own magnitude too."""
    n, k, S = 1500, 512, 9
    w = G.normal(G.stream_seed(902, n, k, bits), (n, k), 0.02)
    rng = np.random.default_rng(5)
    big = rng.random((n, k // 32)) < 0.02
    big[:400] = False                      # the first 400 rows: no large block at all
    w = w.reshape(n, k // 32, 32)
    w[big] *= np.float32(1.5e4)
    w = w.reshape(n, k)
    codes, scales, stored = oracle_weight(w, bits)
    head = device_weight(stored, scales, bits, n, k)
    ref, _, _, _ = _window(sdv, head, codes, scales, _x(S, k, 3), 3, k)
    logits, _, _, _ = run_head(head, _x(S, k, 3), np.zeros(S - 1, np.int32), 0)
    plain = ~big.any(axis=1)
    assert_gemm_close(logits[:, plain], ref["logits"][:, plain], k, "logits of rows without large blocks")


def test_planted_ties_and_tail_maximum(sdv, path):
    # rows with identical codes and scales give identical logits: lowest index wins;
    # a dominant row in the last (ragged) tile must be found
    n, k, S = 4099, 256, 9
    codes, scales, stored = _synthetic_head(n, k, 8, 7)
    codes = codes.copy()
    scales = scales.copy()
    big = np.full(k, 127, np.int8)
    for r in (5, 1234, 4098):
        codes[r] = big
        scales[r] = scales[0]
    x = np.ones((S, k), np.float16)
    head = device_weight(codes, scales, 8, n, k)
    ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
    logits, am, acc, nxt = run_head(head, x, np.zeros(S - 1, np.int32), 0)
    assert np.all(ref["argmax"] == 5) and np.all(am == 5)
    # now make only the last row dominant
    codes[5] = codes[0]
    codes[1234] = codes[0]
    head = device_weight(codes, scales, 8, n, k)
    ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
    _, am, _, _ = run_head(head, x, np.zeros(S - 1, np.int32), 0)
    assert np.all(ref["argmax"] == 4098) and np.all(am == 4098)


def test_accept_paths_on_device(sdv, path):
    # all drafts equal the argmax -> bonus; first mismatch at 0; pads never accepted
    n, k, S = 2048, 256, 9
    codes, scales, stored = _synthetic_head(n, k, 8, 3)
    head = device_weight(stored, scales, 8, n, k)
    # a window whose rows are all well separated, so every decision is compared exactly
    for seed in range(200):
        x = _x(S, k, seed)
        ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
        if (ref["gap"] > GAP).all():
            break
    assert (ref["gap"] > GAP).all()
    am_ref = ref["argmax"]
    _, am, acc, nxt = run_head(head, x, am_ref[: S - 1].copy(), S - 1, want_logits=False)
    assert acc == S - 1 and nxt == am_ref[S - 1]
    bad = am_ref[: S - 1].copy()
    bad[0] = (bad[0] + 1) % n
    _, am, acc, nxt = run_head(head, x, bad, S - 1, want_logits=False)
    assert acc == 0 and nxt == am_ref[0]
    _, am, acc, nxt = run_head(head, x, am_ref[: S - 1].copy(), 3, want_logits=False)
    assert acc == 3 and nxt == am_ref[3]
    _, am, acc, nxt = run_head(head, x, am_ref[: S - 1].copy(), 0, want_logits=False)
    assert acc == 0 and nxt == am_ref[0]


def test_workspace_reused_across_calls(sdv, path):
    n, k, S = 3000, 512, 9
    codes, scales, stored = _synthetic_head(n, k, 4, 9)
    head = device_weight(stored, scales, 4, n, k)
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, n, k, S)
    for rep in range(5):
        x = _x(S, k, 100 + rep)
        ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
        logits, am, acc, nxt = run_head(head, x, np.zeros(S - 1, np.int32), 0, ws=ws)
        check_head_outputs(ref, am, acc, nxt)
    assert int(ws[4:8].view(torch.int32).item()) == 0  # ticket counter back at zero

"""The CUDA-core GEMV (sdv_set_gemm_path(3)) for windows of one or two rows, vs
the oracle under the same rules as the tensor-core paths: logits / Y within
2e-3 sqrt(k / 256) of the output's RMS, ids exact where the oracle's top-2 gap
exceeds 1e-2, the accept exact.  Ragged vocabularies and reduction lengths
(chunks of 16 bytes not a multiple of a warp's), int8, int4 and FP4.  The
full-size heads run every seeded window on this path in test_gpu_windows.py."""
import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from tests.helpers import (assert_gemm_close, check_head_outputs, device_weight, gemm_path, oracle_weight, run_head,
                           to_dev_f16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _case(bits, n, k, S, seed):
    w = G.normal(G.stream_seed(1300, n, k, bits, seed), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, bits)
    x = G.normal(G.stream_seed(1301, n, k, S, seed), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    return codes, scales, stored, x


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("S", [1, 2])
@pytest.mark.parametrize("n,k", [(1, 32), (17, 64), (4097, 96), (2000, 288), (3001, 800), (1500, 2048),
                                 (1000, 2560), (300, 5120)])
def test_head(sdv, bits, S, n, k):
    codes, scales, stored, x = _case(bits, n, k, S, 1)
    head = device_weight(stored, scales, bits, n, k)
    ref0 = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
    drafts = ref0["argmax"][: S - 1].copy()
    ref = verify.verify_head(x, codes, scales, drafts, S - 1)
    with gemm_path("gemv"):
        logits, am, acc, nxt = run_head(head, x, drafts, S - 1)
        _, am2, acc2, nxt2 = run_head(head, x, drafts, S - 1, want_logits=False)
    assert_gemm_close(logits, ref["logits"], k, "gemv logits")
    check_head_outputs(ref, am, acc, nxt)
    np.testing.assert_array_equal(am2, am)
    assert (acc2, nxt2) == (acc, nxt)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("S", [1, 2])
def test_qlinear(sdv, bits, S):
    n, k = 5120, 2048
    codes, scales, stored, x = _case(bits, n, k, S, 2)
    qw = device_weight(stored, scales, bits, n, k)
    y = torch.full((S, n), float("nan"), dtype=torch.float32, device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
    with gemm_path("gemv"):
        sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
    assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    assert_gemm_close(y.cpu().numpy(), verify.dequant_gemm64(x, codes, scales), k, "gemv Y")


def test_planted_ties(sdv):
    """Identical rows give identical logits: the lowest index wins; a dominant row
    at the very end of the vocabulary is found."""
    n, k, S = 4099, 256, 2
    codes, scales, stored, _ = _case(8, n, k, S, 3)
    codes = codes.copy()
    for r in (5, 1234, 4098):
        codes[r] = 127
        scales[r] = scales[0]
    x = np.ones((S, k), np.float16)
    head = device_weight(codes, scales, 8, n, k)
    with gemm_path("gemv"):
        _, am, _, _ = run_head(head, x, np.zeros(S - 1, np.int32), 0, want_logits=False)
        assert np.all(am == 5)
        codes[5] = codes[0]
        codes[1234] = codes[0]
        head = device_weight(codes, scales, 8, n, k)
        _, am, _, _ = run_head(head, x, np.zeros(S - 1, np.int32), 0, want_logits=False)
    assert np.all(am == 4098)

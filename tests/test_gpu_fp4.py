"""FP4 (E2M1) weights on the GPU vs the oracle.

* sdv_quantize_block32(SDV_F4) bit-exact against oracle.quant.quantize_fp4_block32
  (random blocks and the hand-worked tie blocks of tests/golden);
* the verify head, the sampling verify's draws and sdv_qlinear on FP4 weights
  against the oracle's fp64 GEMM of the decoded values, within the logits bound;
* the mma.sync path does not take FP4 weights (SDV_ERR_UNSUPPORTED).
"""
import os

import numpy as np
import pytest
import torch

from oracle import quant, sample, verify
from synth import generator as G
from tests.helpers import assert_gemm_close, check_head_outputs, gemm_path, run_head, to_dev, to_dev_f16, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _fp4_weight(sdv, w):
    n, k = w.shape
    c4, scales = quant.quantize_fp4_block32(w)
    packed = quant.pack_nibbles(c4)
    codes_t = to_dev(packed)
    scales_t = torch.from_numpy(np.ascontiguousarray(scales.view(np.int16))).cuda().view(torch.float16)
    return c4, scales, sdv.QWeight(codes_t, scales_t, sdv.SDV_F4, n, k)


def test_quantize_bit_exact(sdv):
    rng = np.random.default_rng(0)
    w = rng.normal(0, 0.02, (300, 512)).astype(np.float32)
    w[5, :32] = 0.0
    w[6, :32] = np.float32(1e4)
    golden = os.path.join(os.path.dirname(__file__), "golden", "fp4_block32_worked.txt")
    rows = [np.array([eval(t) for t in line.split(":", 1)[1].split()], np.float32)
            for line in open(golden) if line.startswith("w:")]
    w[7, :32], w[8, :32] = rows[0], rows[1]
    c_ref, s_ref = quant.quantize_fp4_block32(w)
    q = sdv.quantize(torch.from_numpy(w).cuda(), sdv.SDV_F4)
    assert np.array_equal(q.codes.cpu().numpy(), quant.pack_nibbles(c_ref))
    assert np.array_equal(q.scales.cpu().numpy().view(np.uint16), s_ref.view(np.uint16))


@pytest.mark.parametrize("n,k", [(3000, 512), (4097, 2048), (1000, 288)])
@pytest.mark.parametrize("S", [1, 9, 17, 32])
def test_verify_head(sdv, n, k, S):
    w = G.normal(G.stream_seed(990, n, k), (n, k), 0.02)
    vals, scales, qw = _fp4_weight(sdv, w)
    x = G.normal(G.stream_seed(991, S, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    drafts = np.zeros(max(S - 1, 0), np.int32)
    ref0 = verify.verify_head(x, vals, scales, drafts, 0)
    drafts[:S // 2] = ref0["argmax"][:S // 2]
    ref = verify.verify_head(x, vals, scales, drafts, S - 1)
    try:
        logits, am, acc, nxt = run_head(qw, x, drafts, S - 1)
    except sdv.SdvError as e:
        assert e.status == sdv.SDV_ERR_UNSUPPORTED
        pytest.skip("window rows x reduction length beyond the tensor-core plan")
    assert_gemm_close(logits, ref["logits"], k, "logits")
    check_head_outputs(ref, am, acc, nxt)


def test_qlinear(sdv):
    n, k, S = 777, 288, 5
    w = G.normal(G.stream_seed(992, n, k), (n, k), 0.02)
    vals, scales, qw = _fp4_weight(sdv, w)
    x = G.normal(G.stream_seed(993, S, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    y = torch.full((S, n), float("nan"), device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
    sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
    assert_gemm_close(y.cpu().numpy(), verify.dequant_gemm64(x, vals, scales), k, "Y")


def test_sampling_draws(sdv):
    n, k, S, T = 4096, 512, 9, 1.0
    w = G.normal(G.stream_seed(994, n, k), (n, k), 0.02)
    vals, scales, qw = _fp4_weight(sdv, w)
    x = G.normal(G.stream_seed(995, S, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    L = verify.dequant_gemm64(x, vals, scales)
    ref = sample.verify_sample(L, np.zeros(S - 1, np.int64), 0, T, 3, 4)
    smp = torch.empty(S, dtype=torch.int32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_SAMPLE, n, k, S)
    sdv.sdv_verify_sample(qw, to_dev_f16(x), S, torch.zeros(S - 1, dtype=torch.int32, device="cuda"), 0, T, 3, 4,
                          None, smp, acc, nxt, ws)
    rms = float(np.sqrt(np.mean(L ** 2)))
    zt = 4 * tol(k) * rms / T + 1e-4
    got = smp.cpu().numpy()
    checked = 0
    for i in range(S):
        if ref["z_gap"][i] > zt:
            assert got[i] == ref["samples"][i]
            checked += 1
    assert checked >= S // 2


def test_mma_path_rejects_fp4(sdv):
    n, k, S = 512, 256, 4
    w = G.normal(G.stream_seed(996, n, k), (n, k), 0.02)
    _, _, qw = _fp4_weight(sdv, w)
    x = np.zeros((S, k), np.float16)
    with gemm_path("mma"):
        with pytest.raises(sdv.SdvError) as e:
            run_head(qw, x, np.zeros(S - 1, np.int32), 0)
    assert e.value.status == sdv.SDV_ERR_UNSUPPORTED


@pytest.mark.parametrize("n,k,S", [(384, 512, 9), (200, 512, 17)])
def test_swiglu(sdv, n, k, S):
    from tests.test_gpu_mlp_moe import _swiglu_case
    _swiglu_case(sdv, 2, n, k, S, seed=n + S)


@pytest.mark.parametrize("S,E,I,H,top_k", [(5, 8, 256, 512, 2), (17, 32, 256, 512, 8)])
def test_moe(sdv, S, E, I, H, top_k):
    from tests.test_gpu_mlp_moe import _moe_case
    _moe_case(sdv, 2, S, E, I, H, top_k, seed=S * 3 + E)


def test_full_size_a3b_fp4_head(sdv):
    """The 35B-A3B-shaped head (248320 x 2048) with FP4 weights at S = 17, in the
    launch configuration the bench times: quantised on the GPU (bit-exact against
    the oracle), logits within the bound, ids where the oracle's gap allows, and
    the timed form (no logits) returning the same ids."""
    from synth import workloads as W
    wl, S = W.A3B, 17
    w = W.head_weights(wl)
    c4, scales = quant.quantize_fp4_block32(w)
    qw = sdv.quantize(to_dev(w), sdv.SDV_F4)
    del w
    torch.cuda.synchronize()
    assert np.array_equal(qw.codes.cpu().numpy(), quant.pack_nibbles(c4))
    assert np.array_equal(qw.scales.cpu().numpy().view(np.uint16), scales.view(np.uint16))
    vals = c4  # E2M1 codes: the oracle's GEMM decodes them exactly
    x = W.activations(wl, 0, S)
    ref0 = verify.verify_head(x, vals, scales, np.zeros(S - 1, np.int32), 0)
    drafts, n_valid = W.drafts(wl, 0, S, ref0["argmax"])
    ref = verify.verify_head(x, vals, scales, drafts, n_valid)
    logits, am, acc, nxt = run_head(qw, x, drafts, n_valid)
    assert_gemm_close(logits, ref["logits"], wl.h, "a3b fp4 logits")
    check_head_outputs(ref, am, acc, nxt)
    _, am2, acc2, nxt2 = run_head(qw, x, drafts, n_valid, want_logits=False)
    np.testing.assert_array_equal(am2, am)
    assert (acc2, nxt2) == (acc, nxt)

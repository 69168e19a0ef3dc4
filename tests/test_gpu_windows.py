"""Parity on every seeded window of the full-size workloads, in the launch
configuration the benchmark times (the tiny head's 1000 windows are in
test_gpu_verify_head.py).

* Verify heads -- the Qwen3-4B-shaped head (151936 x 2560 int8, S = 9) and the
  35B-A3B-shaped head (248320 x 2048 int4, S = 1, 2, 9, 17), 200 windows each,
  on both tensor-core implementations (and on the CUDA-core GEMV at S = 1, 2).  Every window: argmax bit-exact on every row
  whose oracle top-2 gap exceeds 1e-2, accepted and next_a0 bit-exact when
  every row the accept scan read is eligible, the window's drafts rebuilt from
  the oracle's argmax chain by the seeded draft rule.  The oracle's per-window
  results come from tests/golden/head_windows_*.jsonl (written by
  tests/golden/make_head_windows.py, which calls only oracle/); every tenth
  window the oracle runs here as well: full logits within the bound, and the
  stored results equal to the oracle's.  At least 85 % of all rows must be
  eligible, so that the exemption stays rare.
* SwiGLU projection stack (mlp27: gate/up 17408 x 5120, down 5120 x 17408,
  int8, S = 1, 9, 17), 200 windows each, both implementations: h against the
  propagated SwiGLU bound and Y of the down projection (on the GPU's own h)
  against the oracle, on 128 sampled columns of every window (the oracle
  evaluated column by column) and on the whole output every tenth window.
  The sampled checks take the scale of the bound from the oracle's RMS of g
  and u over the whole window (tests/golden/mlp_windows_mlp27_s*.jsonl) and,
  for Y, from the GPU output: if max |Y_gpu - Y| <= t RMS(Y) holds, then
  RMS(Y) <= RMS(Y_gpu) / (1 - t), so t RMS(Y_gpu) / (1 - t) bounds the
  sampled errors whenever the full check would pass.
* MoE (256 experts, top-8, int4, S = 17), 200 windows: routing ids bit-exact,
  weights to 2e-6 relative, rel-L2 <= 1e-3 over out[S, H], the oracle run
  here on every window.  The layer exists on the tcgen05 path only: with the
  mma.sync path selected the call returns SDV_ERR_UNSUPPORTED.
"""
import numpy as np
import pytest
import torch

from oracle import mlp, quant, verify
from synth import workloads as W
from tests.helpers import (GAP, assert_gemm_close, check_head_outputs, gemm_path, load_windows, run_head, to_dev,
                           to_dev_f16, tol)

pytestmark = pytest.mark.gpu

FULL_EVERY = 10


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _quantized_pair(sdv, w, bits):
    """The weight quantised on the GPU and by the oracle, checked bit-exact."""
    n, k = w.shape
    dw = sdv.quantize(to_dev(w), bits)
    codes, scales = quant.quantize_block32(w, bits)
    torch.cuda.synchronize()
    stored = codes if bits == 8 else quant.pack_int4(codes)
    np.testing.assert_array_equal(dw.codes.cpu().numpy().view(np.uint8), stored.view(np.uint8))
    np.testing.assert_array_equal(dw.scales.cpu().numpy().view(np.uint16), scales.view(np.uint16))
    return dw, codes, scales


# ------------------------------------------------------------------ heads ----

_HEADS = {}
_ORACLE_LOGITS = {}


def _head(sdv, wl):
    if wl.name not in _HEADS:
        w = W.head_weights(wl)
        _HEADS[wl.name] = _quantized_pair(sdv, w, wl.bits)
        del w
    return _HEADS[wl.name]


HEAD_CASES = ([(name, S, p) for name, s_list in (("q4b", (9,)), ("a3b", (1, 2, 9, 17)))
               for S in s_list for p in ("tc", "mma")]
              + [("a3b", 1, "gemv"), ("a3b", 2, "gemv")])


@pytest.mark.parametrize("name,S,path_name", HEAD_CASES)
def test_head_every_window(sdv, name, S, path_name):
    wl = W.BY_NAME[name]
    _, recs = load_windows("head_windows", name, S)
    assert [r["window"] for r in recs] == list(range(wl.windows))
    head, codes, scales = _head(sdv, wl)
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, wl.n, wl.h, S)
    eligible = total = scanned = 0
    with gemm_path(path_name):
        for rec in recs:
            win = rec["window"]
            x = W.activations(wl, win, S)
            drafts, n_valid = W.drafts(wl, win, S, rec["argmax"])
            assert drafts.tolist() == rec["drafts"] and n_valid == rec["n_valid"]
            full = win % FULL_EVERY == 0
            logits, am, acc, nxt = run_head(head, x, drafts, n_valid, want_logits=full, ws=ws)
            ref = {"argmax": np.asarray(rec["argmax"], np.int32), "gap": np.asarray(rec["gap"]),
                   "accepted": rec["accepted"], "next_a0": rec["next_a0"]}
            eligible += check_head_outputs(ref, am, acc, nxt)
            total += S
            scanned += int((ref["gap"][: ref["accepted"] + 1] > GAP).all())
            if full:
                key = (name, S, win)
                if key not in _ORACLE_LOGITS:
                    _ORACLE_LOGITS[key] = verify.verify_head(x, codes, scales, drafts, n_valid)
                o = _ORACLE_LOGITS[key]
                assert_gemm_close(logits, o["logits"], wl.h, f"{name} S={S} window {win} logits")
                # the stored results are this oracle's
                np.testing.assert_array_equal(o["argmax"], ref["argmax"])
                assert (o["accepted"], o["next_a0"]) == (rec["accepted"], rec["next_a0"])
                np.testing.assert_allclose(o["gap"], ref["gap"], rtol=1e-7, atol=1e-12)
                # the timed form (no logits) gives the same ids
                _, am2, acc2, nxt2 = run_head(head, x, drafts, n_valid, want_logits=False, ws=ws)
                np.testing.assert_array_equal(am2, am)
                assert (acc2, nxt2) == (acc, nxt)
    assert eligible >= 0.85 * total, f"only {eligible} of {total} rows eligible"
    assert scanned >= 0.5 * wl.windows


# ------------------------------------------------------------------ mlp27 ----

_MLP = {}


def _mlp(sdv):
    if not _MLP:
        wl = W.MLP27
        for which in ("gate", "up", "down"):
            w = W.mlp_weights(wl, which)
            _MLP[which] = _quantized_pair(sdv, w, wl.bits)
            del w
    return _MLP


def _dsilu(t):
    sg = 1.0 / (1.0 + np.exp(-t))
    return sg * (1.0 + t * (1.0 - sg))


def _swiglu_bound(g64, u64, eg, eu):
    """Per-element bound on |h_gpu - SiLU(g) u| (see test_gpu_mlp_moe.py)."""
    h64 = mlp.silu(g64) * u64
    ulp = np.spacing(np.abs(h64).astype(np.float16)).astype(np.float64)
    return h64, (np.abs(_dsilu(g64)) * np.abs(u64) * eg + (np.abs(mlp.silu(g64)) + 1.1 * eg) * eu
                 + 0.5 * eg * eg * np.abs(u64) + 0.5 * ulp + 1e-30)


def _mlp_window(sdv, M, x, ws_g, ws_d):
    S = x.shape[0]
    (gate, _, _), (up, _, _), (down, _, _) = M["gate"], M["up"], M["down"]
    h = torch.full((S, gate.n), float("nan"), dtype=torch.float16, device="cuda")
    y = torch.full((S, down.n), float("nan"), dtype=torch.float32, device="cuda")
    sdv.sdv_qlinear_swiglu(gate, up, to_dev_f16(x), S, h, ws_g)
    sdv.sdv_qlinear(down, h, S, y, ws_d)
    assert sdv.sdv_last_device_status(ws_g) == sdv.SDV_OK
    assert sdv.sdv_last_device_status(ws_d) == sdv.SDV_OK
    return h.cpu().numpy(), y.cpu().numpy()


@pytest.mark.parametrize("S", [1, 9, 17])
def test_mlp27_every_window(sdv, S):
    wl = W.MLP27
    _, recs = load_windows("mlp_windows", "mlp27", S)
    assert [r["window"] for r in recs] == list(range(wl.windows))
    M = _mlp(sdv)
    (_, cg, sg), (_, cu, su), (_, cd, sd) = M["gate"], M["up"], M["down"]
    ws_g = sdv.workspace(sdv.SDV_OP_QLINEAR_SWIGLU, wl.inter, wl.h, S)
    ws_d = sdv.workspace(sdv.SDV_OP_QLINEAR, wl.h, wl.inter, S)
    t_gu, t_d = tol(wl.h), tol(wl.inter)
    for rec in recs:
        win = rec["window"]
        x = W.activations(wl, win, S)
        rng = np.random.default_rng([77, S, win])
        cols_h = np.sort(rng.choice(wl.inter, 128, replace=False))
        cols_y = np.sort(rng.choice(wl.h, 128, replace=False))
        g_s = verify.dequant_gemm64(x, cg[cols_h], sg[cols_h])
        u_s = verify.dequant_gemm64(x, cu[cols_h], su[cols_h])
        eg, eu = t_gu * rec["rms_g"], t_gu * rec["rms_u"]
        full = win % FULL_EVERY == 0
        if full:
            g64, u64 = verify.dequant_gemm64(x, cg, sg), verify.dequant_gemm64(x, cu, su)
            np.testing.assert_allclose([np.sqrt(np.mean(g64 ** 2)), np.sqrt(np.mean(u64 ** 2))],
                                       [rec["rms_g"], rec["rms_u"]], rtol=1e-12)
        for path_name in ("tc", "mma"):
            with gemm_path(path_name):
                h, y = _mlp_window(sdv, M, x, ws_g, ws_d)
            what = f"mlp27 S={S} window {win} {path_name}"
            h64_s, bound = _swiglu_bound(g_s, u_s, eg, eu)
            err = np.abs(h[:, cols_h].astype(np.float64) - h64_s)
            assert (err <= bound).all(), f"{what}: h beyond the bound on {int((err > bound).sum())} sampled entries"
            y_s = verify.dequant_gemm64(h, cd[cols_y], sd[cols_y])
            rms_gpu = float(np.sqrt(np.mean(y.astype(np.float64) ** 2)))
            yb = t_d * rms_gpu / (1.0 - t_d)
            assert np.abs(y[:, cols_y] - y_s).max() <= yb, f"{what}: sampled Y beyond the bound"
            if full:
                h64, bound = _swiglu_bound(g64, u64, eg, eu)
                assert (np.abs(h.astype(np.float64) - h64) <= bound).all(), f"{what}: h beyond the bound"
                assert_gemm_close(y, verify.dequant_gemm64(h, cd, sd), wl.inter, f"{what}: Y")


# -------------------------------------------------------------------- moe ----

_MOE = {}


def _moe(sdv):
    if not _MOE:
        wl = W.MOE
        for which in ("gate", "up", "down"):
            w = W.moe_weights(wl, which)
            dw, codes, scales = _quantized_pair(sdv, w, wl.bits)
            del w
            _MOE[which] = ((codes, scales), dw)
    return _MOE


def _run_moe(sdv, T, wl, x, logits, ws):
    E, I, H, k = wl.experts, wl.inter, wl.h, wl.top_k
    S = x.shape[0]
    out = torch.full((S, H), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((S, k), -1, dtype=torch.int32, device="cuda")
    wts = torch.full((S, k), float("nan"), dtype=torch.float32, device="cuda")
    sdv.sdv_moe_gather_qmm(T["gate"][1], T["up"][1], T["down"][1], E, I, H, k, to_dev_f16(x), to_dev(logits), S,
                           out, ids, wts, ws)
    assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    return out.cpu().numpy(), ids.cpu().numpy(), wts.cpu().numpy()


def test_moe_every_window(sdv):
    wl = W.MOE
    S = wl.s_default
    T = _moe(sdv)
    ws = sdv.workspace(sdv.SDV_OP_MOE, wl.inter, wl.h, S, wl.experts, wl.top_k)
    worst = 0.0
    for win in range(wl.windows):
        x = W.activations(wl, win, S)
        logits = W.router_logits(wl, win, S)
        out, ids, wts = _run_moe(sdv, T, wl, x, logits, ws)
        ref, rid, rw = mlp.moe_forward(x, logits, T["gate"][0], T["up"][0], T["down"][0], wl.experts, wl.inter,
                                       wl.h, wl.top_k)
        np.testing.assert_array_equal(ids, rid)
        np.testing.assert_allclose(wts, rw, rtol=2e-6, atol=1e-7)
        r = float(np.linalg.norm(out.astype(np.float64) - ref) / np.linalg.norm(ref.astype(np.float64)))
        assert r <= 1e-3, f"MoE window {win}: rel-L2 {r:.3e}"
        worst = max(worst, r)
    print(f"MoE: 200 windows, worst rel-L2 {worst:.2e}")


def test_moe_mma_path_is_unsupported(sdv):
    wl = W.MOE
    S = wl.s_default
    T = _moe(sdv)
    ws = sdv.workspace(sdv.SDV_OP_MOE, wl.inter, wl.h, S, wl.experts, wl.top_k)
    x = W.activations(wl, 0, S)
    with gemm_path("mma"):
        with pytest.raises(sdv.SdvError) as e:
            _run_moe(sdv, T, wl, x, W.router_logits(wl, 0, S), ws)
    assert e.value.status == sdv.SDV_ERR_UNSUPPORTED

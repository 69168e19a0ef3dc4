"""The bounded-wait timeout path of the tcgen05 kernels, made to run on purpose
without faulting or hanging anything.

sdv_debug_fault withholds the weight copy of one ring stage in every CTA: the
converters waiting for it find a barrier that nothing will complete and give up
after a short limit (2 ms here), with no copy in flight behind that stage.  The
kernel then drains what it issued, frees its tensor memory, writes undefined
outputs and records the timeout in the status word.  The tests check that the
status read returns SDV_ERR_TIMEOUT exactly once and that the next normal call
on the same workspace (or the no-workspace head's fixed scratch) is correct.
"""
import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from tests.helpers import (assert_gemm_close, check_head_outputs, device_weight, gemm_path, oracle_weight,
                           run_head, to_dev, to_dev_f16)

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


class fault:
    """Withhold one stage per CTA and shorten the waits, for the block's calls only."""

    def __init__(self, sdv, stage):
        self.sdv, self.stage = sdv, stage

    def __enter__(self):
        self.sdv.sdv_debug_fault(self.stage, LIMIT_NS)

    def __exit__(self, *a):
        self.sdv.sdv_debug_fault(-1, 0)


def _head_case(bits, n=3000, k=512, S=9):
    w = G.normal(G.stream_seed(1200, n, k, bits), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, bits)
    x = G.normal(G.stream_seed(1201, n, k, bits), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    return codes, scales, stored, x


def _launch_head(sdv, head, x, ws=None):
    S = x.shape[0]
    am = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    acc = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    d = torch.zeros(S - 1, dtype=torch.int32, device="cuda")
    if ws is None:
        sdv.sdv_verify_head_noalloc(head, to_dev_f16(x), S, d, 0, None, am, acc, nxt)
    else:
        sdv.sdv_verify_head(head, to_dev_f16(x), S, d, 0, None, am, acc, nxt, ws)


def test_invalid_fault_arguments_are_rejected(sdv):
    with pytest.raises(sdv.SdvError):
        sdv.sdv_debug_fault(-2, 0)
    with pytest.raises(sdv.SdvError):
        sdv.sdv_debug_fault(1, 10)  # a limit below 0.1 ms
    sdv.sdv_debug_fault(-1, 0)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("stage", [0, 1])
def test_head_timeout_reported_then_next_call_correct(sdv, bits, stage):
    n, k, S = 3000, 512, 9
    codes, scales, stored, x = _head_case(bits, n, k, S)
    head = device_weight(stored, scales, bits, n, k)
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, n, k, S)
    with gemm_path("tc"):
        with fault(sdv, stage):
            _launch_head(sdv, head, x, ws)
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_ERR_TIMEOUT
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK  # read and cleared
        # the next normal call on the same workspace is correct
        ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
        logits, am, acc, nxt = run_head(head, x, np.zeros(S - 1, np.int32), 0, ws=ws)
        assert_gemm_close(logits, ref["logits"], k, "logits after a timeout")
        check_head_outputs(ref, am, acc, nxt)
        assert int(ws[4:8].view(torch.int32).item()) == 0  # the ticket is back at zero


def test_qlinear_split_timeout_reported_then_next_call_correct(sdv):
    """Y mode with split-K partials (the reduce that follows reads undefined
    partials after the timeout, then everything is correct again)."""
    n, k, S = 1024, 4096, 9
    w = G.normal(G.stream_seed(1210, n, k), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, 8)
    qw = device_weight(stored, scales, 8, n, k)
    x = G.normal(G.stream_seed(1211, n, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
    y = torch.full((S, n), float("nan"), dtype=torch.float32, device="cuda")
    with gemm_path("tc"):
        with fault(sdv, 0):  # 16 splits of one 256-column stage per CTA: stage 0 is every CTA's only one
            sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_ERR_TIMEOUT
        # every output is written again (a skipped one would stay NaN)
        y.fill_(float("nan"))
        sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    assert_gemm_close(y.cpu().numpy(), verify.dequant_gemm64(x, codes, scales), k, "Y after a timeout")


def test_swiglu_split_timeout_reported_then_next_calls_correct(sdv):
    """Gate/up with split-K partials (then the SwiGLU reduce): after the
    timeout, the next calls on the same workspace write every h value again,
    correctly."""
    from tests.test_gpu_mlp_moe import assert_swiglu_close
    n, k, S = 1024, 5120, 17
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR_SWIGLU, n, k, S)
    mats = []
    for m in range(2):
        w = G.normal(G.stream_seed(1220, m, n, k), (n, k), 0.02)
        codes, scales, stored = oracle_weight(w, 8)
        mats.append((codes, scales, device_weight(stored, scales, 8, n, k)))
    (cg, sg, gate), (cu, su, up) = mats
    h = torch.full((S, n), float("nan"), dtype=torch.float16, device="cuda")
    with gemm_path("tc"):
        x0 = G.normal(G.stream_seed(1221, n, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
        with fault(sdv, 0):
            sdv.sdv_qlinear_swiglu(gate, up, to_dev_f16(x0), S, h, ws)
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_ERR_TIMEOUT
        for call in range(2):
            x = G.normal(G.stream_seed(1222, call, n, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
            h.fill_(float("nan"))
            sdv.sdv_qlinear_swiglu(gate, up, to_dev_f16(x), S, h, ws)
            assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
            assert_swiglu_close(h.cpu().numpy().astype(np.float64), verify.dequant_gemm64(x, cg, sg),
                                verify.dequant_gemm64(x, cu, su), k, f"h, call {call} after a timeout")


def test_noalloc_timeout_reported_then_next_call_correct(sdv):
    n, k, S = 3000, 512, 9
    codes, scales, stored, x = _head_case(4, n, k, S)
    head = device_weight(stored, scales, 4, n, k)
    assert sdv.sdv_noalloc_device_status() == sdv.SDV_OK
    with gemm_path("tc"):
        with fault(sdv, 1):
            _launch_head(sdv, head, x)
        assert sdv.sdv_noalloc_device_status() == sdv.SDV_ERR_TIMEOUT
        assert sdv.sdv_noalloc_device_status() == sdv.SDV_OK
        ref = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
        am = torch.full((S,), -1, dtype=torch.int32, device="cuda")
        acc = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        nxt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        lg = torch.full((S, n), float("nan"), dtype=torch.float32, device="cuda")
        sdv.sdv_verify_head_noalloc(head, to_dev_f16(x), S, to_dev(np.zeros(S - 1, np.int32)), 0, lg, am, acc, nxt)
        assert sdv.sdv_noalloc_device_status() == sdv.SDV_OK
    assert_gemm_close(lg.cpu().numpy(), ref["logits"], k, "noalloc logits after a timeout")
    check_head_outputs(ref, am.cpu().numpy(), int(acc.item()), int(nxt.item()))

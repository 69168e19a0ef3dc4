"""The verify head entry point that allocates nothing (sdv_verify_head_noalloc).

It serves callers that cannot allocate device memory themselves (a host
framework owns every byte of device memory, or the call sits in a loop where
an allocation is not allowed): the scratch lives in a fixed device array
inside the library.  Two calls in a row must match the workspace entry point
(sdv_verify_head) within the parity tolerance, with identical ids.  This file
is collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from oracle import quant
from synth import generator as G
from tests.helpers import assert_gemm_close, device_weight, to_dev, to_dev_f16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _outs(S, n, dev="cuda"):
    return (torch.full((S, n), float("nan"), dtype=torch.float32, device=dev),
            torch.full((S,), -1, dtype=torch.int32, device=dev),
            torch.full((1,), -1, dtype=torch.int32, device=dev),
            torch.full((1,), -1, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("bits", [8, 4])
def test_noalloc_matches_workspace_entry_point(sdv, bits):
    n, k, S = 20000, 512, 9
    w = G.normal(G.stream_seed(990, n, k, bits), (n, k), 0.02)
    codes, scales = quant.quantize_block32(w, bits)
    stored = codes if bits == 8 else quant.pack_int4(codes)
    head = device_weight(stored, scales, bits, n, k)
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, n, k, S)
    for call in range(2):  # two calls in a row share (and must re-clear) the fixed scratch
        x = G.normal(G.stream_seed(991, call, bits), (S, k), 1.0, dtype=np.float64).astype(np.float16)
        xt = to_dev_f16(x)
        lg_a, am_a, acc_a, nx_a = _outs(S, n)
        sdv.sdv_verify_head(head, xt, S, None, 0, lg_a, am_a, acc_a, nx_a, ws)
        # drafts: the first four ids of the window's own argmax chain, then a miss
        chain = am_a.cpu().numpy()
        drafts = chain[: S - 1].copy()
        drafts[4] = (drafts[4] + 1) % n
        dt = to_dev(drafts.astype(np.int32))
        lg_a, am_a, acc_a, nx_a = _outs(S, n)
        sdv.sdv_verify_head(head, xt, S, dt, S - 1, lg_a, am_a, acc_a, nx_a, ws)
        lg_b, am_b, acc_b, nx_b = _outs(S, n)
        sdv.sdv_verify_head_noalloc(head, xt, S, dt, S - 1, lg_b, am_b, acc_b, nx_b)
        torch.cuda.synchronize()
        assert_gemm_close(lg_b.cpu().numpy(), lg_a.cpu().numpy(), k, f"call {call} logits")
        np.testing.assert_array_equal(am_b.cpu().numpy(), am_a.cpu().numpy())
        assert int(acc_b.item()) == int(acc_a.item()) == 4
        assert int(nx_b.item()) == int(nx_a.item()) == int(chain[4])


def test_noalloc_rejects_bad_window(sdv):
    n, k = 64, 256
    head = device_weight(np.zeros((n, k), np.int8), np.ones((n, k // 32), np.float16), 8, n, k)
    x = torch.zeros((33, k), dtype=torch.float16, device="cuda")
    lg, am, acc, nx = _outs(33, n)
    with pytest.raises(sdv.SdvError) as e:
        sdv.sdv_verify_head_noalloc(head, x, 33, None, 0, lg, am, acc, nx)
    assert e.value.status == sdv.SDV_ERR_UNSUPPORTED

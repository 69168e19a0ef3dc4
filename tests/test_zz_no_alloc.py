"""The verify head entry point that allocates nothing (sdv_verify_head_noalloc).

It serves callers that cannot allocate device memory themselves (a host
framework owns every byte of device memory, or the call sits in a loop where
an allocation is not allowed): the scratch lives in a fixed device array
inside the library.  Two calls in a row must match the workspace entry point
(sdv_verify_head) -- bit for bit where both run the same plan, within the
parity tolerance where the workspace entry point splits the reduction and the
fixed scratch runs row chunks -- and the oracle.  The cases cover a plain
window, the widest window (S = 32, the largest scratch need) and the
row-chunked int8 head with k = 2560 at S = 17, where several launches reuse
the array in sequence.  This file is collected
last so that a run stopping at the first failure has already run every other
test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from tests.helpers import assert_gemm_close, check_head_outputs, device_weight, oracle_weight, to_dev, to_dev_f16

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


@pytest.mark.parametrize("bits,n,k,S", [(8, 20000, 512, 9), (4, 20000, 512, 9), (4, 3000, 2048, 32),
                                        (8, 3000, 2560, 17)])
def test_noalloc_matches_workspace_entry_point(sdv, bits, n, k, S):
    w = G.normal(G.stream_seed(990, n, k, bits), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, bits)
    head = device_weight(stored, scales, bits, n, k)
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, n, k, S)
    for call in range(2):  # two calls in a row share (and must re-clear) the fixed scratch
        x = G.normal(G.stream_seed(991, call, bits, S), (S, k), 1.0, dtype=np.float64).astype(np.float16)
        xt = to_dev_f16(x)
        ref0 = verify.verify_head(x, codes, scales, np.zeros(S - 1, np.int32), 0)
        # drafts: the first four ids of the oracle's argmax chain, then a miss
        drafts = ref0["argmax"][: S - 1].copy()
        drafts[4] = (drafts[4] + 1) % n
        ref = verify.verify_head(x, codes, scales, drafts, S - 1)
        dt = to_dev(drafts.astype(np.int32))
        lg_a, am_a, acc_a, nx_a = _outs(S, n)
        sdv.sdv_verify_head(head, xt, S, dt, S - 1, lg_a, am_a, acc_a, nx_a, ws)
        lg_b, am_b, acc_b, nx_b = _outs(S, n)
        sdv.sdv_verify_head_noalloc(head, xt, S, dt, S - 1, lg_b, am_b, acc_b, nx_b)
        assert sdv.sdv_noalloc_device_status() == sdv.SDV_OK
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
        if S <= 16 or bits == 4:
            # the same kernel and plan: the two entry points agree exactly
            np.testing.assert_array_equal(lg_b.cpu().numpy(), lg_a.cpu().numpy())
            np.testing.assert_array_equal(am_b.cpu().numpy(), am_a.cpu().numpy())
            assert (int(acc_b.item()), int(nx_b.item())) == (int(acc_a.item()), int(nx_a.item()))
        else:
            # int8 with k = 2560 at S = 17: the workspace entry point splits the
            # reduction, the fixed scratch runs row chunks: agreement within the
            # parity tolerance, ids exact where the oracle's gap allows
            assert_gemm_close(lg_b.cpu().numpy(), lg_a.cpu().numpy(), k, f"call {call} logits, the two forms")
            check_head_outputs(ref, am_a.cpu().numpy(), int(acc_a.item()), int(nx_a.item()))
        # and both match the oracle under the parity rules
        assert_gemm_close(lg_b.cpu().numpy(), ref["logits"], k, f"call {call} logits")
        check_head_outputs(ref, am_b.cpu().numpy(), int(acc_b.item()), int(nx_b.item()))


def test_noalloc_rejects_bad_arguments(sdv):
    n, k = 64, 256
    head = device_weight(np.zeros((n, k), np.int8), np.ones((n, k // 32), np.float16), 8, n, k)
    x = torch.zeros((33, k), dtype=torch.float16, device="cuda")
    lg, am, acc, nx = _outs(33, n)
    with pytest.raises(sdv.SdvError) as e:
        sdv.sdv_verify_head_noalloc(head, x, 33, None, 0, lg, am, acc, nx)
    assert e.value.status == sdv.SDV_ERR_UNSUPPORTED
    # a weight whose reduction length is not a multiple of 32 is an argument error
    bad = sdv.QWeight(head.codes, head.scales, 8, n, 40)
    with pytest.raises(sdv.SdvError) as e:
        sdv.sdv_verify_head_noalloc(bad, x, 9, None, 0, lg, am, acc, nx)
    assert e.value.status == sdv.SDV_ERR_INVALID_ARG
    assert sdv.sdv_noalloc_device_status() == sdv.SDV_OK

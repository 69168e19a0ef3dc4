"""The two integer-code -> fp16 conversions of the tcgen05 converters give the
same bits.

Where every row of a warp's 32-row slab has its block scales in range (int4:
2^-13 <= s <= 65504 * 2^-20 or s = 0, i.e. max |w| <= ~0.44 per block; int8:
s <= 65504 * 2^-24, max |w| <= ~0.5) the converters apply scale and bias in one
fp16 FMA on the code placed in the subnormal range; a slab with any scale out
of range takes the two-step form (exact code, then times s).  (int4 holds the
codes at bits 0-3 of a half as fp16(n * s / 16) in both forms; their
accumulators are scaled back by 16.)  Both round n * s once, so
a row's logits must not depend on which form its slab took: the same head is
run as is (every slab on the one-FMA form) and with the first row of every
32-row slab scaled up (those slabs on the two-step form), and the logits of the
rows the two share must agree bit for bit; every row also matches the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from tests.helpers import assert_gemm_close, check_head_outputs, device_weight, gemm_path, oracle_weight, run_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("S", [1, 9, 17])
@pytest.mark.parametrize("n,k", [(4096, 2048), (1000, 512)])
def test_fma_and_two_step_forms_agree(sdv, bits, n, k, S):
    w = G.normal(G.stream_seed(1300, n, k), (n, k), 0.02)
    big = w.copy()
    big[::32] *= 40.0  # first row of every 32-row slab: scales around 0.3, past the one-FMA range
    x = G.normal(G.stream_seed(1301, n, k, S), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    drafts = np.zeros(max(S - 1, 0), np.int32)
    keep = np.ones(n, bool)
    keep[::32] = False
    out = {}
    limit = 65504 * 2.0 ** (-20 if bits == 4 else -24)
    with gemm_path("tc"):
        for name, wm in (("plain", w), ("big", big)):
            codes, scales, stored = oracle_weight(wm, bits)
            if name == "big":
                assert float(np.min(np.max(scales[::32].astype(np.float32), axis=1))) > limit
            if name == "plain":
                assert float(np.max(scales.astype(np.float32))) <= limit
            head = device_weight(stored, scales, bits, n, k)
            logits, am, acc, nxt = run_head(head, x, drafts, 0)
            ref = verify.verify_head(x, codes, scales, drafts, 0)
            # the parity bound is relative to the RMS of the logits it covers:
            # the scaled-up rows and the others each against their own
            for rows, what in ((keep, "rows as drawn"), (~keep, "scaled-up rows")):
                assert_gemm_close(logits[:, rows], ref["logits"][:, rows], k, f"{name} logits, {what}")
            check_head_outputs(ref, am, acc, nxt)
            out[name] = logits
    np.testing.assert_array_equal(out["plain"][:, keep], out["big"][:, keep])


def test_int4_y_mode_large_scales(sdv):
    """sdv_qlinear on int4 weights whose every block scale is past the one-FMA
    range (N(0, 1) weights): the two-step form throughout, against the oracle."""
    n, k, S = 2048, 1024, 17
    w = G.normal(G.stream_seed(1310, n, k), (n, k), 1.0)
    codes, scales, stored = oracle_weight(w, 4)
    assert float(np.min(scales.astype(np.float32))) > 65504 * 2.0 ** -20
    qw = device_weight(stored, scales, 4, n, k)
    x = G.normal(G.stream_seed(1311, n, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
    y = torch.full((S, n), float("nan"), dtype=torch.float32, device="cuda")
    with gemm_path("tc"):
        from tests.helpers import to_dev_f16
        sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
        assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    assert_gemm_close(y.cpu().numpy(), verify.dequant_gemm64(x, codes, scales), k, "Y, large scales")


@pytest.mark.parametrize("S", [1, 17])
def test_int4_small_scales_take_the_two_step_form(sdv, S):
    """int4 slabs with a block scale below 2^-13 (s / 2 not exact) take the
    two-step form; both forms hold the pairs at bits 0-3 as fp16(n * s / 16),
    so the rows the two runs share agree bit for bit.  The tiny rows' own
    values carry the fp16 subnormal spacing of n * s / 16 (2^-24, i.e. 2^-20
    once the accumulator is scaled back): within the parity bound relative to
    the logits of the whole head, as the contract states it."""
    n, k = 4096, 2048
    w = G.normal(G.stream_seed(1320, n, k), (n, k), 0.02)
    small = w.copy()
    small[::32] /= 300.0  # first row of every 32-row slab: scales ~2e-5, below 2^-13
    x = G.normal(G.stream_seed(1321, n, k, S), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    drafts = np.zeros(max(S - 1, 0), np.int32)
    keep = np.ones(n, bool)
    keep[::32] = False
    out = {}
    with gemm_path("tc"):
        for name, wm in (("plain", w), ("small", small)):
            codes, scales, stored = oracle_weight(wm, 4)
            if name == "small":
                assert float(np.max(scales[::32].astype(np.float32))) < 2.0 ** -13
            head = device_weight(stored, scales, 4, n, k)
            logits, am, acc, nxt = run_head(head, x, drafts, 0)
            ref = verify.verify_head(x, codes, scales, drafts, 0)
            assert_gemm_close(logits, ref["logits"], k, f"{name} logits (whole head)")
            out[name] = logits
    np.testing.assert_array_equal(out["plain"][:, keep], out["small"][:, keep])

"""sdv_quantize_block32 on the GPU vs the oracle quantiser: bit-exact codes and
fp16 scale bits (integer outcome of fp32 arithmetic taken in the same
precision on both sides)."""
import os

import numpy as np
import pytest
import torch

from oracle import quant
from synth import generator as G
from synth import workloads as W
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


def _check(sdv, w, bits):
    qw = sdv.quantize(to_dev(w), bits)
    torch.cuda.synchronize()
    codes, scales = quant.quantize_block32(w, bits)
    stored = codes if bits == 8 else quant.pack_int4(codes)
    got = qw.codes.cpu().numpy()
    np.testing.assert_array_equal(got.view(np.uint8), stored.view(np.uint8))
    np.testing.assert_array_equal(qw.scales.cpu().numpy().view(np.uint16), scales.view(np.uint16))


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("shape", [(1, 32), (7, 96), (129, 256), (300, 2048)])
def test_random_shapes(sdv, bits, shape):
    w = G.normal(G.stream_seed(77, *shape, bits), shape, 0.02)
    _check(sdv, w, bits)


@pytest.mark.parametrize("bits", [8, 4])
def test_edge_values(sdv, bits):
    rng = np.random.default_rng(bits)
    w = (rng.standard_normal((64, 128)) * 0.02).astype(np.float32)
    w[0, :32] = 0.0                                   # zero block -> scale 0, codes 0
    w[1, :32] = np.float32(3e-6) * rng.standard_normal(32).astype(np.float32)  # subnormal fp16 scale
    w[2, 32:64] = (np.arange(32) - 16) / 2.0 * 2.0 ** -5  # exact ties
    w[3, :] = 1e4                                       # large, equal values
    w[4, 64:96] = -w[4, 64:96]
    _check(sdv, w, bits)


def test_golden_blocks(sdv):
    from tests.test_oracle_quant import _load_golden
    for blk in _load_golden():
        qw = sdv.quantize(to_dev(blk["w"][None, :].copy()), blk["bits"])
        torch.cuda.synchronize()
        assert int(qw.scales.cpu().numpy().view(np.uint16)[0, 0]) == blk["scale_bits"]
        if blk["bits"] == 8:
            np.testing.assert_array_equal(qw.codes.cpu().numpy()[0], blk["codes"])
        else:
            np.testing.assert_array_equal(qw.codes.cpu().numpy()[0], blk["packed"])


def test_full_size_head_a3b_int4(sdv):
    # the 248320 x 2048 int4 head, compared on a row sample and in full by hash
    wl = W.A3B
    w = W.head_weights(wl)
    qw = sdv.quantize(to_dev(w), 4)
    torch.cuda.synchronize()
    rows = np.r_[0:64, wl.n - 64:wl.n, np.random.default_rng(0).integers(0, wl.n, 512)]
    codes, scales = quant.quantize_block32(w[rows], 4)
    np.testing.assert_array_equal(qw.codes.cpu().numpy()[rows], quant.pack_int4(codes))
    np.testing.assert_array_equal(qw.scales.cpu().numpy()[rows].view(np.uint16), scales.view(np.uint16))

"""sdv_greedy_accept (bit-exact on a given argmax) and sdv_qlinear (fp32 Y)
on the GPU vs the oracle."""
import itertools

import numpy as np
import pytest
import torch

from oracle import verify
from synth import generator as G
from tests.helpers import assert_gemm_close, device_weight, gemm_path, oracle_weight, to_dev, to_dev_f16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


@pytest.fixture(params=["mma", "tc"])
def path(request, sdv):
    """Run the test on each GEMM implementation (mma.sync and tcgen05)."""
    with gemm_path(request.param):
        yield request.param


def test_greedy_accept_exhaustive_small(sdv):
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    for s in (1, 2, 3, 4):
        for am in itertools.product(range(2), repeat=s):
            for dr in itertools.product(range(2), repeat=max(s - 1, 1)):
                for n_valid in range(s):
                    amt = to_dev(np.array(am, np.int32))
                    drt = to_dev(np.array(dr, np.int32))
                    sdv.sdv_greedy_accept(amt, s, drt, n_valid, acc, nxt)
                    ref = verify.greedy_accept(np.array(am), np.array(dr[: s - 1]), n_valid)
                    assert (int(acc.item()), int(nxt.item())) == ref


def test_greedy_accept_random_windows(sdv):
    rng = np.random.default_rng(5)
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    for _ in range(300):
        s = int(rng.integers(1, 33))
        am = rng.integers(0, 5, s).astype(np.int32)
        dr = am[: max(s - 1, 1)].copy() if s > 1 else np.zeros(1, np.int32)
        if s > 1:
            flip = rng.integers(0, s)
            if flip < s - 1:
                dr[flip] = (dr[flip] + 1) % 5
        n_valid = int(rng.integers(0, s))
        sdv.sdv_greedy_accept(to_dev(am), s, to_dev(dr), n_valid, acc, nxt)
        assert (int(acc.item()), int(nxt.item())) == verify.greedy_accept(am, dr[: s - 1], n_valid)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("n,k,S", [(5120, 1024, 1), (5120, 1024, 9), (5120, 1024, 17), (777, 288, 5),
                                   (64, 4096, 32), (17408, 512, 17), (300, 8192, 17), (5120, 17408, 17),
                                   (100, 352, 3)])
def test_qlinear(sdv, path, bits, n, k, S):
    w = G.normal(G.stream_seed(910, n, k, bits), (n, k), 0.02)
    codes, scales, stored = oracle_weight(w, bits)
    qw = device_weight(stored, scales, bits, n, k)
    x = G.normal(G.stream_seed(911, S, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    y = torch.full((S, n), float("nan"), dtype=torch.float32, device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
    sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
    assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    assert_gemm_close(y.cpu().numpy(), verify.dequant_gemm(x, codes, scales), k, "Y")


def test_qlinear_integer_case_exact(sdv, path):
    # unit scales, small integer activations: the result is an exact integer GEMM
    n, k, S = 300, 512, 9
    rng = np.random.default_rng(1)
    codes = rng.integers(-127, 128, (n, k)).astype(np.int8)
    scales = np.ones((n, k // 32), np.float16)
    x = rng.integers(-4, 5, (S, k)).astype(np.float16)
    qw = device_weight(codes, scales, 8, n, k)
    y = torch.empty((S, n), dtype=torch.float32, device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
    sdv.sdv_qlinear(qw, to_dev_f16(x), S, y, ws)
    exact = x.astype(np.int64) @ codes.astype(np.int64).T
    np.testing.assert_array_equal(y.cpu().numpy(), exact.astype(np.float32))

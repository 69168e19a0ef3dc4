"""sdv_qlinear_swiglu (fp16 h), sdv_moe_route and sdv_moe_gather_qmm on the GPU
vs the oracle.

SwiGLU bound.  The GPU's g and u each carry the GEMM error allowed for a
reduction of length k (at most tol(k) * RMS, see tests.helpers), and h is then
rounded to fp16.  Propagating those through h = SiLU(g) * u gives, per element,
    |dh| <= |SiLU'(g)| |u| eg + (|SiLU(g)| + 1.1 eg) eu + eg^2 |u| / 2 + ulp16(h) / 2
with eg = tol(k) RMS(g), eu = tol(k) RMS(u), |SiLU'| <= 1.1 and |SiLU''| <= 1/2.
MoE: rel-L2(out) <= 1e-3 over the whole [S, H] output; routing ids and the
grouping are integers and bit-exact.
"""
import numpy as np
import pytest
import torch

from oracle import mlp, verify
from synth import generator as G
from tests.helpers import assert_gemm_close, device_weight, gemm_path, oracle_weight, to_dev, to_dev_f16, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decode_verify_sdv_gb300 import build, sdv as _sdv
    build.build()
    _sdv.load()
    return _sdv


@pytest.fixture(params=["mma", "tc"])
def path(request, sdv):
    with gemm_path(request.param):
        yield request.param


def _dsilu(t):
    sg = 1.0 / (1.0 + np.exp(-t))
    return sg * (1.0 + t * (1.0 - sg))


def assert_swiglu_close(h_gpu, g64, u64, k, what="h"):
    h64 = mlp.silu(g64) * u64
    eg = tol(k) * float(np.sqrt(np.mean(g64 ** 2)))
    eu = tol(k) * float(np.sqrt(np.mean(u64 ** 2)))
    ulp = np.spacing(np.abs(h64).astype(np.float16)).astype(np.float64)
    bound = (np.abs(_dsilu(g64)) * np.abs(u64) * eg + (np.abs(mlp.silu(g64)) + 1.1 * eg) * eu
             + 0.5 * eg * eg * np.abs(u64) + 0.5 * ulp + 1e-30)
    err = np.abs(np.asarray(h_gpu, dtype=np.float64) - h64)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} beyond the bound; worst "
                           f"err {err[bad].max():.3e} vs bound {bound[bad][np.argmax(err[bad])]:.3e}")


def _run_swiglu(sdv, gate, up, x):
    S = x.shape[0]
    h = torch.full((S, gate.n), float("nan"), dtype=torch.float16, device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_QLINEAR_SWIGLU, gate.n, gate.k, S)
    sdv.sdv_qlinear_swiglu(gate, up, to_dev_f16(x), S, h, ws)
    assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    return h.cpu().numpy().astype(np.float64)


def _swiglu_case(sdv, bits, n, k, S, seed):
    wg = G.normal(G.stream_seed(700, seed, 1), (n, k), 0.02)
    wu = G.normal(G.stream_seed(700, seed, 2), (n, k), 0.02)
    x = G.normal(G.stream_seed(700, seed, 3), (S, k), 1.0, dtype=np.float64).astype(np.float16)
    cg, sg, stg = oracle_weight(wg, bits)
    cu, su, stu = oracle_weight(wu, bits)
    gate = device_weight(stg, sg, bits, n, k)
    up = device_weight(stu, su, bits, n, k)
    h = _run_swiglu(sdv, gate, up, x)
    g64 = verify.dequant_gemm64(x, cg, sg)
    u64 = verify.dequant_gemm64(x, cu, su)
    assert_swiglu_close(h, g64, u64, k, f"swiglu bits={bits} n={n} k={k} S={S}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("n,k,S", [(256, 256, 1), (384, 512, 9), (200, 512, 17), (130, 768, 32),
                                   (256, 96, 5), (1000, 1024, 16)])
def test_swiglu_shapes(sdv, path, bits, n, k, S):
    _swiglu_case(sdv, bits, n, k, S, seed=n * 7 + k + S + bits)


@pytest.mark.parametrize("op", ["swiglu", "qlinear"])
def test_split_k_repeated_calls_one_workspace(sdv, op):
    """Split-K plans (the partials in the workspace, then the reduce): three
    consecutive calls on one workspace each write every output again (outputs
    refilled with NaN between calls) and match the oracle."""
    n, k, S = (1024, 5120, 17) if op == "swiglu" else (640, 17408, 17)
    w = [G.normal(G.stream_seed(730, m, n, k), (n, k), 0.02) for m in range(2)]
    q = [oracle_weight(wm, 8) for wm in w]
    dw = [device_weight(st, sc, 8, n, k) for _, sc, st in q]
    with gemm_path("tc"):
        if op == "swiglu":
            ws = sdv.workspace(sdv.SDV_OP_QLINEAR_SWIGLU, n, k, S)
            out = torch.empty((S, n), dtype=torch.float16, device="cuda")
        else:
            ws = sdv.workspace(sdv.SDV_OP_QLINEAR, n, k, S)
            out = torch.empty((S, n), dtype=torch.float32, device="cuda")
        for call in range(3):
            x = G.normal(G.stream_seed(731, call, n, k), (S, k), 1.0, dtype=np.float64).astype(np.float16)
            out.fill_(float("nan"))
            if op == "swiglu":
                sdv.sdv_qlinear_swiglu(dw[0], dw[1], to_dev_f16(x), S, out, ws)
            else:
                sdv.sdv_qlinear(dw[0], to_dev_f16(x), S, out, ws)
            assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
            got = out.cpu().numpy().astype(np.float64)
            g64 = verify.dequant_gemm64(x, q[0][0], q[0][1])
            if op == "swiglu":
                assert_swiglu_close(got, g64, verify.dequant_gemm64(x, q[1][0], q[1][1]), k, f"h, call {call}")
            else:
                assert_gemm_close(got, g64, k, f"y, call {call}")


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("n,k,S", [(3000, 3328, 9), (5000, 4352, 17), (7000, 4352, 9), (3000, 5376, 17)])
def test_swiglu_uneven_splits_ragged_rows(sdv, path, bits, n, k, S):
    """Split gate/up plans whose last reduction split is shorter than the others,
    whose tiles do not divide evenly over the CTAs, and whose last tile of rows
    is ragged."""
    _swiglu_case(sdv, bits, n, k, S, seed=n + k + S + bits)


def test_swiglu_integer_exact(sdv, path):
    """Scales 1 and small integer x: g and u are exact integers on both sides,
    so h differs from the oracle's fp16 at most by the last-bit of an fp32
    SiLU evaluation (one fp16 ulp)."""
    rng = np.random.default_rng(11)
    n, k, S = 256, 512, 9
    cg = rng.integers(-3, 4, (n, k)).astype(np.int8)
    cu = rng.integers(-3, 4, (n, k)).astype(np.int8)
    sc = np.full((n, k // 32), 1.0, dtype=np.float16)
    x = rng.integers(-2, 3, (S, k)).astype(np.float16)
    gate = device_weight(cg, sc, 8, n, k)
    up = device_weight(cu, sc, 8, n, k)
    h = _run_swiglu(sdv, gate, up, x)
    ref = mlp.qlinear_swiglu(x, cg, sc, cu, sc).astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    assert (np.abs(h - ref) <= ulp + 1e-30).all()


# ---------------------------------------------------------------- MoE ----

def _route_dev(sdv, logits, top_k):
    S, E = logits.shape
    ids = torch.full((S, top_k), -1, dtype=torch.int32, device="cuda")
    wts = torch.full((S, top_k), float("nan"), dtype=torch.float32, device="cuda")
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    rows = torch.full((S * top_k,), -1, dtype=torch.int32, device="cuda")
    nh = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    hit = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    sdv.sdv_moe_route(to_dev(np.ascontiguousarray(logits, np.float32)), S, E, top_k, ids, wts, offs, rows, nh, hit)
    torch.cuda.synchronize()
    n_hit = int(nh.item())
    return (ids.cpu().numpy(), wts.cpu().numpy(), offs.cpu().numpy(), rows.cpu().numpy(), n_hit,
            hit.cpu().numpy()[:n_hit])


def _check_route(sdv, logits, top_k):
    ids, wts, offs, rows, n_hit, hit = _route_dev(sdv, logits, top_k)
    rid, rw = mlp.route_topk(logits, top_k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(wts, rw, rtol=2e-6, atol=1e-7)
    roffs, rrows, _ = mlp.group_by_expert(rid, logits.shape[1])
    np.testing.assert_array_equal(offs, roffs)
    np.testing.assert_array_equal(rows, rrows)
    uniq = np.unique(rid)
    assert n_hit == len(uniq)
    np.testing.assert_array_equal(hit, uniq)


@pytest.mark.parametrize("S,E,top_k", [(1, 8, 1), (9, 8, 2), (17, 256, 8), (32, 256, 8), (5, 1000, 3),
                                       (17, 64, 32)])
def test_moe_route_random(sdv, S, E, top_k):
    logits = G.normal(G.stream_seed(710, S, E, top_k), (S, E), 1.0, dtype=np.float32)
    _check_route(sdv, logits, top_k)


def test_moe_route_ties(sdv):
    """Many equal logits: ties go to the lower expert id."""
    rng = np.random.default_rng(3)
    for E, top_k in ((16, 4), (256, 8), (33, 8)):
        logits = rng.integers(0, 3, (17, E)).astype(np.float32)
        _check_route(sdv, logits, top_k)


def _moe_tensors(sdv, rng_seed, E, I, H, bits, same_experts=False):
    out = {}
    for tid, (t, (rows, cols)) in enumerate((("gate", (E * I, H)), ("up", (E * I, H)), ("down", (E * H, I)))):
        if same_experts:
            one = G.normal(G.stream_seed(720, rng_seed, tid), (rows // E, cols), 0.02)
            w = np.tile(one, (E, 1))
        else:
            w = G.normal(G.stream_seed(720, rng_seed, tid), (rows, cols), 0.02)
        codes, scales, stored = oracle_weight(w, bits)
        out[t] = ((codes, scales), device_weight(stored, scales, bits, rows, cols))
    return out


def _run_moe(sdv, T, E, I, H, top_k, x, logits):
    S = x.shape[0]
    out = torch.full((S, H), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((S, top_k), -1, dtype=torch.int32, device="cuda")
    wts = torch.full((S, top_k), float("nan"), dtype=torch.float32, device="cuda")
    ws = sdv.workspace(sdv.SDV_OP_MOE, I, H, S, E, top_k)
    sdv.sdv_moe_gather_qmm(T["gate"][1], T["up"][1], T["down"][1], E, I, H, top_k, to_dev_f16(x),
                           to_dev(np.ascontiguousarray(logits, np.float32)), S, out, ids, wts, ws)
    assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    return out.cpu().numpy(), ids.cpu().numpy(), wts.cpu().numpy()


def _rel_l2(a, b):
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / max(np.linalg.norm(b), 1e-300))


def _moe_case(sdv, bits, S, E, I, H, top_k, seed, same_experts=False, logits=None):
    T = _moe_tensors(sdv, seed, E, I, H, bits, same_experts)
    x = G.normal(G.stream_seed(721, seed, S), (S, H), 1.0, dtype=np.float64).astype(np.float16)
    if logits is None:
        logits = G.normal(G.stream_seed(722, seed, S), (S, E), 1.0, dtype=np.float32)
    out, ids, wts = _run_moe(sdv, T, E, I, H, top_k, x, logits)
    ref, rid, rw = mlp.moe_forward(x, logits, T["gate"][0], T["up"][0], T["down"][0], E, I, H, top_k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(wts, rw, rtol=2e-6, atol=1e-7)
    r = _rel_l2(out, ref)
    assert r <= 1e-3, f"MoE rel-L2 {r:.3e}"
    return out, ref


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("S,E,I,H,top_k", [(1, 8, 256, 256, 2), (5, 8, 256, 512, 2), (17, 16, 512, 256, 4),
                                           (17, 32, 256, 512, 8), (32, 12, 256, 256, 3)])
def test_moe_shapes(sdv, bits, S, E, I, H, top_k):
    _moe_case(sdv, bits, S, E, I, H, top_k, seed=S * 31 + E + I + H + top_k + bits)


def test_moe_top1_dominant_expert(sdv):
    """top_k = 1: each row's output is its one expert's SwiGLU MLP."""
    E, I, H, S = 8, 256, 256, 9
    logits = np.full((S, E), -4.0, dtype=np.float32)
    logits[np.arange(S), np.arange(S) % E] = 5.0
    _moe_case(sdv, 4, S, E, I, H, 1, seed=901, logits=logits)


def test_moe_identical_experts(sdv):
    """All experts equal: the weights sum to one, so out equals one expert's MLP."""
    E, I, H, S, top_k = 8, 256, 256, 5, 4
    out, _ = _moe_case(sdv, 4, S, E, I, H, top_k, seed=902, same_experts=True)
    T = _moe_tensors(sdv, 902, E, I, H, 4, same_experts=True)
    x = G.normal(G.stream_seed(721, 902, S), (S, H), 1.0, dtype=np.float64).astype(np.float16)
    one = mlp.expert_swiglu64(x, 0, I, H, T["gate"][0], T["up"][0], T["down"][0])
    assert _rel_l2(out, one) <= 1e-3


def test_moe_prologue_routing_matches_router(sdv):
    """Up to 256 experts and 8 picks the gate/up launch routes the window in its
    own prologue: its picks and weights (the call's top-k outputs) equal the
    routing kernel's bit for bit, on logits full of ties."""
    E, I, H, S, top_k = 256, 256, 256, 17, 8
    rng = np.random.default_rng(11)
    logits = rng.integers(0, 3, (S, E)).astype(np.float32)
    T = _moe_tensors(sdv, 903, E, I, H, 4)
    x = G.normal(G.stream_seed(721, 903, S), (S, H), 1.0, dtype=np.float64).astype(np.float16)
    out, ids, wts = _run_moe(sdv, T, E, I, H, top_k, x, logits)
    rids, rwts = _route_dev(sdv, logits, top_k)[:2]
    np.testing.assert_array_equal(ids, rids)
    np.testing.assert_array_equal(wts, rwts)
    ref = mlp.moe_forward(x, logits, T["gate"][0], T["up"][0], T["down"][0], E, I, H, top_k)[0]
    assert _rel_l2(out, ref) <= 1e-3


@pytest.mark.parametrize("E,top_k", [(320, 4), (64, 12)])
def test_moe_routing_launch_beyond_prologue_limits(sdv, E, top_k):
    """More than 256 experts or 8 picks: the routing launch runs first and the
    gate/up launch reads its hit list."""
    _moe_case(sdv, 4, 9, E, 256, 256, top_k, seed=904 + E + top_k)

"""Launch plans of the C ABI, checked on the CPU (no GPU).

libsdv's host code is linked against a stand-in CUDA runtime
(``tests/launch_trace``) that answers device queries for a GB300 (152 SMs,
232448 bytes of opt-in shared memory per block) and records every kernel
launch, tensor map and copy.  The tests check:

* the plans the committed ncu summaries were taken on (``profiles/``): grid,
  block, ring depth, split-K and row chunking of the timed workloads;
* hardware limits over a sweep of shapes, window sizes, weight types and GEMM
  paths: shared memory within the opt-in limit, one wave of tcgen05 CTAs, rings
  of at least four stages, 16-byte TMA rows, strides and boxes;
* the routing rules between the two GEMM implementations and the errors the
  host returns before any launch.
"""
import os
import re
import shutil
import sys

import pytest

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "launch_trace"))
import build_trace  # noqa: E402

SMS, SMEM = 152, 232448
OK, UNSUPPORTED = 0, 2


@pytest.fixture(scope="module")
def tracer():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    return build_trace.build()


def trace(tracer, *cmds, sms=SMS, smem=SMEM, path=0):
    calls = build_trace.run(tracer, [f"device {sms} {smem}", f"path {path}", *cmds])
    return calls[2:]


def tc_args(launch):
    """(weight type, mode, MMA N) of a tcgen05 GEMM launch, else None."""
    m = re.search(r"tc_gemm_kernelILi(\d+)ELi(\d+)ELi(\d+)E", launch.get("name", ""))
    return tuple(int(g) for g in m.groups()) if m else None


def grid(launch):
    x, y = launch["grid"].split(",")
    return int(x), int(y)


# ---- the plans of the profiled workloads ---------------------------------------------

def test_q4b_head_plan(tracer):
    # profiles/tc_gemm_verify_head_q4b.md: 152 CTAs x 448 threads, ring depth 4
    (c,) = trace(tracer, "head 8 151936 2560 9 8 0")
    assert c["status"] == OK and len(c["launches"]) == 1
    (l,) = c["launches"]
    assert tc_args(l) == (8, 1, 16)
    assert grid(l) == (152, 1) and l["block"] == "448" and l["depth"] == "4" and l["splits"] == "1"
    # codes as 128-byte x 128-row boxes (128-byte swizzle), scales by TMA (k % 256 == 0)
    codes, scales = c["tmaps"]
    assert codes["box"] == "128,128" and codes["swizzle"] == "3" and codes["dims"] == "2560,151936"
    assert scales["box"] == "8,128" and l["scales_tma"] == "1"


def test_q4b_sampling_plan(tracer):
    # profiles/tc_gemm_verify_sample_q4b.md: 152 CTAs x 448 threads, ring depth 4
    (c,) = trace(tracer, "sample 8 151936 2560 9 8")
    (l,) = c["launches"]
    assert c["status"] == OK and tc_args(l) == (8, 2, 16)
    assert grid(l) == (152, 1) and l["block"] == "448" and l["depth"] == "4"


@pytest.mark.parametrize("qt", [4, 2])
def test_a3b_head_plan(tracer, qt):
    # profiles/tc_gemm_verify_head_a3b_s17.md and ..._fp4_a3b_s17.md:
    # 152 CTAs x 576 threads (three converter groups), ring depth 6
    (c,) = trace(tracer, f"head {qt} 248320 2048 17 16 0")
    (l,) = c["launches"]
    assert c["status"] == OK and tc_args(l) == (qt, 1, 32)
    assert grid(l) == (152, 1) and l["block"] == "576" and l["depth"] == "6"


def test_mlp27_plans(tracer):
    # profiles/tc_gemm_mlp27_s17.md: gate/up 4 splits x 38 CTAs + SwiGLU reduce,
    # down 14 splits x 10 CTAs + split-K sum
    sw, dn = trace(tracer, "swiglu 8 17408 5120 17", "qlinear 8 5120 17408 17")
    assert [grid(l) for l in sw["launches"][:1]] == [(38, 4)] and "swiglu_reduce" in sw["launches"][1]["name"]
    assert sw["launches"][0]["dual"] == "1"
    assert [grid(l) for l in dn["launches"][:1]] == [(10, 14)] and "splitk_reduce" in dn["launches"][1]["name"]
    assert dn["launches"][0]["k_chunk"] == "1280"


def test_launch_counter_counts_every_launch(tracer):
    # sdv_launch_count (the bench's gpu_launches) against the launches the
    # stand-in runtime records, over calls that use every launch site
    cmds = ["count", "head 8 151936 2560 9 8 0", "head 8 151936 2560 17 16 0", "sample 8 151936 2560 9 8",
            "qlinear 8 5120 17408 17", "swiglu 8 17408 5120 17", "swiglu 8 17408 5120 1",
            "moe 4 256 512 2048 8 17", "noalloc 8 151936 2560 17 16"]
    calls = build_trace.run(tracer, [f"device {SMS} {SMEM}", "path 0", *cmds, "path 1", "qlinear 8 5120 17408 17",
                                     "swiglu 8 17408 5120 17", "count"])
    counts = [int(c["other"][0].split("=")[1]) for c in calls if c["cmd"] == "count"]
    launched = sum(len(c["launches"]) for c in calls if c["cmd"] != "count")
    assert len(counts) == 2 and counts[1] - counts[0] == launched and launched > 10


def test_moe_plan(tracer):
    # gate/up over the hit list with the SwiGLU epilogue, routing the window in
    # its own prologue (no routing launch), down over 38 expert-segment slots x 4
    # CTAs reading the hit list gate/up's CTA 0 wrote, split sum
    (c,) = trace(tracer, "moe 4 256 512 2048 8 17")
    gu, dn, red = c["launches"]
    assert tc_args(gu) == (4, 0, 32) and grid(gu) == (152, 1) and gu["dual"] == "2"
    assert gu["rows_per_expert"] == "512" and gu["seg_k"] == "0"
    assert gu["route"] == "1" and gu["route_E"] == "256" and gu["route_top_k"] == "8" and gu["listed"] == "0"
    assert tc_args(dn) == (4, 0, 32) and grid(dn) == (4, 38) and dn["seg_k"] == "512"
    assert dn["route"] == "0" and dn["listed"] == "1"
    assert "splitk_reduce" in red["name"]


def test_moe_plan_beyond_prologue_routing(tracer):
    # more experts or picks than the prologue routing takes: the routing launch
    # (one block) runs first and gate/up reads the hit list it wrote
    (c,) = trace(tracer, "moe 4 1024 256 256 32 9")
    route, gu = c["launches"][:2]
    assert "moe_route_kernel" in route["name"] and grid(route) == (1, 1) and route["block"] == "1024"
    assert tc_args(gu) == (4, 0, 16) and gu["route"] == "0" and gu["listed"] == "1"


def test_q4b_head_beyond_one_launch_splits_the_reduction(tracer):
    # int8, k = 2560: S = 17 window rows leave no room for a 4-stage ring next to
    # them; with a full workspace each CTA takes part of the reduction (one pass
    # over the head writing partial logits), then the split-sum tail
    (c,) = trace(tracer, "head 8 151936 2560 17 16 0")
    assert c["status"] == OK and len(c["launches"]) == 2
    gemm, tail = c["launches"]
    assert tc_args(gemm) == (8, 0, 32) and int(gemm["splits"]) >= 2 and gemm["S"] == "17"
    assert int(gemm["k_chunk"]) * (int(gemm["splits"]) - 1) < 2560 <= int(gemm["k_chunk"]) * int(gemm["splits"])
    assert "head_splitsum_kernel" in tail["name"] and int(tail["grid"].split(",")[0]) <= 2 * SMS


def test_q4b_head_beyond_one_launch_without_room_is_row_chunked(tracer):
    # the same window through the fixed scratch of the no-workspace head, which
    # cannot hold partial logits: row chunks on the tcgen05 path, then one accept
    (c,) = trace(tracer, "noalloc 8 151936 2560 17 16")
    gemms = [l for l in c["launches"] if tc_args(l)]
    assert c["status"] == OK and [int(l["S"]) for l in gemms] == [9, 8]
    assert all(l["n_valid"] == "0" for l in gemms)
    assert c["launches"][-1]["kind"] == "chevron" and c["launches"][-1]["block"] == "32"  # the accept


# ---- limits over a sweep ---------------------------------------------------------------

SHAPES = [(4096, 256), (151936, 2560), (248320, 2048), (3001, 800), (1000, 288), (4097, 2048), (17408, 5120),
          (5120, 17408), (64, 64), (1, 32)]
WINDOWS = [1, 2, 8, 9, 16, 17, 24, 32]


def _check_limits(c, sms, smem):
    for l in c["launches"]:
        assert int(l["smem"]) <= smem, (c["cmd"], l)
        args = tc_args(l)
        if args:
            gx, gy = grid(l)
            assert gx * gy <= sms, ("more than one wave", c["cmd"], l)
            assert int(l["depth"]) >= 4, (c["cmd"], l)
            assert l["block"] == ("448" if args[0] == 8 else "576"), (c["cmd"], l)
            assert int(l["smem"]) > smem // 2, ("one CTA per SM", c["cmd"], l)
    for t in c["tmaps"]:
        inner, rows = (int(v) for v in t["box"].split(","))
        elem = 1 if t["dtype"] == "0" else 2
        assert (inner * elem) % 16 == 0 and int(t["stride"]) % 16 == 0, (c["cmd"], t)
        assert rows <= 256 and inner <= 256, (c["cmd"], t)


@pytest.mark.parametrize("sms,smem", [(152, 232448), (148, 232448)])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_limits_over_a_sweep(tracer, sms, smem, path):
    cmds = []
    for n, k in SHAPES:
        for qt in (8, 4, 2):
            for S in WINDOWS:
                cmds += [f"head {qt} {n} {k} {S} {S - 1} 1", f"sample {qt} {n} {k} {S} {S - 1}",
                         f"qlinear {qt} {n} {k} {S}", f"swiglu {qt} {n} {k} {S}"]
    for E, I, H, top_k in [(256, 512, 2048, 8), (64, 256, 512, 4), (1024, 256, 256, 32)]:
        for qt in (8, 4, 2):
            for S in (1, 9, 17, 32):
                cmds.append(f"moe {qt} {E} {I} {H} {top_k} {S}")
    calls = trace(tracer, *cmds, sms=sms, smem=smem, path=path)
    assert len(calls) == len(cmds)
    n_ok = 0
    for c in calls:
        assert c["status"] in (OK, UNSUPPORTED), c
        if c["status"] == UNSUPPORTED:
            assert not c["launches"], ("no launch before an unsupported answer", c["cmd"])
            continue
        n_ok += 1
        _check_limits(c, sms, smem)
        op, qt = c["cmd"].split()[:2]
        if path == 1 and op in ("head", "qlinear"):
            assert not any(tc_args(l) for l in c["launches"]), c["cmd"]
        if path == 2 or op in ("sample", "moe") or qt == "2":
            assert not any(l["kind"] == "chevron" and l["block"] == "128" for l in c["launches"]), c["cmd"]
    assert n_ok > len(cmds) // 3


def test_fp4_and_sampling_stay_off_the_mma_path(tracer):
    calls = trace(tracer, "head 2 4096 256 9 8 0", "qlinear 2 4096 256 9", "sample 8 4096 256 9 8",
                  "head 8 4096 256 9 8 0", path=1)
    assert [c["status"] for c in calls] == [UNSUPPORTED, UNSUPPORTED, UNSUPPORTED, OK]
    assert not calls[0]["launches"] and not calls[2]["launches"]
    assert calls[3]["launches"] and not any(tc_args(l) for l in calls[3]["launches"])


def test_head_workspace_layout(tracer):
    # workspace = 256-byte header + [grid][S] fp32 maxima + [grid][S] int32 indices
    (ws,) = trace(tracer, "ws 3 151936 2560 9 0 0")
    assert ws["other"] == [f"ws bytes={256 + SMS * 9 * 8}"]
    (c,) = trace(tracer, "head 8 151936 2560 9 8 0")
    (l,) = c["launches"]
    assert int(l["part_v"], 16) == 0x100  # right behind the header (workspace at offset 0)

"""Host logic of bench.py (CPU only): the algorithmic byte counts behind the
roofline, the committed DRAM-traffic summaries it reads, the clock-record
summary, the peak lookup, and the order the end-to-end loop imposes on its
copies and calls."""
import dataclasses
import os

import pytest

import bench
from synth import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_head_bytes_by_hand():
    # q4b, S = 9: int8 codes 151936 x 2560, fp16 scales 151936 x 80, fp16 x 9 x 2560,
    # 8 drafts, 9 argmax, accepted + next_a0
    want = 151936 * 2560 + 151936 * 80 * 2 + 9 * 2560 * 2 + 8 * 4 + 9 * 4 + 8
    assert bench.head_bytes(W.Q4B, 9) == want == 413312076
    # int4 and FP4 codes are two per byte
    assert bench.head_bytes(W.A3B, 1) == 248320 * 1024 + 248320 * 64 * 2 + 2048 * 2 + 4 + 8
    fp4 = dataclasses.replace(W.A3B, bits=2)
    assert bench.head_bytes(fp4, 17) == bench.head_bytes(W.A3B, 17)


def test_weight_and_layer_bytes():
    assert bench.weight_bytes(64, 256, 8) == 64 * 256 + 64 * 8 * 2
    assert bench.weight_bytes(64, 256, 4) == 64 * 128 + 64 * 8 * 2
    # head bytes = its weight + the window's own I/O
    S = 17
    assert bench.head_bytes(W.A3B, S) - bench.weight_bytes(W.A3B.n, W.A3B.h, 4) == S * 2048 * 2 + 16 * 4 + S * 4 + 8
    wl = W.MLP27
    three = 2 * bench.weight_bytes(17408, 5120, 8) + bench.weight_bytes(5120, 17408, 8)
    assert bench.mlp_bytes(wl, 1) == three + 5120 * 2 + 2 * 17408 * 2 + 5120 * 4
    m = W.MOE
    assert bench.moe_expert_bytes(m) == 3 * bench.weight_bytes(512, 2048, 4)
    assert bench.moe_bytes(m, 17, 0) == 17 * 2048 * 2 + 17 * 256 * 4 + 17 * 2048 * 4


@pytest.mark.parametrize("key,wl,S", [("q4b S=9", W.Q4B, 9), ("a3b S=17", W.A3B, 17),
                                      ("q4b S=9 sample", W.Q4B, 9),
                                      ("a3b S=17 fp4", dataclasses.replace(W.A3B, bits=2), 17)])
def test_committed_traffic_is_near_the_algorithmic_bytes(key, wl, S):
    # a committed summary for each head workload; its DRAM bytes per launch sit just
    # above the algorithmic bytes (no wasted re-reads) and never below the weight stream
    traffic, src = bench.profiled_traffic(key)
    if traffic is None:
        assert src is None or "stale" in src, src
        pytest.skip(f"no current summary for {key}: {src}")
    alg = bench.head_bytes(wl, S)
    assert bench.weight_bytes(wl.n, wl.h, wl.bits) <= traffic <= 1.05 * alg, (key, traffic, alg)


def _fake_root(tmp_path, hash_line):
    csrc = tmp_path / "speculative_decode_verify_sdv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        (csrc / f).write_text(f"// {f}\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "a_other.md").write_text("workload: other S=1\ntraffic_bytes_per_launch: 5\n")
    (prof / "b_head.md").write_text(f"# title\n\n{hash_line}\nworkload: q4b S=9\n"
                                    "traffic_bytes_per_launch: 123456\n")


def test_profiled_traffic_reads_current_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_root(tmp_path, "kernel_source_sha256: PLACEHOLDER")
    cur = bench.kernel_source_hash()
    p = tmp_path / "profiles" / "b_head.md"
    p.write_text(p.read_text().replace("PLACEHOLDER", cur))
    assert bench.profiled_traffic("q4b S=9") == (123456.0, "profiles/b_head.md")
    assert bench.profiled_traffic("q4b S=9 sample") == (None, None)


def test_profiled_traffic_is_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_root(tmp_path, "kernel_source_sha256: 0000000000000000")
    traffic, src = bench.profiled_traffic("q4b S=9")
    assert traffic is None and "stale" in src


def test_clock_summary():
    cs = bench.ClockSampler(0)
    cs.kind = "nvidia-smi"
    for line in (
        "0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2010, 2070, 950.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 930.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ):
        cs._add_smi(line)
    s = cs.summary()
    assert s["sm_mhz"] == 1980.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    cs = bench.ClockSampler(0)
    cs._add_smi("0, 1900, 2070, 1.0, 0x0, Active, Not Active, Not Active, Not Active")
    assert cs.summary()["reasons"] == ["hw_slowdown"]
    cs = bench.ClockSampler(0)
    assert cs.summary()["reasons"] == ["unsampled"]


def test_clock_summary_nvml_phases():
    """NVML readings: the median is taken over the readings during the timed
    region; the readings before and after are kept, and reason bits map to names."""
    cs = bench.ClockSampler(0)
    cs.kind = "nvml"
    cs._add_nvml("1.0,1200,2070,200000,0")        # before: idle clock
    cs.phase = "during"
    for sm in (2070, 2055, 2070):
        cs._add_nvml(f"1.1,{sm},2070,900000,0")
    cs._add_nvml("1.2,2040,2070,950000,4")         # sw_power_cap bit
    cs.phase = "after"
    cs._add_nvml("1.3,2070,2070,800000,0")
    s = cs.summary()
    assert s["sm_mhz"] == 2062.5 and s["samples"] == 6 and s["samples_during"] == 4
    assert s["reasons"] == ["sw_power_cap"] and s["sm_mhz_before_after"] == [1200.0, 2070.0]
    cs._add_nvml("1.4,1000,2070,0,72")             # 8 | 64: hw_slowdown, hw_thermal_slowdown
    assert cs.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]


def test_measured_peak(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6783.1, "bf16_tflops": 2000}')
    assert bench.measured_peak() == (6783.1, "measured")


def test_workload_names():
    assert bench.workload_name(W.Q4B, 9) == "q4b: verify head 151936x2560 int8 per-block-32, S=9"
    assert "fp4 (E2M1)" in bench.workload_name(dataclasses.replace(W.A3B, bits=2), 17)
    assert bench.workload_name(W.MOE, 17).startswith("moe: MoE 256 experts")


def test_oracle_threads_is_positive():
    assert bench.oracle_threads() >= 1


def _args(**kw):
    base = dict(also="auto", config="q4b", fp4=False, verify="greedy", path="auto")
    base.update(kw)
    return bench.argparse.Namespace(**base)


def test_also_measured_defaults_to_the_other_workloads():
    # the default single-GPU run also times the int4 head (S = 17 and 1), the
    # dense MLP stack, the MoE layer and the L2-resident tiny head; any other run
    # measures only its own line
    got = [(wl.name, S) for wl, S in bench.also_specs(_args(), 1)]
    assert got == [("a3b", 17), ("a3b", 1), ("mlp27", 17), ("moe", 17), ("tiny", 9)]
    assert bench.also_specs(_args(), 2) == []
    assert bench.also_specs(_args(config="a3b"), 1) == []
    assert bench.also_specs(_args(fp4=True), 1) == []
    assert bench.also_specs(_args(verify="sample"), 1) == []
    assert bench.also_specs(_args(also="none"), 1) == []
    assert [(wl.name, S) for wl, S in bench.also_specs(_args(also="mlp27:9, a3b"), 1)] == [("mlp27", 9), ("a3b", 17)]
    with pytest.raises(SystemExit):
        bench.also_specs(_args(also="nosuch:3"), 1)


def test_l2_label_separates_l2_warm_from_hbm():
    # the tiny head's 1.12 MB fits the 129 MB L2: its numbers are labelled
    # L2-warm, never HBM; the full-size weight streams are larger than L2
    assert bench.l2_label(1.12e6).startswith("L2-warm")
    assert bench.l2_label(286e6).startswith("inputs larger than L2")


# ---- the end-to-end loop's stream ordering, on a model of streams and events ----

class _Op:
    def __init__(self, kind, stream, **kw):
        self.kind, self.stream, self.deps, self.kw = kind, stream, set(), kw


class _FakeCuda:
    """Streams as ordered op lists and events as 'the op recorded last', enough
    to decide what the device may run before what: an op follows the previous
    op of its stream and every event record its stream waited for."""

    def __init__(self):
        self.ops = []
        self.main = self.Stream()
        self.cur = self.main

    def _add(self, kind, stream=None, **kw):
        s = stream or self.cur
        op = _Op(kind, s, **kw)
        if s.last is not None:
            op.deps.add(s.last)
        op.deps |= s.pending
        s.pending = set()
        s.last = op
        self.ops.append(op)
        return op

    def Stream(self, device=None):
        class S:
            last, device = None, "cuda:0"

            def __init__(s):
                s.pending = set()

            def wait_event(s, ev):
                if ev.op is not None:
                    s.pending.add(ev.op)

            def wait_stream(s, other):
                if other.last is not None:
                    s.pending.add(other.last)
        return S()

    def Event(self, enable_timing=False):
        cuda = self

        class E:
            op = None

            def record(e, stream=None):
                e.op = cuda._add("record", stream)

            def elapsed_time(e, other):
                return 1.0
        return E()

    def current_stream(self):
        return self.cur

    def stream(self, s):
        cuda = self

        class Ctx:
            def __enter__(c):
                c.prev, cuda.cur = cuda.cur, s

            def __exit__(c, *a):
                cuda.cur = c.prev
        return Ctx()

    def synchronize(self):
        self._add("sync", self.main)
        for s in {op.stream for op in self.ops}:
            s.pending = set()


class _FakeTorch:
    def __init__(self):
        self.cuda = _FakeCuda()


class _Slot:
    def __init__(self, cuda, kind, idx):
        self.cuda, self.kind, self.idx = cuda, kind, idx

    def copy_(self, src, non_blocking=False):
        if self.kind == "in":      # H2D into device record idx
            self.cuda._add("h2d", slot=self.idx, win=src.idx)
        else:                      # D2H into host row idx from device record src
            self.cuda._add("d2h", slot=src.idx, win=self.idx)


class _FakeJob:
    def __init__(self, cuda, slots, nwin):
        self.cuda, self.nwin = cuda, nwin
        self.e2e_in = [_Slot(cuda, "in", r) for r in range(slots)]
        self.e2e_out = [_Slot(cuda, "dev", r) for r in range(slots)]
        self.in_rows = [_Slot(cuda, "host", j) for j in range(nwin)]
        self.out_rows = [_Slot(cuda, "out", j) for j in range(nwin)]

    def e2e_call(self, r, i):
        self.cuda._add("call", slot=r, step=i)


def _before(a, b):
    """Whether op a must finish before op b may start."""
    seen, todo = set(), [b]
    while todo:
        op = todo.pop()
        for d in op.deps:
            if d is a:
                return True
            if id(d) not in seen:
                seen.add(id(d))
                todo.append(d)
    return False


@pytest.mark.parametrize("overlap", [True, False])
def test_e2e_region_orders_copies_and_calls(overlap):
    torch = _FakeTorch()
    cuda = torch.cuda
    steps, warmup, nwin = 11, 3, 4
    job = _FakeJob(cuda, bench.E2E_SLOTS, nwin)
    assert bench.e2e_region(job, steps, warmup, 1, torch, overlap) == 1.0
    # the timed steps: the ops after the last synchronize
    last_sync = max(i for i, op in enumerate(cuda.ops) if op.kind == "sync" and i < len(cuda.ops) - 1)
    ops = cuda.ops[last_sync + 1:]
    calls = [op for op in ops if op.kind == "call"]
    h2d = [op for op in ops if op.kind == "h2d"]
    d2h = [op for op in ops if op.kind == "d2h"]
    assert len(calls) == len(h2d) == len(d2h) == steps
    assert all(c.stream is cuda.main for c in calls)
    if overlap:
        assert all(o.stream is not cuda.main for o in h2d + d2h)
        assert h2d[0].stream is not d2h[0].stream
    R = bench.E2E_SLOTS
    for i in range(steps):
        r = i % R
        assert calls[i].kw == {"slot": r, "step": i}
        assert h2d[i].kw == {"slot": r, "win": i % nwin} and d2h[i].kw == {"slot": r, "win": i % nwin}
        # the call reads its inputs after they land and before its result is read
        assert _before(h2d[i], calls[i]) and _before(calls[i], d2h[i])
        if i + R < steps:
            # record r is refilled only after the call that read it, and
            # rewritten only after its result went back to the host
            assert _before(calls[i], h2d[i + R])
            assert _before(d2h[i], calls[i + R])
    # the end event follows every read-back
    end = [op for op in ops if op.kind == "record" and op.stream is cuda.main][-1]
    assert all(_before(o, end) for o in d2h)
    if overlap:
        # and the copies are free to overlap other windows' calls: the next
        # window's inputs do not wait for this window's call
        assert not _before(calls[0], h2d[1])


def test_e2e_record_reports_the_faster_ordering():
    rec = lambda v, ok: {"value": v, "unit": "windows/s", "copies": "...", "outputs_match_resident": ok}
    r = bench.e2e_record({"overlapped": rec(14000.0, True), "in_line": rec(12000.0, True)}, 100, 8)
    assert (r["value"], r["ordering"], r["outputs_match_resident"]) == (14000.0, "overlapped", True)
    assert r["in_line"]["value"] == 12000.0 and r["h2d_bytes_per_step"] == 100 and r["d2h_bytes_per_step"] == 8
    r = bench.e2e_record({"overlapped": rec(9000.0, True), "in_line": rec(24000.0, False)}, 100, 8)
    assert (r["value"], r["ordering"], r["outputs_match_resident"]) == (24000.0, "in_line", False)
    # results that depend on the step (sampling draws) are not compared
    r = bench.e2e_record({"overlapped": rec(1.0, None), "in_line": rec(2.0, None)}, 1, 1)
    assert r["outputs_match_resident"] is None
    assert [name for name, _, _ in bench.E2E_ORDERINGS] == ["overlapped", "in_line"]


def test_oracle_sample_runs_successive_windows_until_the_budget():
    import re
    # the tiny head: a window takes the oracle well under the budget, so the
    # sample goes on to the windows after window 0
    rate, desc = bench.oracle_sample(W.TINY, 9, 0.3, 1)
    n_win = int(re.search(r"of (\d+) successive window", desc).group(1))
    work = float(re.search(r"([\d.]+) windows of work", desc).group(1))
    assert n_win > 1 and rate > 0 and abs(work - n_win) <= 1.0
    # one window at most (the reference arm's step)
    rate1, desc1 = bench.oracle_sample(W.TINY, 9, 30.0, 1, max_windows=1)
    assert "of 1 successive window" in desc1 and "1.00 windows of work" in desc1 and rate1 > 0

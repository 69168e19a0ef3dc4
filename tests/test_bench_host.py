"""Host logic of bench.py (CPU only): the algorithmic byte counts behind the
roofline, the committed DRAM-traffic summaries it reads, the clock-record
summary and the peak lookup."""
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

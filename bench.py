"""Benchmark of the verify forward: verify windows/s and weight GB/s.

Default workload: the Qwen3-4B-shaped verify head (vocab 151936 x hidden
2560, int8 per-block-32, S = 9), one ``sdv_verify_head`` call per step (fused
dequant GEMM + argmax + greedy accept; logits never leave the chip), over
200 seeded windows.  Inputs are resident in HBM before timing; the weight
stream (413 MB) is larger than L2, so every window reads it from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sdv|reference]
                    [--config q4b|a3b|tiny] [--S S]

Prints one JSON line.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload.  With N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU (the path has no exchange
step); ``value`` is all ranks' windows over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402

METRIC = "verify windows/s and weight GB/s (% of GB300 HBM peak) for S=K+1 dequant-GEMM+argmax"


def head_bytes(wl, S: int) -> int:
    """Algorithmic bytes of one verify-head window: codes + fp16 scales +
    activations in + drafts in + argmax/accepted/next_a0 out."""
    codes = wl.n * wl.h if wl.bits == 8 else wl.n * wl.h // 2
    scales = wl.n * (wl.h // 32) * 2
    return codes + scales + S * wl.h * 2 + max(S - 1, 0) * 4 + S * 4 + 8


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- CPU oracle (the reference arm and the cpu_baseline leg) ----------------------

def oracle_sample(wl, S: int, budget_s: float):
    """Time the CPU oracle's verify-head arithmetic on a bounded row sample of
    one window and scale to windows/s.  Returns (windows/s, description)."""
    from oracle import quant, verify
    rows = 4096
    w = W.head_weights(wl, slice(0, rows))
    codes, scales = quant.quantize_block32(w, wl.bits)
    x = W.activations(wl, 0, S)
    done, t_used = 0, 0.0
    t0 = time.perf_counter()
    while True:
        y = verify.dequant_gemm64(x, codes, scales)
        verify.argmax_rows(y.astype(np.float32))
        done += rows
        t_used = time.perf_counter() - t0
        if t_used >= budget_s or done >= wl.n:
            break
    per_window = t_used * wl.n / done
    desc = (f"oracle dequant GEMM + argmax on {done} of {wl.n} vocab rows of window 0 "
            f"({rows}-row batches, {t_used:.1f} s), scaled to a full window")
    return 1.0 / per_window, desc


def run_reference(args, wl, S, world, rank):
    if rank != 0:
        return 0
    budget = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    rates = []
    for i in range(args.warmup + args.steps):
        r, desc = oracle_sample(wl, S, budget)
        if i >= args.warmup:
            rates.append(r)
    value = float(np.mean(rates))
    peak, kind = measured_peak()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: head {wl.n}x{wl.h} int{wl.bits}, S={S}", "S": S},
        "cpu_baseline": {"value": value, "unit": "windows/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "windows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---- GPU path ------------------------------------------------------------------------

def run_sdv(args, wl, S, world, rank, local):
    import torch
    from speculative_decode_verify_sdv_gb300 import build, sdv

    build.build()
    sdv.load()
    sdv.sdv_set_gemm_path({"auto": 0, "mma": 1, "tc": 2}[args.path])
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    # resident inputs: weights (quantised on the GPU), all windows' activations and drafts
    w = torch.from_numpy(W.head_weights(wl)).to(dev)
    head = sdv.quantize(w, wl.bits)
    del w
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    nwin = min(wl.windows, max(1, args.windows))
    xs = np.stack([W.activations(wl, i, S) for i in range(nwin)])
    x_dev = torch.from_numpy(xs.view(np.int16)).to(dev).view(torch.float16)
    ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, wl.n, wl.h, S, device=dev)
    am = torch.empty((nwin, S), dtype=torch.int32, device=dev)
    acc = torch.empty((nwin, 1), dtype=torch.int32, device=dev)
    nxt = torch.empty((nwin, 1), dtype=torch.int32, device=dev)
    zero_d = torch.zeros((nwin, max(S - 1, 1)), dtype=torch.int32, device=dev)
    # drafts: the draft rule over this path's own argmax chain (an untimed pre-pass)
    for i in range(nwin):
        sdv.sdv_verify_head(head, x_dev[i], S, zero_d[i], 0, None, am[i], acc[i], nxt[i], ws)
    chain = am.cpu().numpy()
    dr = np.stack([W.drafts(wl, i, S, chain[i])[0] if S > 1 else np.zeros(1, np.int32) for i in range(nwin)])
    d_dev = torch.from_numpy(np.ascontiguousarray(dr.reshape(nwin, -1))).to(dev)
    n_valid = S - 1
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % nwin
        sdv.sdv_verify_head(head, x_dev[j], S, d_dev[j], n_valid, None, am[j], acc[j], nxt[j], ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if sdv.sdv_device_status(ws) != sdv.SDV_OK:
        raise RuntimeError("device status reported a timeout during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_all0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
        t_all1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = t_all0.elapsed_time(t_all1)
    kernel_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    if sdv.sdv_device_status(ws) != sdv.SDV_OK:
        raise RuntimeError("device status reported a timeout during the timed region")
    elapsed_ms = max_over_ranks(world, elapsed_ms, dev)
    kernel_ms = max_over_ranks(world, kernel_ms, dev)

    # end to end through the C ABI with host buffers: H2D of the window's inputs,
    # the call, D2H of the ids, every step
    x_host = torch.from_numpy(xs.view(np.int16)).view(torch.float16).pin_memory()
    d_host = torch.from_numpy(np.ascontiguousarray(dr.reshape(nwin, -1))).pin_memory()
    x_stage = torch.empty_like(x_dev[0])
    d_stage = torch.empty_like(d_dev[0])
    out_host = torch.empty((nwin, S + 2), dtype=torch.int32).pin_memory()
    am1 = torch.empty(S, dtype=torch.int32, device=dev)
    acc1 = torch.empty(1, dtype=torch.int32, device=dev)
    nxt1 = torch.empty(1, dtype=torch.int32, device=dev)

    def e2e_step(i):
        j = i % nwin
        x_stage.copy_(x_host[j], non_blocking=True)
        d_stage.copy_(d_host[j], non_blocking=True)
        sdv.sdv_verify_head(head, x_stage, S, d_stage, n_valid, None, am1, acc1, nxt1, ws)
        out_host[j, :S].copy_(am1, non_blocking=True)
        out_host[j, S:S + 1].copy_(acc1, non_blocking=True)
        out_host[j, S + 1:].copy_(nxt1, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1), dev)
    h2d = S * wl.h * 2 + max(S - 1, 1) * 4
    d2h = (S + 2) * 4

    if rank != 0:
        return 0
    value = world * args.steps / (elapsed_ms / 1000.0)
    nbytes = head_bytes(wl, S)
    peak, kind = measured_peak()
    achieved = nbytes / (kernel_ms / 1000.0) / 1e9
    cpu_rate, cpu_desc = oracle_sample(wl, S, args.cpu_budget) if args.cpu_budget > 0 else (None, "skipped")
    line = {
        "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 x int%d -> f32" % wl.bits, "data": "synthetic",
        "config": {"workload": f"{wl.name}: verify head {wl.n}x{wl.h} int{wl.bits} per-block-32, S={S}",
                   "S": S, "windows": nwin, "bytes_per_window": nbytes,
                   "l2": "inputs larger than L2 (weight stream %.0f MB > 129 MB)" % (nbytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "weight_gbs": achieved, "hbm_frac": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_kind": kind, "kernel": f"verify-head GEMM ({args.path} path)",
                     "kernel_ms": kernel_ms},
        "cpu_baseline": {"value": cpu_rate, "unit": "windows/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": cpu_desc},
        "e2e": {"value": world * args.steps / (e2e_ms / 1000.0), "unit": "windows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["sdv", "reference"], default="sdv")
    ap.add_argument("--config", default="q4b", choices=["tiny", "q4b", "a3b"])
    ap.add_argument("--S", type=int, default=0)
    ap.add_argument("--windows", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--path", choices=["auto", "mma", "tc"], default="auto",
                    help="GEMM implementation (auto: tcgen05 where its plan fits)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    wl = W.BY_NAME[args.config]
    S = args.S or wl.s_default
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, wl, S, world, rank)
    return run_sdv(args, wl, S, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

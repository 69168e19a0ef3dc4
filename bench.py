"""Benchmark of the verify forward: verify windows/s and weight GB/s.

Default workload: the Qwen3-4B-shaped verify head (vocab 151936 x hidden
2560, int8 per-block-32, S = 9), one ``sdv_verify_head`` call per step (fused
dequant GEMM + argmax + greedy accept; logits never leave the chip), over
200 seeded windows.  Inputs are resident in HBM before timing; the weight
stream (413 MB) is larger than L2, so every window reads it from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sdv|reference]
                    [--config q4b|a3b|tiny|mlp27|moe] [--S S]

Other workloads (--config): the 35B-A3B-shaped int4 head (a3b), the tiny
L2-resident head (tiny), the 27B-shaped dense SwiGLU MLP (mlp27: gate/up
17408 x 5120 + down 5120 x 17408, int8) and the 256-expert int4 MoE layer
(moe).

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


KERNEL_SOURCES = ("tc_gemm.cu", "sdv_device.cuh", "sdv_kernels.h")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "speculative_decode_verify_sdv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
    the committed ncu summary of this workload, or None when there is none or the
    kernel sources changed since it was taken."""
    pdir = os.path.join(ROOT, "profiles")
    try:
        names = sorted(os.listdir(pdir))
    except OSError:
        return None, None
    cur = kernel_source_hash()
    for name in names:
        if not name.endswith(".md"):
            continue
        fields = {}
        with open(os.path.join(pdir, name)) as fh:
            for line in fh:
                if ":" in line and line.split(":", 1)[0] in ("kernel_source_sha256", "workload",
                                                             "traffic_bytes_per_launch"):
                    k, v = line.split(":", 1)
                    fields[k] = v.strip()
        if fields.get("workload") == workload and "traffic_bytes_per_launch" in fields:
            if fields.get("kernel_source_sha256") != cur:
                return None, f"profiles/{name} (stale: kernel changed since the capture)"
            return float(fields["traffic_bytes_per_launch"]), f"profiles/{name}"
    return None, None


# NVML (the driver's management library, read-only queries) through ctypes: the
# SM clock, its maximum, power and the clock-event reasons of one GPU.  Used by
# the poller process below and for single readings before and after a region.
NVML_POLLER = r"""
import ctypes, sys, time
bus, index, interval = sys.argv[1], int(sys.argv[2]), float(sys.argv[3])
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(3)
h = ctypes.c_void_p()
if not bus or nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
    if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
        sys.exit(4)
clk, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
rs = ctypes.c_ulonglong()
nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
try:
    get_reasons = nv.nvmlDeviceGetCurrentClocksEventReasons
except AttributeError:
    get_reasons = nv.nvmlDeviceGetCurrentClocksThrottleReasons
def reading():
    clk.value = 0; pw.value = 0; rs.value = 0
    nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
    nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
    get_reasons(h, ctypes.byref(rs))
    return "%.6f,%d,%d,%d,%d" % (time.time(), clk.value, mx.value, pw.value, rs.value)
out = sys.stdout
out.write("ready," + reading() + "\n"); out.flush()
while True:
    out.write(reading() + "\n"); out.flush()
    time.sleep(interval)
"""

# clock-event reason bits (NVML) and the names the contract uses
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}


def nvml_bus_id(device_index: int) -> str:
    """PCI bus id of a CUDA device in NVML's form (domain:bus:device.function)."""
    try:
        import torch
        p = torch.cuda.get_device_properties(device_index)
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        return ""


class ClockSampler:
    """SM clocks and clock-event reasons of the timed GPU: one reading right
    before the timed region, readings every ``interval`` seconds during it
    (NVML in a separate process, so the launch loop never waits on it), and one
    right after.  Falls back to ``nvidia-smi -lms`` when NVML cannot be loaded."""

    SMI_Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval: float = 0.002):
        self.index, self.interval = index, interval
        self.proc = None
        self.kind = None
        self.rows = []      # (sm_mhz, max_mhz, reasons set, phase)
        self.lock = threading.Lock()
        self.phase = "before"

    def __enter__(self):
        bus = nvml_bus_id(self.index)
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", NVML_POLLER, bus, str(self.index), str(self.interval)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline()
            if not first.startswith("ready,"):
                raise RuntimeError("NVML poller did not start")
            self.kind = "nvml"
            self._add_nvml(first[len("ready,"):])
        except Exception:
            self._stop()
            self.kind = "nvidia-smi"
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={bus or self.index}", f"--query-gpu={self.SMI_Q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
        if self.proc is not None:
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        time.sleep(2 * self.interval)
        with self.lock:
            self.phase = "during"
        return self

    def _add_nvml(self, line):
        f = line.strip().split(",")
        if len(f) < 5:
            return
        try:
            sm, mx, bits = float(f[1]), float(f[2]), int(f[4])
        except ValueError:
            return
        reasons = {nm for b, nm in NVML_REASONS.items() if bits & b}
        with self.lock:
            self.rows.append((sm, mx, reasons, self.phase))

    def _add_smi(self, line):
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            return
        try:
            sm, mx = float(f[1]), float(f[2])
        except ValueError:
            return
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {nm for nm, v in zip(names, f[5:9]) if v.lower() == "active"}
        with self.lock:
            self.rows.append((sm, mx, reasons, self.phase))

    def _read(self):
        add = self._add_nvml if self.kind == "nvml" else self._add_smi
        for line in self.proc.stdout:
            add(line)

    def _stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.proc = None

    def __exit__(self, *a):
        with self.lock:
            self.phase = "after"
        time.sleep(2 * self.interval)
        self._stop()

    def summary(self):
        with self.lock:
            rows = list(self.rows)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        during = [r for r in rows if r[3] == "during"]
        use = during if during else rows
        reasons = set()
        for r in rows:
            reasons |= r[2]
        return {"sm_mhz": float(np.median([r[0] for r in use])), "sm_max_mhz": rows[-1][1],
                "reasons": sorted(reasons), "samples": len(rows), "samples_during": len(during),
                "sampler": self.kind,
                "sm_mhz_before_after": [rows[0][0], rows[-1][0]]}


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


# ---- algorithmic bytes ------------------------------------------------------------

def weight_bytes(n: int, k: int, bits: int) -> int:
    """Codes + fp16 per-block-32 scales of one [n, k] quantised weight."""
    return (n * k if bits == 8 else n * k // 2) + n * (k // 32) * 2


def mlp_bytes(wl, S: int) -> int:
    """One dense SwiGLU MLP window: gate, up, down weights + x in + h out and
    back in (fp16) + y out (fp32)."""
    return (2 * weight_bytes(wl.inter, wl.h, wl.bits) + weight_bytes(wl.h, wl.inter, wl.bits)
            + S * wl.h * 2 + 2 * S * wl.inter * 2 + S * wl.h * 4)


def moe_expert_bytes(wl) -> int:
    return 2 * weight_bytes(wl.inter, wl.h, wl.bits) + weight_bytes(wl.h, wl.inter, wl.bits)


def moe_bytes(wl, S: int, n_hit: int) -> int:
    """One MoE window: the distinct hit experts' weights + x in + router
    logits in + out."""
    return n_hit * moe_expert_bytes(wl) + S * wl.h * 2 + S * wl.experts * 4 + S * wl.h * 4


# ---- CPU oracle (the reference arm and the cpu_baseline leg) ----------------------

def oracle_sample(wl, S: int, budget_s: float, threads: int = 0, max_windows: int | None = None):
    """Time the CPU oracle (the plain C++ one) with ``threads`` OpenMP threads
    (0: every core) on a bounded sample of the workload: window 0, then the
    windows after it, until ``budget_s`` seconds of oracle calls are used or
    ``max_windows`` windows are done (a window stopped by the budget counts by
    the share of its work done).  Returns (windows/s, description)."""
    import oracle
    from oracle import mlp, quant, verify
    prev = oracle.set_threads(threads)
    try:
        return _oracle_sample(wl, S, budget_s, max_windows, mlp, quant, verify)
    finally:
        oracle.set_threads(prev)


def _oracle_sample(wl, S, budget_s, max_windows, mlp, quant, verify):
    """The sample behind oracle_sample.  Each workload's weights are quantised
    once, before the clock: the head a block of its vocabulary rows, the MLP a
    row block of gate/up and of down, the MoE one expert; the work of a window
    runs over those blocks (the oracle's time per row is the same for every
    row).  Only the oracle's own calls are timed, not the input generator."""
    rng = np.random.default_rng(0)
    if wl.kind == "head":
        rows = 4096
        w = W.head_weights(wl, slice(0, rows))
        if wl.bits == 2:
            codes, scales = quant.quantize_fp4_block32(w)  # E2M1 codes, decoded by the oracle's GEMM
        else:
            codes, scales = quant.quantize_block32(w, wl.bits)
        total, unit = wl.n, "vocab rows"

        def window(i):
            x = W.activations(wl, i, S)

            def step(done):
                take = min(rows, total - done)  # the last block stops at the vocabulary's end
                y = verify.dequant_gemm64(x, codes[:take], scales[:take])
                verify.argmax_rows(y.astype(np.float32))
                return take
            return step
        what = "oracle dequant GEMM + argmax"
    elif wl.kind == "mlp":
        rows = 1024
        wg = rng.normal(0, 0.02, (rows, wl.h)).astype(np.float32)
        wd = rng.normal(0, 0.02, (rows, wl.inter)).astype(np.float32)
        cg, sg = quant.quantize_block32(wg, wl.bits)
        cd, sd = quant.quantize_block32(wd, wl.bits)
        h = rng.normal(0, 1, (S, wl.inter)).astype(np.float16)
        total, unit = wl.inter + wl.h, "weight rows (gate/up pairs + down)"

        def window(i):
            x = W.activations(wl, i, S)

            def step(done):
                mlp.qlinear_swiglu(x, cg, sg, cg, sg)
                verify.dequant_gemm64(h, cd, sd)
                return 2 * rows
            return step
        what = "oracle SwiGLU + down"
    else:
        E, I, H = wl.experts, wl.inter, wl.h
        one = {}
        for name, shape in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
            one[name] = quant.quantize_block32(rng.normal(0, 0.02, shape).astype(np.float32), wl.bits)
        total, unit = S * wl.top_k, "routed (row, expert) pairs"

        def window(i):
            x = W.activations(wl, i, S)
            logits = W.router_logits(wl, i, S)

            def step(done):
                if done == 0:
                    mlp.route_topk(logits, wl.top_k)
                s = done // wl.top_k
                mlp.expert_swiglu64(x[s:s + 1], 0, I, H, one["gate"], one["up"], one["down"])
                return 1
            return step
        what = "oracle route + expert SwiGLU MLP"
    t_used, windows, n_win = 0.0, 0.0, 0
    while True:
        step, done = window(n_win % wl.windows), 0
        while done < total and t_used < budget_s:
            t0 = time.perf_counter()
            done += step(done)
            t_used += time.perf_counter() - t0
        windows += min(done, total) / total
        n_win += 1
        if t_used >= budget_s or (max_windows is not None and n_win >= max_windows):
            break
    desc = (f"{what} on the {unit} of {n_win} successive window(s) from window 0 (index mod {wl.windows}): "
            f"{windows:.2f} windows of work in {t_used:.1f} s of oracle calls")
    return windows / t_used, desc


def oracle_threads() -> int:
    """OpenMP threads the C++ oracle runs on when all cores are used."""
    import oracle
    prev = oracle.set_threads(0)
    n = oracle.threads()
    oracle.set_threads(prev)
    return n


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, S: int, budget_s: float):
    """The C++ oracle as it stands, all cores and one thread, each on a bounded
    sample of the workload (budget_s seconds of oracle calls each, over as many
    windows as fit), scaled to windows/s."""
    if budget_s <= 0:
        return {"value": None, "unit": "windows/s", "cores": None, "kind": "oracle", "sample": "skipped"}
    cores = oracle_threads()
    r_all, d_all = oracle_sample(wl, S, budget_s, cores)
    r_one, d_one = oracle_sample(wl, S, budget_s, 1)
    return {"value": r_all, "unit": "windows/s", "cores": cores, "kind": "oracle",
            "sample": f"plain C++ oracle (fp64, OpenMP over output rows) on {cores} threads: {d_all}",
            "single_thread": {"value": r_one, "unit": "windows/s", "cores": 1, "sample": d_one},
            "cpu_model": cpu_model()}


def wtype(bits: int) -> str:
    return "fp4 (E2M1)" if bits == 2 else f"int{bits}"


def workload_name(wl, S: int) -> str:
    if wl.kind == "head":
        return f"{wl.name}: verify head {wl.n}x{wl.h} {wtype(wl.bits)} per-block-32, S={S}"
    if wl.kind == "mlp":
        return (f"{wl.name}: SwiGLU MLP gate/up {wl.inter}x{wl.h}, down {wl.h}x{wl.inter} "
                f"int{wl.bits} per-block-32, S={S}")
    return (f"{wl.name}: MoE {wl.experts} experts (gate/up {wl.inter}x{wl.h}, down {wl.h}x{wl.inter}) "
            f"int{wl.bits}, top-{wl.top_k}, S={S}")


def run_reference(args, wl, S, world, rank):
    if rank != 0:
        return 0
    budget = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    rates = []
    desc = ""
    for i in range(args.warmup + args.steps):
        r, desc = oracle_sample(wl, S, budget, 0, max_windows=1)
        if i >= args.warmup:
            rates.append(r)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(wl, S), "S": S},
        "cpu_baseline": {"value": value, "unit": "windows/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": "plain C++ oracle (fp64, OpenMP over output rows), each step: " + desc,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "windows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---- GPU jobs: resident inputs, one window per step ----------------------------------

class HeadJob:
    """sdv_verify_head with logits = NULL: one launch per window."""

    def __init__(self, sdv, torch, wl, S, dev, nwin):
        self.sdv, self.torch, self.wl, self.S, self.dev, self.nwin = sdv, torch, wl, S, dev, nwin
        w = torch.from_numpy(W.head_weights(wl)).to(dev)
        self.head = sdv.quantize(w, wl.bits)
        del w
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self.xs = np.stack([W.activations(wl, i, S) for i in range(nwin)])
        self.x_dev = torch.from_numpy(self.xs.view(np.int16)).to(dev).view(torch.float16)
        self.ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, wl.n, wl.h, S, device=dev)
        i32 = torch.int32
        self.am = torch.empty((nwin, S), dtype=i32, device=dev)
        self.acc = torch.empty((nwin, 1), dtype=i32, device=dev)
        self.nxt = torch.empty((nwin, 1), dtype=i32, device=dev)
        zero_d = torch.zeros((nwin, max(S - 1, 1)), dtype=i32, device=dev)
        # drafts: the draft rule over this path's own argmax chain (an untimed pre-pass)
        for i in range(nwin):
            sdv.sdv_verify_head(self.head, self.x_dev[i], S, zero_d[i], 0, None, self.am[i], self.acc[i],
                                self.nxt[i], self.ws)
        chain = self.am.cpu().numpy()
        dr = np.stack([W.drafts(wl, i, S, chain[i])[0] if S > 1 else np.zeros(1, np.int32) for i in range(nwin)])
        self.dr = np.ascontiguousarray(dr.reshape(nwin, -1))
        self.d_dev = torch.from_numpy(self.dr).to(dev)
        self.n_valid = S - 1
        # each window's argument views, made once (a view per call costs the host
        # more than the tiny head's kernel)
        self.win = [(self.x_dev[j], self.d_dev[j], self.am[j], self.acc[j], self.nxt[j]) for j in range(nwin)]
        self.kernel = "verify-head GEMM + argmax + accept (one launch)"
        self.ws_list = [self.ws]

    def bytes(self, i):
        return head_bytes(self.wl, self.S)

    def step(self, i):
        x, d, am, acc, nxt = self.win[i % self.nwin]
        self.sdv.sdv_verify_head(self.head, x, self.S, d, self.n_valid, None, am, acc, nxt, self.ws)

    def e2e_setup(self, slots):
        # one pinned host record per window (hidden states, then drafts) and
        # `slots` device records they land in: one H2D copy per step; the results
        # (ids, accepted, next token) are one device record per slot, read back by
        # one D2H copy
        t, S, dev = self.torch, self.S, self.dev
        xb, db = S * self.wl.h * 2, self.dr.shape[1] * 4
        rec = np.zeros((self.nwin, xb + db), dtype=np.uint8)
        rec[:, :xb] = self.xs.reshape(self.nwin, -1).view(np.uint8)
        rec[:, xb:] = self.dr.view(np.uint8).reshape(self.nwin, -1)
        self.in_host = t.from_numpy(rec).pin_memory()
        self.e2e_in = [t.empty(xb + db, dtype=t.uint8, device=dev) for _ in range(slots)]
        self.e2e_out = [t.empty(S + 2, dtype=t.int32, device=dev) for _ in range(slots)]
        self.e2e_args = [(a[:xb].view(t.float16).view(S, self.wl.h), a[xb:].view(t.int32), o[:S], o[S:S + 1],
                          o[S + 1:]) for a, o in zip(self.e2e_in, self.e2e_out)]
        self.out_host = t.empty((self.nwin, S + 2), dtype=t.int32).pin_memory()
        self.in_rows, self.out_rows = list(self.in_host.unbind(0)), list(self.out_host.unbind(0))
        self.h2d = xb + db
        self.d2h = (S + 2) * 4

    def e2e_call(self, r, i):
        x, d, am, acc, nxt = self.e2e_args[r]
        self.sdv.sdv_verify_head(self.head, x, self.S, d, self.n_valid, None, am, acc, nxt, self.ws)

    def resident_out(self):
        """Each window's result record as the resident timed region left it."""
        return self.torch.cat([self.am, self.acc, self.nxt], dim=1).cpu()


class SampleJob(HeadJob):
    """sdv_verify_sample (temperature 1, a fresh counter per window) on the head
    workload: the same weight stream with the sampling epilogue."""

    def __init__(self, sdv, torch, wl, S, dev, nwin):
        super().__init__(sdv, torch, wl, S, dev, nwin)
        self.ws = sdv.workspace(sdv.SDV_OP_VERIFY_SAMPLE, wl.n, wl.h, S, device=dev)
        self.ws_list = [self.ws]
        self.kernel = "sampling verify: GEMM + Gumbel-max draws + softmax + accept (one launch)"

    def step(self, i):
        x, d, am, acc, nxt = self.win[i % self.nwin]
        self.sdv.sdv_verify_sample(self.head, x, self.S, d, self.n_valid, 1.0, 1, i, None, am, acc, nxt, self.ws)

    def e2e_call(self, r, i):
        x, d, am, acc, nxt = self.e2e_args[r]
        self.sdv.sdv_verify_sample(self.head, x, self.S, d, self.n_valid, 1.0, 1, i, None, am, acc, nxt, self.ws)

    def resident_out(self):
        # the draws depend on the step's counter, which differs between the two
        # regions: nothing to compare
        return None


class MlpJob:
    """Dense SwiGLU MLP: sdv_qlinear_swiglu (gate/up) then sdv_qlinear (down)."""

    def __init__(self, sdv, torch, wl, S, dev, nwin):
        self.sdv, self.torch, self.wl, self.S, self.dev, self.nwin = sdv, torch, wl, S, dev, nwin
        self.w = {}
        for which in ("gate", "up", "down"):
            w = torch.from_numpy(W.mlp_weights(wl, which)).to(dev)
            self.w[which] = sdv.quantize(w, wl.bits)
            del w
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        self.xs = np.stack([W.activations(wl, i, S) for i in range(nwin)])
        self.x_dev = torch.from_numpy(self.xs.view(np.int16)).to(dev).view(torch.float16)
        self.y = torch.empty((nwin, S, wl.h), dtype=torch.float32, device=dev)
        self.h = torch.empty((S, wl.inter), dtype=torch.float16, device=dev)
        self.ws_sw = sdv.workspace(sdv.SDV_OP_QLINEAR_SWIGLU, wl.inter, wl.h, S, device=dev)
        self.ws_dn = sdv.workspace(sdv.SDV_OP_QLINEAR, wl.h, wl.inter, S, device=dev)
        self.kernel = "gate/up + down GEMMs (sdv_qlinear_swiglu + sdv_qlinear)"
        self.ws_list = [self.ws_sw, self.ws_dn]

    def bytes(self, i):
        return mlp_bytes(self.wl, self.S)

    def _call(self, x, y):
        sdv = self.sdv
        sdv.sdv_qlinear_swiglu(self.w["gate"], self.w["up"], x, self.S, self.h, self.ws_sw)
        sdv.sdv_qlinear(self.w["down"], self.h, self.S, y, self.ws_dn)

    def step(self, i):
        j = i % self.nwin
        if not hasattr(self, "win"):
            self.win = [(self.x_dev[w], self.y[w]) for w in range(self.nwin)]
        self._call(*self.win[j])

    def e2e_setup(self, slots):
        t = self.torch
        self.in_host = t.from_numpy(self.xs.view(np.int16)).view(t.float16).pin_memory()
        self.e2e_in = [t.empty_like(self.x_dev[0]) for _ in range(slots)]
        self.e2e_out = [t.empty_like(self.y[0]) for _ in range(slots)]
        self.out_host = t.empty((self.nwin,) + tuple(self.y.shape[1:]), dtype=t.float32).pin_memory()
        self.in_rows, self.out_rows = list(self.in_host.unbind(0)), list(self.out_host.unbind(0))
        self.h2d = self.S * self.wl.h * 2
        self.d2h = self.S * self.wl.h * 4

    def e2e_call(self, r, i):
        self._call(self.e2e_in[r], self.e2e_out[r])

    def resident_out(self):
        return self.y.cpu()


class MoeJob:
    """sdv_moe_gather_qmm: route + group, gate/up over the hit experts, down."""

    def __init__(self, sdv, torch, wl, S, dev, nwin):
        self.sdv, self.torch, self.wl, self.S, self.dev, self.nwin = sdv, torch, wl, S, dev, nwin
        self.w = {}
        for which in ("gate", "up", "down"):
            w = torch.from_numpy(W.moe_weights(wl, which)).to(dev)
            self.w[which] = sdv.quantize(w, wl.bits)
            del w
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        self.xs = np.stack([W.activations(wl, i, S) for i in range(nwin)])
        self.ls = np.stack([W.router_logits(wl, i, S) for i in range(nwin)])
        self.x_dev = torch.from_numpy(self.xs.view(np.int16)).to(dev).view(torch.float16)
        self.l_dev = torch.from_numpy(self.ls).to(dev)
        self.out = torch.empty((nwin, S, wl.h), dtype=torch.float32, device=dev)
        self.ws = sdv.workspace(sdv.SDV_OP_MOE, wl.inter, wl.h, S, wl.experts, wl.top_k, device=dev)
        # distinct experts each window hits (for its algorithmic bytes)
        from oracle import mlp
        self.n_hit = [len(np.unique(mlp.route_topk(self.ls[i], wl.top_k)[0])) for i in range(nwin)]
        self.kernel = "MoE call (route, gate/up GEMM, SwiGLU, down GEMM, reduce)"
        self.ws_list = [self.ws]

    def bytes(self, i):
        return moe_bytes(self.wl, self.S, self.n_hit[i % self.nwin])

    def _call(self, x, l, out):
        wl = self.wl
        self.sdv.sdv_moe_gather_qmm(self.w["gate"], self.w["up"], self.w["down"], wl.experts, wl.inter, wl.h,
                                    wl.top_k, x, l, self.S, out, None, None, self.ws)

    def step(self, i):
        j = i % self.nwin
        if not hasattr(self, "win"):
            self.win = [(self.x_dev[w], self.l_dev[w], self.out[w]) for w in range(self.nwin)]
        self._call(*self.win[j])

    def e2e_setup(self, slots):
        # one pinned host record per window (hidden states, then router logits)
        # and `slots` device records they land in: one H2D copy and one D2H per step
        t, S, dev = self.torch, self.S, self.dev
        xb, lb = S * self.wl.h * 2, S * self.wl.experts * 4
        rec = np.zeros((self.nwin, xb + lb), dtype=np.uint8)
        rec[:, :xb] = self.xs.reshape(self.nwin, -1).view(np.uint8)
        rec[:, xb:] = self.ls.astype(np.float32).reshape(self.nwin, -1).view(np.uint8)
        self.in_host = t.from_numpy(rec).pin_memory()
        self.e2e_in = [t.empty(xb + lb, dtype=t.uint8, device=dev) for _ in range(slots)]
        self.e2e_out = [t.empty_like(self.out[0]) for _ in range(slots)]
        self.e2e_args = [(a[:xb].view(t.float16).view(S, self.wl.h), a[xb:].view(t.float32).view(S, self.wl.experts),
                          o) for a, o in zip(self.e2e_in, self.e2e_out)]
        self.out_host = t.empty((self.nwin,) + tuple(self.out.shape[1:]), dtype=t.float32).pin_memory()
        self.in_rows, self.out_rows = list(self.in_host.unbind(0)), list(self.out_host.unbind(0))
        self.h2d = xb + lb
        self.d2h = S * self.wl.h * 4

    def e2e_call(self, r, i):
        self._call(*self.e2e_args[r])

    def resident_out(self):
        return self.out.cpu()


JOBS = {"head": HeadJob, "mlp": MlpJob, "moe": MoeJob}


def timed_region(job, steps, world, local, sdv, torch):
    """K back-to-back windows between two events on the launching stream, with
    the clocks sampled during the region and this library's kernel launches
    counted.  A window's GEMM is a programmatic dependent launch, so its start-up
    overlaps the previous window's tail; an event between windows would
    serialise them, so the per-launch duration is the region / K.
    Returns (region ms, launches, the clock sampler)."""
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        n0 = sdv.sdv_launch_count()
        t0.record(stream)
        for i in range(steps):
            job.step(i)
        t1.record(stream)
        n_launched = sdv.sdv_launch_count() - n0
        torch.cuda.synchronize()
    barrier(world)
    return t0.elapsed_time(t1), n_launched, clk


# Device records the end-to-end loop rotates through: a window's inputs land in
# one while the calls of the windows before it still read the others.
E2E_SLOTS = 3


def e2e_region(job, steps, warmup, world, torch, overlap):
    """The windows end to end through the C ABI from pinned host memory: every
    step copies its window's inputs host to device, makes the call and reads its
    result back device to host.  With `overlap` the two copies run on two copy
    streams and each window uses one of the job's E2E_SLOTS device records, so a
    window's copies overlap the calls of its neighbours: the call waits for its
    inputs, and a record is refilled only after the call that read it has
    finished and its result is back on the host.  That costs the host ten more
    stream and event calls per step, so a window shorter than the host's issue
    time runs faster with the copies and the call in line on the launching
    stream, the other ordering.  Returns the region's ms (events on the
    launching stream, which waits for the last read-back before the end
    event)."""
    stream = torch.cuda.current_stream()
    R = len(job.e2e_in)
    cin, cout = torch.cuda.Stream(device=stream.device), torch.cuda.Stream(device=stream.device)
    ready, done, read = ([torch.cuda.Event() for _ in range(R)] for _ in range(3))

    def one(i):
        r, j = i % R, i % job.nwin
        if not overlap:
            job.e2e_in[r].copy_(job.in_rows[j], non_blocking=True)
            job.e2e_call(r, i)
            job.out_rows[j].copy_(job.e2e_out[r], non_blocking=True)
            return
        with torch.cuda.stream(cin):
            cin.wait_event(done[r])      # the call that last read record r has finished
            job.e2e_in[r].copy_(job.in_rows[j], non_blocking=True)
            ready[r].record(cin)
        stream.wait_event(ready[r])
        stream.wait_event(read[r])       # record r's previous result is back on the host
        job.e2e_call(r, i)
        done[r].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(done[r])
            job.out_rows[j].copy_(job.e2e_out[r], non_blocking=True)
            read[r].record(cout)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cin.wait_event(e0)
    cout.wait_event(e0)
    for i in range(steps):
        one(i)
    stream.wait_stream(cout)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


E2E_ORDERINGS = (
    ("overlapped", True, f"H2D and D2H on two copy streams, {E2E_SLOTS} device records in rotation "
                         "(a window's copies overlap its neighbours' calls)"),
    ("in_line", False, "H2D, call, D2H in line on the launching stream"),
)


def e2e_record(by_ordering: dict, h2d: int, d2h: int) -> dict:
    """The bench line's e2e record: the faster ordering's rate as the value,
    named in `ordering`, with both orderings' records beside it."""
    best = max(by_ordering, key=lambda k: by_ordering[k]["value"])
    checks = [r["outputs_match_resident"] for r in by_ordering.values()]
    return {"value": by_ordering[best]["value"], "unit": by_ordering[best]["unit"],
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ordering": best,
            "outputs_match_resident": None if None in checks else all(checks), **by_ordering}


def e2e_matches(job, steps, torch):
    """Whether the results the end-to-end loop read back equal, bit for bit,
    those the resident timed region left for the same windows (None where the
    job's results depend on the step, as the sampling draws do)."""
    ref = job.resident_out()
    if ref is None:
        return None
    n = min(steps, job.nwin)
    return bool(torch.equal(job.out_host[:n].reshape(n, -1), ref[:n].reshape(n, -1)))


# The other workloads a default single-GPU run measures beside the headline one
# (name:S), so that one driver run records every config's number with its own
# clocks: the int4 head at the window the pages' cliff is quoted on and at one
# row, the dense MLP stack, the MoE layer, and the L2-resident tiny head (with
# its CUDA-graph number).
ALSO_DEFAULT = "a3b:17,a3b:1,mlp27:17,moe:17,tiny:9"


def also_specs(args, world) -> list:
    """(workload, S) pairs of --also: "auto" is ALSO_DEFAULT on the default
    single-GPU run (q4b greedy, integer weights) and nothing otherwise."""
    spec = args.also
    if spec == "auto":
        default_run = args.config == "q4b" and not args.fp4 and args.verify == "greedy" and args.path == "auto"
        spec = ALSO_DEFAULT if (default_run and world == 1) else ""
    out = []
    for item in filter(None, (t.strip() for t in spec.split(","))):
        if item == "none":
            return []
        name, _, s = item.partition(":")
        if name not in W.BY_NAME:
            raise SystemExit(f"--also: unknown workload {name!r}")
        wl = W.BY_NAME[name]
        out.append((wl, int(s) if s else wl.s_default))
    return out


L2_BYTES = 129e6  # the GB300's L2


def l2_label(nbytes: float) -> str:
    if nbytes > L2_BYTES:
        return "inputs larger than L2 (weight stream %.0f MB > 129 MB)" % (nbytes / 1e6)
    return "L2-warm: the working set (%.2f MB) fits the 129 MB L2; not an HBM number" % (nbytes / 1e6)


def graph_record(job, steps, nbytes, torch, replays=10) -> dict:
    """The secondary back-to-back number: `steps` windows captured once as a CUDA
    graph (the library's launches keep their programmatic dependencies as graph
    edges) and replayed `replays` times between two events on the stream."""
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                job.step(i)
        g.replay()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / (replays * steps)
        del g
    except Exception as exc:  # a capture the runtime refuses: say why, keep the line
        return {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
    return {"value": 1000.0 / per, "unit": "windows/s", "ms_per_step": per, "windows_per_graph": steps,
            "replays": replays, "l2": l2_label(nbytes)}


def measure_also(args, specs, sdv, torch, dev, local) -> list:
    """Each (workload, S): warm-up, the timed region (as the headline line),
    a status check; one compact record per workload."""
    peak, kind = measured_peak()
    out = []
    for wl, S in specs:
        nwin = min(wl.windows, max(1, args.windows))
        job = JOBS[wl.kind](sdv, torch, wl, S, dev, nwin)
        for i in range(args.warmup):
            job.step(i)
        torch.cuda.synchronize()
        ms, n_launched, clk = timed_region(job, args.steps, 1, local, sdv, torch)
        if not all(sdv.sdv_last_device_status(w) == sdv.SDV_OK for w in job.ws_list):
            raise RuntimeError(f"device status reported an error measuring {wl.name} S={S}")
        nbytes = float(np.mean([job.bytes(i) for i in range(args.steps)]))
        per = ms / args.steps
        achieved = nbytes / (per / 1000.0) / 1e9
        rec = {"workload": workload_name(wl, S), "S": S, "value": 1000.0 / per, "unit": "windows/s",
               "ms_per_step": per, "bytes_per_window": nbytes, "l2": l2_label(nbytes), "weight_gbs": achieved,
               "hbm_frac": achieved / peak, "peak_kind": kind, "gpu_launches": n_launched,
               "kernel": f"{job.kernel} ({args.path} path)", "clocks": clk.summary()}
        if wl.kind == "head":
            rec["graph"] = graph_record(job, args.steps, nbytes, torch)
            if not all(sdv.sdv_last_device_status(w) == sdv.SDV_OK for w in job.ws_list):
                raise RuntimeError(f"device status reported an error in the graph replays of {wl.name} S={S}")
        out.append(rec)
        del job
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_sdv(args, wl, S, world, rank, local):
    import torch
    from speculative_decode_verify_sdv_gb300 import build, sdv

    build.build()
    sdv.load()
    sdv.sdv_set_gemm_path({"auto": 0, "mma": 1, "tc": 2, "gemv": 3}[args.path])
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    nwin = min(wl.windows, max(1, args.windows))
    sampling = args.verify == "sample" and wl.kind == "head"
    job = (SampleJob if sampling else JOBS[wl.kind])(sdv, torch, wl, S, dev, nwin)
    stream = torch.cuda.current_stream()

    def status_ok():
        return all(sdv.sdv_last_device_status(w) == sdv.SDV_OK for w in job.ws_list)

    for i in range(args.warmup):
        job.step(i)
    torch.cuda.synchronize()
    if not status_ok():
        raise RuntimeError("device status reported an error during warm-up")

    elapsed_ms, n_launched, clk = timed_region(job, args.steps, world, local, sdv, torch)
    kernel_ms = elapsed_ms / args.steps
    if not status_ok():
        raise RuntimeError("device status reported an error during the timed region")
    # for reference: each launch alone, bracketed by its own events (serialised)
    n_iso = min(args.steps, 50)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iso)]
    for i in range(n_iso):
        ev[i][0].record(stream)
        job.step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    iso_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    elapsed_ms = max_over_ranks(world, elapsed_ms, dev)
    kernel_ms = max_over_ranks(world, kernel_ms, dev)
    iso_ms = max_over_ranks(world, iso_ms, dev)
    nbytes = float(np.mean([job.bytes(i) for i in range(args.steps)]))

    # end to end through the C ABI with host buffers: H2D of the window's inputs,
    # the call, D2H of the result, every step; timed in both orderings (the
    # copies on copy streams, then in line on the launching stream), the faster
    # one reported as the value
    job.e2e_setup(E2E_SLOTS)
    e2e = {}
    for name, overlap, copies in E2E_ORDERINGS:
        ms = max_over_ranks(world, e2e_region(job, args.steps, args.warmup, world, torch, overlap), dev)
        e2e[name] = {"value": world * args.steps / (ms / 1000.0), "unit": "windows/s", "copies": copies,
                     "outputs_match_resident": e2e_matches(job, args.steps, torch)}
    if not status_ok():
        raise RuntimeError("device status reported an error in the end-to-end regions")

    if rank != 0:
        return 0
    also = measure_also(args, also_specs(args, world), sdv, torch, dev, local)
    value = world * args.steps / (elapsed_ms / 1000.0)
    peak, kind = measured_peak()
    achieved = nbytes / (kernel_ms / 1000.0) / 1e9
    prof_key = f"{wl.name} S={S}" + (" sample" if sampling else "") + (" fp4" if wl.bits == 2 else "")
    traffic, traffic_src = (profiled_traffic(prof_key) if wl.kind == "head" else (None, None))
    cpu = cpu_baseline(wl, S, args.cpu_budget)
    line = {
        "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 x %s -> f32" % wtype(wl.bits), "data": "synthetic",
        "config": {"workload": workload_name(wl, S) + (", sampling verify T=1" if sampling else ""), "S": S,
                   "windows": nwin, "bytes_per_window": nbytes,
                   "l2": l2_label(nbytes),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "weight_gbs": achieved, "hbm_frac": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "traffic_source": traffic_src, "peak_kind": kind, "kernel": f"{job.kernel} ({args.path} path)",
                     "kernel_ms": kernel_ms, "kernel_ms_serialised": iso_ms,
                     "timing": "events around the K back-to-back launches of the timed region, / K"},
        "cpu_baseline": cpu,
        "e2e": e2e_record(e2e, job.h2d, job.d2h),
        "gpu_launches": n_launched,
        "clocks": clk.summary(),
    }
    if wl.kind == "head":
        line["graph"] = graph_record(job, args.steps, nbytes, torch)
        if not status_ok():
            raise RuntimeError("device status reported an error in the graph replays")
    if also:
        line["also_measured"] = also
    print(json.dumps(line))
    return 0


def run_spec_loop(args, wl, S):
    """End-to-end greedy n-gram speculative decoding through the verify head:
    the toy model body of ``synth.toy_model`` feeds hidden rows, the host loop
    drafts and commits, every round is one ``sdv_verify_head`` call.  Prints one
    JSON line: spec tokens/s against plain greedy (S = 1 per token), both wall
    clock on the host (the loop is synchronous), losslessness, tokens per
    round against E(alpha, K)."""
    import torch
    from speculative_decode_verify_sdv_gb300 import build, sdv, specdec
    from synth.toy_model import ToyHidden
    if wl.kind != "head":
        raise SystemExit("--spec-loop needs a head workload (tiny, q4b, a3b)")
    build.build()
    sdv.load()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    w = torch.from_numpy(W.head_weights(wl)).to(dev)
    head = sdv.quantize(w, wl.bits)
    del w
    torch.cuda.synchronize()
    K = S - 1
    hidden = ToyHidden(wl.h, W.stream_seed(wl.key, 90), lambda t: W.head_weights(wl, slice(t, t + 1))[0],
                       W.W_SIGMA, p_echo=args.p_echo, period=5)
    prompt = [int(t) for t in W.randint(W.stream_seed(wl.key, 91), 32, wl.n)]
    ver1, verS = specdec.HeadVerifier(head, 1, device=dev), specdec.HeadVerifier(head, S, device=dev)
    specdec.spec_decode(verS, hidden, prompt, 16, K, args.ngram)   # warm-up (shapes, caches)
    specdec.greedy_decode(ver1, hidden, prompt, 16)
    t0 = time.perf_counter()
    greedy = specdec.greedy_decode(ver1, hidden, prompt, args.gen)
    t1 = time.perf_counter()
    stats = {}
    spec = specdec.spec_decode(verS, hidden, prompt, args.gen, K, args.ngram, stats)
    t2 = time.perf_counter()
    if ver1.status() != sdv.SDV_OK or verS.status() != sdv.SDV_OK:
        raise RuntimeError("device status reported an error in the spec loop")
    alpha = specdec.alpha_estimate(stats)
    per_round = (stats["accepted"] + stats["rounds"]) / max(1, stats["rounds"])
    line = {
        "metric": "greedy n-gram spec-decode tokens/s through the verify head (toy model body)",
        "value": args.gen / (t2 - t1), "unit": "tokens/s", "higher_is_better": True,
        "greedy_tokens_per_s": args.gen / (t1 - t0), "speedup": (t1 - t0) / (t2 - t1),
        "lossless": spec == greedy, "rounds": stats["rounds"], "accepted": stats["accepted"],
        "tokens_per_round": per_round, "alpha": alpha,
        "E_alpha_K": specdec.expected_tokens_per_round(alpha, K), "K": K, "ngram": args.ngram,
        "gen": args.gen, "p_echo": args.p_echo,
        "config": {"workload": workload_name(wl, S), "S": S, "model_body": "synth.toy_model.ToyHidden (period 5)"},
        "timing": "host wall clock around each whole decode (per round: H2D of the window, the call, D2H, "
                  "one stream sync; the round's GPU work replayed as a CUDA graph per window size)",
    }
    print(json.dumps(line), flush=True)
    return 0 if line["lossless"] else 1


def run_sweep(args, wl):
    """Verify-head time per window against the window size S (1..32): the GB300
    analogue of the pages' c_v(S) = t(S) / t(1).  One JSON line."""
    import torch
    from speculative_decode_verify_sdv_gb300 import build, sdv
    if wl.kind != "head":
        raise SystemExit("--sweep-S needs a head workload (tiny, q4b, a3b)")
    build.build()
    sdv.load()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    w = torch.from_numpy(W.head_weights(wl)).to(dev)
    head = sdv.quantize(w, wl.bits)
    del w
    torch.cuda.synchronize()
    points = []
    for S in [int(v) for v in args.sweep_S.split(",")]:
        x = torch.from_numpy(W.activations(wl, 0, S).view(np.int16)).to(dev).view(torch.float16)
        dr = torch.zeros(max(S - 1, 1), dtype=torch.int32, device=dev)
        am = torch.empty(S, dtype=torch.int32, device=dev)
        acc = torch.empty(1, dtype=torch.int32, device=dev)
        nxt = torch.empty(1, dtype=torch.int32, device=dev)
        ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, wl.n, wl.h, S, device=dev)
        for _ in range(3):
            sdv.sdv_verify_head(head, x, S, dr, 0, None, am, acc, nxt, ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            sdv.sdv_verify_head(head, x, S, dr, 0, None, am, acc, nxt, ws)
        e1.record()
        torch.cuda.synchronize()
        points.append({"S": S, "us": e0.elapsed_time(e1) * 1000.0 / args.steps})
    t1 = next((p["us"] for p in points if p["S"] == 1), points[0]["us"])
    for p in points:
        p["c_v"] = p["us"] / t1
        p["weight_gbs"] = head_bytes(wl, p["S"]) / (p["us"] * 1e-6) / 1e9
    line = {"metric": "verify-head us per window against S; c_v(S) = t(S) / t(1)", "unit": "us",
            "config": {"workload": f"{wl.name}: verify head {wl.n}x{wl.h} int{wl.bits}", "steps": args.steps,
                       "timing": "events around the back-to-back launches, / steps"},
            "points": points}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["sdv", "reference"], default="sdv")
    ap.add_argument("--config", default="q4b", choices=["tiny", "q4b", "a3b", "mlp27", "moe"])
    ap.add_argument("--S", type=int, default=0)
    ap.add_argument("--windows", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--path", choices=["auto", "mma", "tc", "gemv"], default="auto",
                    help="GEMM implementation (auto: tcgen05 where its plan fits; gemv: CUDA cores for S <= 2)")
    ap.add_argument("--verify", choices=["greedy", "sample"], default="greedy",
                    help="head workloads: greedy verify (sdv_verify_head) or sampling verify at T = 1")
    ap.add_argument("--sweep-S", default="", help="comma-separated window sizes: verify-head time per S")
    ap.add_argument("--also", default="auto",
                    help="other workloads measured after the headline one, name:S comma-separated, 'none', or "
                         f"'auto' ({ALSO_DEFAULT} on the default single-GPU run)")
    ap.add_argument("--fp4", action="store_true",
                    help="head workloads: the same head quantised to FP4 (E2M1) instead of its integer type")
    ap.add_argument("--spec-loop", action="store_true",
                    help="end-to-end n-gram speculative decoding on the head workload instead of the kernel bench")
    ap.add_argument("--gen", type=int, default=512, help="--spec-loop: tokens to generate")
    ap.add_argument("--ngram", type=int, default=3, help="--spec-loop: n-gram order of the drafter")
    ap.add_argument("--p-echo", type=float, default=0.7, help="--spec-loop: share of echo contexts in the toy model")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    wl = W.BY_NAME[args.config]
    if args.fp4:
        if wl.kind != "head":
            raise SystemExit("--fp4 needs a head workload")
        import dataclasses
        wl = dataclasses.replace(wl, bits=2)
    S = args.S or wl.s_default
    if args.spec_loop:
        return run_spec_loop(args, wl, S)
    if args.sweep_S:
        return run_sweep(args, wl)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, wl, S, world, rank)
    return run_sdv(args, wl, S, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

"""Builds the host-only launch tracer (test infrastructure).

The library's CUDA sources are compiled as for the product, except that the
device code is kept as PTX only (no machine code is generated: it is never
loaded), and linked with ``stub_runtime.cpp`` and ``trace_main.cpp`` instead of
the CUDA runtime.  The result runs on a machine without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
CSRC = os.path.join(ROOT, "speculative_decode_verify_sdv_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(ROOT, "_build", "launch_trace")
SOURCES = ["api.cu", "dq_gemm.cu", "tc_gemm.cu", "gemv.cu", "small_kernels.cu", "moe_kernels.cu", "noalloc.cu"]
HOST = ["stub_runtime.cpp", "trace_main.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build(csrc: str = CSRC, out_dir: str = OUT) -> str:
    """Compile and link the tracer; returns the executable's path (rebuilt only
    when a source or header is newer)."""
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "trace")
    deps = [os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".h", ".cuh"))]
    deps += [os.path.join(INCLUDE, "sdv.h")] + [os.path.join(HERE, f) for f in HOST]
    if os.path.exists(exe) and all(os.path.getmtime(d) <= os.path.getmtime(exe) for d in deps):
        return exe
    nvcc = _nvcc()
    common = ["-std=c++17", "-O1", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", csrc]

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        path = os.path.join(csrc, src) if src.endswith(".cu") else os.path.join(HERE, src)
        arch = ["-gencode", "arch=compute_103a,code=compute_103a"] if src.endswith(".cu") else []
        res = subprocess.run([nvcc] + arch + common + ["-c", path, "-o", obj], capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"tracer build failed on {src}:\n{res.stderr[-4000:]}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES) + len(HOST)) as ex:
        objs = list(ex.map(compile_one, SOURCES + HOST))
    cxx = shutil.which("g++") or "c++"
    res = subprocess.run([cxx, "-o", exe] + objs + ["-lpthread"], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"tracer link failed:\n{res.stderr[-4000:]}")
    return exe


def run(exe: str, commands: list[str]) -> list[dict]:
    """Run the commands; returns one record per call: the command, its launches
    (dicts of the printed fields), tensor maps, memsets and status."""
    res = subprocess.run([exe], input="\n".join(commands) + "\n", capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        raise RuntimeError(f"tracer exited with {res.returncode}:\n{res.stderr[-2000:]}")
    calls, cur = [], None
    for line in res.stdout.splitlines():
        head, _, rest = line.partition(" ")
        if head == "call":
            cur = {"cmd": rest, "launches": [], "tmaps": [], "other": [], "status": None}
            calls.append(cur)
        elif head in ("launch", "tmap"):
            fields = dict(kv.split("=", 1) for kv in rest.split())
            (cur["launches"] if head == "launch" else cur["tmaps"]).append(fields)
        elif head == "status":
            cur["status"] = int(rest)
        else:
            cur["other"].append(line)
    return calls

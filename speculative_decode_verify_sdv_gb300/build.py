"""Build libsdv.so in-tree with nvcc for sm_103a (compute_103a / sm_103a).

Each translation unit is compiled in parallel, then linked into
``speculative_decode_verify_sdv_gb300/libsdv.so`` (the CUDA runtime is
linked statically; the driver's tensor-map encoder is fetched at run time).
An object or the library is rebuilt unless a stamp beside it records the sha256
of exactly the inputs it would be built from (sources, headers, flags, the nvcc
version and the machine type), so a binary built elsewhere is never reused.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsdv.so")

SOURCES = ["api.cu", "dq_gemm.cu", "tc_gemm.cu", "gemv.cu", "small_kernels.cu", "moe_kernels.cu", "noalloc.cu",
           "ngram_drafter.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA extension cannot be built")


_NVCC_VERSION = {}


def _nvcc_version() -> str:
    exe = nvcc()
    if exe not in _NVCC_VERSION:
        _NVCC_VERSION[exe] = subprocess.run([exe, "--version"], capture_output=True, text=True).stdout
    return _NVCC_VERSION[exe]


def _digest(parts) -> str:
    """sha256 over the given byte strings / file contents (a build's inputs)."""
    h = hashlib.sha256()
    for part in parts:
        if isinstance(part, str) and os.path.isfile(part):
            with open(part, "rb") as f:
                data = f.read()
            h.update(os.path.basename(part).encode() + b"\0")
        else:
            data = part.encode() if isinstance(part, str) else part
        h.update(len(data).to_bytes(8, "little") + data)
    return h.hexdigest()


def _up_to_date(out: str, digest: str) -> bool:
    """An output is reused only when it exists and was built from inputs with this digest
    (sources, headers, flags, compiler version and machine); modification times play no part."""
    stamp = out + ".sha256"
    if not (os.path.exists(out) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == digest


def _stamp(out: str, digest: str) -> None:
    with open(out + ".sha256", "w") as f:
        f.write(digest + "\n")


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "sdv.h"))
    objs = []

    common = [_nvcc_version(), platform.machine(), " ".join(ARCH + FLAGS)] + sorted(headers)

    def compile_one(src: str) -> str:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        digest = _digest(common + [path])
        if _up_to_date(obj, digest) and not ptxas_info:
            return obj
        cmd = [nvcc()] + ARCH + FLAGS + ["-I", INCLUDE, "-I", CSRC, "-c", path, "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0 or verbose or ptxas_info:
            sys.stderr.write(res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        _stamp(obj, digest)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    link = [nvcc()] + ARCH + ["-shared", "-o", LIB] + objs + ["-cudart", "static"]
    digest = _digest([_nvcc_version(), platform.machine(), " ".join(link)] + [o + ".sha256" for o in objs])
    lib_stamp = os.path.join(BUILD, "libsdv.so")
    if not (os.path.exists(LIB) and _up_to_date(lib_stamp, digest)):
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("link of libsdv.so failed")
        open(lib_stamp, "w").close()
        _stamp(lib_stamp, digest)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))

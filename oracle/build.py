"""Build the plain C++ oracle (``oracle/src/oracle.cpp``) into ``oracle/liboracle.so``.

TEST INFRASTRUCTURE ONLY: the library is loaded by ``oracle/_native.py`` for
the tests, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``.

g++ with ``-ffp-contract=off`` (no fused multiply-add changes a rounding: one
multiply and one add per term, as the oracle's definitions state) and OpenMP
(over output rows only; every element's arithmetic is the same at any thread
count).  No BLAS, no vector intrinsics.  The library is rebuilt unless a stamp
beside it records the sha256 of the source, the flags, the compiler version and
the machine type.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "src", "oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
FLAGS = ["-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("no C++ compiler (g++) found: the oracle cannot be built")


def _digest() -> str:
    h = hashlib.sha256()
    with open(SRC, "rb") as f:
        h.update(f.read())
    ver = subprocess.run([cxx(), "--version"], capture_output=True, text=True).stdout
    h.update(" ".join(FLAGS).encode() + ver.encode() + platform.machine().encode())
    return h.hexdigest()


def build(verbose: bool = False) -> str:
    digest = _digest()
    stamp = LIB + ".sha256"
    if os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read().strip() == digest:
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cxx()] + FLAGS + ["-Wall", "-o", tmp, SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0 or verbose:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("g++ failed on the oracle")
    os.replace(tmp, LIB)  # atomic: concurrent builders never load a half-written file
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))

"""ctypes loader of the plain C++ oracle (``oracle/src/oracle.cpp``).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The Python modules of
this package only marshal numpy arrays into the C++ functions, which hold all of
the oracle's arithmetic.  The library is built on first use (``oracle/build.py``,
g++), here or on the GPU machine.

Threads: the heavy functions spread output rows over ``threads()`` OpenMP
threads (default: every core, or ``ORACLE_THREADS``); results are identical at
any thread count.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_lib = None
_lock = threading.Lock()
_threads = [0]

vp, i32, i64, u64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double

_SIGS = {
    "orc_version": ([], i32),
    "orc_max_threads": ([], i32),
    "orc_half_to_double": ([vp, i64, vp], None),
    "orc_double_to_half": ([vp, i64, vp], None),
    "orc_quantize_block32": ([vp, i64, i64, i32, vp, vp, i32], i32),
    "orc_quantize_fp4_block32": ([vp, i64, i64, vp, vp, i32], i32),
    "orc_e2m1_values": ([vp, i64, vp], None),
    "orc_e2m1_encode": ([vp, i64, vp], None),
    "orc_pack_nibbles": ([vp, i64, i64, vp], i32),
    "orc_unpack_int4": ([vp, i64, i64, vp], None),
    "orc_dequantize": ([i32, vp, vp, i64, i64, vp], None),
    "orc_dequant_gemm64": ([i32, vp, vp, i64, i64, vp, i32, vp, i32], i32),
    "orc_dequant_gemm64_x64": ([i32, vp, vp, i64, i64, vp, i32, vp, i32], i32),
    "orc_argmax_rows_f32": ([vp, i32, i64, vp], None),
    "orc_argmax_rows_f64": ([vp, i32, i64, vp], None),
    "orc_top2_gap": ([vp, i32, i64, vp], None),
    "orc_greedy_accept": ([vp, i32, vp, i32, vp, vp], i32),
    "orc_tree_accept": ([vp, i32, vp, vp, vp, vp, vp], i32),
    "orc_verify_head": ([i32, vp, vp, i64, i64, vp, i32, vp, i32, vp, vp, vp, vp, vp, i32], i32),
    "orc_silu": ([vp, i64, vp], None),
    "orc_swiglu64": ([i32, vp, vp, vp, vp, i64, i64, vp, i32, vp, vp, i32], i32),
    "orc_route_topk": ([vp, i32, i32, i32, vp, vp], i32),
    "orc_group_by_expert": ([vp, i32, i32, i32, vp, vp, vp], i32),
    "orc_expert_swiglu64": ([i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, vp, i32], i32),
    "orc_moe_forward": ([i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, i32, vp, vp, vp, i32], i32),
    "orc_mix": ([u64], u64),
    "orc_mix_array": ([vp, i64, vp], None),
    "orc_rng_key": ([u64, u64], u64),
    "orc_uniforms": ([u64, vp, i64, vp], None),
    "orc_gumbel": ([u64, i32, i64, vp], None),
    "orc_verify_sample": ([vp, i32, i64, vp, i32, dbl, u64, u64, vp, vp, vp, vp, vp, vp, vp, vp, vp], i32),
}


def lib() -> ctypes.CDLL:
    """The loaded oracle library (built on first use)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                from . import build
                path = build.build()
                h = ctypes.CDLL(path)
                for name, (args, res) in _SIGS.items():
                    f = getattr(h, name)
                    f.argtypes = args
                    f.restype = res
                _lib = h
    return _lib


def threads() -> int:
    """OpenMP threads the heavy oracle functions use."""
    if _threads[0] <= 0:
        env = os.environ.get("ORACLE_THREADS", "")
        _threads[0] = int(env) if env.isdigit() and int(env) > 0 else max(1, int(lib().orc_max_threads()))
    return _threads[0]


def set_threads(n: int) -> int:
    """Set the thread count (n <= 0: every core); returns the previous one."""
    prev = threads()
    _threads[0] = n if n > 0 else max(1, int(lib().orc_max_threads()))
    return prev


def ptr(a: np.ndarray):
    """Pointer to a C-contiguous array's data (None passes NULL)."""
    if a is None:
        return None
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle arrays must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def as_c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def half_bits(a) -> np.ndarray:
    """fp16 array -> its uint16 bit patterns (C-contiguous)."""
    return np.ascontiguousarray(np.asarray(a, dtype=np.float16)).view(np.uint16)


def code_kind(codes: np.ndarray):
    """(kind, C-contiguous codes) for the C++ GEMM: int8 -> 0 (integer codes),
    uint8 -> 1 (E2M1 codes, one per byte, 0..15), float64 -> 2 (the values)."""
    c = np.asarray(codes)
    if c.dtype == np.int8:
        return 0, np.ascontiguousarray(c)
    if c.dtype == np.uint8:
        if c.size and int(c.max()) > 15:
            raise ValueError("uint8 codes are E2M1 codes (0..15), one per byte")
        return 1, np.ascontiguousarray(c)
    return 2, np.ascontiguousarray(c, dtype=np.float64)


def check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle: invalid arguments to {what}")

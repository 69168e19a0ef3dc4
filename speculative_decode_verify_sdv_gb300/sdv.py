"""Thin Python binding of libsdv (include/sdv.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch
tensors where the C function takes device pointers.  All arithmetic happens
in the library's CUDA kernels; there is no Python or CPU fallback: if the
shared library is missing or a GPU is absent the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdv.so")

SDV_OK, SDV_ERR_INVALID_ARG, SDV_ERR_UNSUPPORTED, SDV_ERR_CUDA, SDV_ERR_TIMEOUT, SDV_ERR_WORKSPACE = range(6)
SDV_Q8, SDV_Q4, SDV_F4 = 8, 4, 2
SDV_OP_QLINEAR, SDV_OP_QLINEAR_SWIGLU, SDV_OP_VERIFY_HEAD, SDV_OP_MOE, SDV_OP_VERIFY_SAMPLE = 1, 2, 3, 4, 5

EXPORTED = (
    "sdv_quantize_block32", "sdv_qlinear", "sdv_qlinear_swiglu", "sdv_verify_head",
    "sdv_greedy_accept", "sdv_moe_gather_qmm", "sdv_workspace_bytes", "sdv_workspace_init",
    "sdv_last_device_status", "sdv_device_status", "sdv_noalloc_device_status", "sdv_status_string", "sdv_version", "sdv_launch_count", "sdv_verify_head_noalloc", "sdv_set_gemm_path",
    "sdv_moe_route", "sdv_verify_sample", "sdv_tree_accept", "sdv_debug_fault",
    "sdv_ngram_create", "sdv_ngram_destroy", "sdv_ngram_append", "sdv_ngram_propose",
)


class SdvError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} ({status})")
        self.status = status


class sdv_qweight(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int32), ("n", ctypes.c_int32), ("k", ctypes.c_int32),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libsdv.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libsdv.so not found at {LIB_PATH}; run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    qw = ctypes.POINTER(sdv_qweight)
    sig = {
        "sdv_quantize_block32": ([vp, i32, i32, i32, vp, vp, vp], i32),
        "sdv_qlinear": ([qw, vp, i32, vp, vp, sz, vp], i32),
        "sdv_qlinear_swiglu": ([qw, qw, vp, i32, vp, vp, sz, vp], i32),
        "sdv_verify_head": ([qw, vp, i32, vp, i32, vp, vp, vp, vp, vp, sz, vp], i32),
        "sdv_verify_head_noalloc": ([qw, vp, i32, vp, i32, vp, vp, vp, vp, vp], i32),
        "sdv_verify_sample": ([qw, vp, i32, vp, i32, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64, vp, vp, vp,
                               vp, vp, sz, vp], i32),
        "sdv_greedy_accept": ([vp, i32, vp, i32, vp, vp, vp], i32),
        "sdv_tree_accept": ([vp, i32, vp, vp, vp, vp, vp, vp], i32),
        "sdv_moe_gather_qmm": ([qw, qw, qw, i32, i32, i32, i32, vp, vp, i32, vp, vp, vp, vp, sz, vp], i32),
        "sdv_moe_route": ([vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp], i32),
        "sdv_workspace_bytes": ([i32, i32, i32, i32, i32, i32], sz),
        "sdv_workspace_init": ([vp, sz, vp], i32),
        "sdv_last_device_status": ([vp, vp], i32),
        "sdv_device_status": ([vp, vp], i32),
        "sdv_noalloc_device_status": ([vp], i32),
        "sdv_status_string": ([i32], ctypes.c_char_p),
        "sdv_version": ([], i32),
        "sdv_launch_count": ([], ctypes.c_uint64),
        "sdv_set_gemm_path": ([i32], i32),
        "sdv_debug_fault": ([i32, ctypes.c_uint64], i32),
        "sdv_ngram_create": ([i32, ctypes.POINTER(vp)], i32),
        "sdv_ngram_destroy": ([vp], i32),
        "sdv_ngram_append": ([vp, vp, i32], i32),
        "sdv_ngram_propose": ([vp, i32, vp, ctypes.POINTER(i32)], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != SDV_OK:
        raise SdvError(fn, status, load().sdv_status_string(status).decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _want(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class QWeight:
    """A per-block-32 quantised weight: codes (int8 [n, k] or uint8 [n, k/2]),
    fp16 scales [n, k/32], on the GPU."""

    def __init__(self, codes: torch.Tensor, scales: torch.Tensor, bits: int, n: int, k: int):
        self.codes, self.scales, self.bits, self.n, self.k = codes, scales, bits, n, k

    def c(self) -> sdv_qweight:
        return sdv_qweight(self.bits, self.n, self.k, _ptr(self.codes), _ptr(self.scales))


def sdv_launch_count() -> int:
    """Kernels the library has launched in this process (see the header)."""
    return int(load().sdv_launch_count())


def sdv_version() -> int:
    return int(load().sdv_version())


SDV_PATH_AUTO, SDV_PATH_MMA_SYNC, SDV_PATH_TCGEN05, SDV_PATH_GEMV = 0, 1, 2, 3


def sdv_set_gemm_path(path: int) -> int:
    """Select the GEMM implementation (0 auto, 1 mma.sync, 2 tcgen05, 3 CUDA-core GEMV for S <= 2);
    returns the previous one."""
    prev = int(load().sdv_set_gemm_path(path))
    if prev < 0:
        raise ValueError(f"invalid GEMM path {path}")
    return prev


def sdv_debug_fault(withhold_stage: int, wait_limit_ns: int) -> None:
    """Timeout-path test hook: withhold one weight stage of every tcgen05 launch
    and shorten the bounded waits (-1, 0 switches it off)."""
    _check("sdv_debug_fault", load().sdv_debug_fault(withhold_stage, wait_limit_ns))


def sdv_status_string(status: int) -> str:
    return load().sdv_status_string(status).decode()


def sdv_workspace_bytes(op: int, n: int, k: int, S: int, E: int = 0, top_k: int = 0) -> int:
    return int(load().sdv_workspace_bytes(op, n, k, S, E, top_k))


def sdv_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("sdv_workspace_init", load().sdv_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sdv_last_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return (and clear) the workspace's device status."""
    return int(load().sdv_last_device_status(_ptr(ws), _stream(stream)))


def sdv_device_status(ws: torch.Tensor, stream=None) -> int:
    """The same as ``sdv_last_device_status`` (the earlier name)."""
    return int(load().sdv_device_status(_ptr(ws), _stream(stream)))


def sdv_noalloc_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the status of the no-workspace head's fixed scratch."""
    return int(load().sdv_noalloc_device_status(_stream(stream)))


def sdv_quantize_block32(w: torch.Tensor, bits: int, codes: torch.Tensor, scales: torch.Tensor,
                         stream=None) -> None:
    _want(w, torch.float32, "w")
    _want(scales, torch.float16, "scales")
    n, k = w.shape
    _check("sdv_quantize_block32", load().sdv_quantize_block32(
        _ptr(w), n, k, bits, _ptr(codes), _ptr(scales), _stream(stream)))


def sdv_qlinear(w: QWeight, x: torch.Tensor, S: int, y: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    _want(x, torch.float16, "x")
    _want(y, torch.float32, "y")
    cw = w.c()
    _check("sdv_qlinear", load().sdv_qlinear(ctypes.byref(cw), _ptr(x), S, _ptr(y), _ptr(ws),
                                             ws.numel() * ws.element_size(), _stream(stream)))


def sdv_qlinear_swiglu(gate: QWeight, up: QWeight, x: torch.Tensor, S: int, h: torch.Tensor,
                       ws: torch.Tensor, stream=None) -> None:
    _want(x, torch.float16, "x")
    _want(h, torch.float16, "h")
    cg, cu = gate.c(), up.c()
    _check("sdv_qlinear_swiglu", load().sdv_qlinear_swiglu(
        ctypes.byref(cg), ctypes.byref(cu), _ptr(x), S, _ptr(h), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def sdv_verify_head(head: QWeight, x: torch.Tensor, S: int, drafts, n_valid: int, logits,
                    argmax: torch.Tensor, accepted: torch.Tensor, next_a0: torch.Tensor,
                    ws: torch.Tensor, stream=None) -> None:
    _want(x, torch.float16, "x")
    _want(drafts, torch.int32, "drafts")
    _want(logits, torch.float32, "logits")
    for t, nm in ((argmax, "argmax"), (accepted, "accepted"), (next_a0, "next_a0")):
        _want(t, torch.int32, nm)
    cw = head.c()
    _check("sdv_verify_head", load().sdv_verify_head(
        ctypes.byref(cw), _ptr(x), S, _ptr(drafts), n_valid, _ptr(logits), _ptr(argmax),
        _ptr(accepted), _ptr(next_a0), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sdv_verify_sample(head: QWeight, x: torch.Tensor, S: int, drafts, n_valid: int, temperature: float,
                      seed: int, counter: int, logits, samples: torch.Tensor, accepted: torch.Tensor,
                      next_token: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    _want(x, torch.float16, "x")
    _want(drafts, torch.int32, "drafts")
    _want(logits, torch.float32, "logits")
    for t, nm in ((samples, "samples"), (accepted, "accepted"), (next_token, "next_token")):
        _want(t, torch.int32, nm)
    cw = head.c()
    _check("sdv_verify_sample", load().sdv_verify_sample(
        ctypes.byref(cw), _ptr(x), S, _ptr(drafts), n_valid, float(temperature), seed % 2**64, counter % 2**64,
        _ptr(logits), _ptr(samples), _ptr(accepted), _ptr(next_token), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def sdv_verify_head_noalloc(head: QWeight, x: torch.Tensor, S: int, drafts, n_valid: int, logits,
                            argmax: torch.Tensor, accepted: torch.Tensor, next_a0: torch.Tensor,
                            stream=None) -> None:
    """sdv_verify_head with the library's own fixed device scratch (no workspace)."""
    _want(x, torch.float16, "x")
    _want(drafts, torch.int32, "drafts")
    _want(logits, torch.float32, "logits")
    for t, nm in ((argmax, "argmax"), (accepted, "accepted"), (next_a0, "next_a0")):
        _want(t, torch.int32, nm)
    cw = head.c()
    _check("sdv_verify_head_noalloc", load().sdv_verify_head_noalloc(
        ctypes.byref(cw), _ptr(x), S, _ptr(drafts), n_valid, _ptr(logits), _ptr(argmax),
        _ptr(accepted), _ptr(next_a0), _stream(stream)))


def sdv_tree_accept(argmax: torch.Tensor, S: int, tokens, parent, path, accepted: torch.Tensor,
                    next_a0: torch.Tensor, stream=None) -> None:
    for t, nm in ((argmax, "argmax"), (tokens, "tokens"), (parent, "parent"), (path, "path"),
                  (accepted, "accepted"), (next_a0, "next_a0")):
        _want(t, torch.int32, nm)
    _check("sdv_tree_accept", load().sdv_tree_accept(
        _ptr(argmax), S, _ptr(tokens), _ptr(parent), _ptr(path), _ptr(accepted), _ptr(next_a0), _stream(stream)))


def sdv_greedy_accept(argmax: torch.Tensor, S: int, drafts, n_valid: int, accepted: torch.Tensor,
                      next_a0: torch.Tensor, stream=None) -> None:
    for t, nm in ((argmax, "argmax"), (drafts, "drafts"), (accepted, "accepted"), (next_a0, "next_a0")):
        _want(t, torch.int32, nm)
    _check("sdv_greedy_accept", load().sdv_greedy_accept(
        _ptr(argmax), S, _ptr(drafts), n_valid, _ptr(accepted), _ptr(next_a0), _stream(stream)))


def sdv_moe_gather_qmm(gate: QWeight, up: QWeight, down: QWeight, E: int, I: int, H: int, top_k: int,
                       x: torch.Tensor, router_logits: torch.Tensor, S: int, out: torch.Tensor,
                       topk_ids, topk_w, ws: torch.Tensor, stream=None) -> None:
    _want(x, torch.float16, "x")
    _want(router_logits, torch.float32, "router_logits")
    _want(out, torch.float32, "out")
    cg, cu, cd = gate.c(), up.c(), down.c()
    _check("sdv_moe_gather_qmm", load().sdv_moe_gather_qmm(
        ctypes.byref(cg), ctypes.byref(cu), ctypes.byref(cd), E, I, H, top_k, _ptr(x),
        _ptr(router_logits), S, _ptr(out), _ptr(topk_ids), _ptr(topk_w), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def sdv_moe_route(router_logits: torch.Tensor, S: int, E: int, top_k: int, ids: torch.Tensor,
                  weights: torch.Tensor, offsets: torch.Tensor, pair_rows: torch.Tensor,
                  n_hit: torch.Tensor, hit: torch.Tensor, stream=None) -> None:
    _want(router_logits, torch.float32, "router_logits")
    _want(weights, torch.float32, "weights")
    for t, nm in ((ids, "ids"), (offsets, "offsets"), (pair_rows, "pair_rows"), (n_hit, "n_hit"), (hit, "hit")):
        _want(t, torch.int32, nm)
    _check("sdv_moe_route", load().sdv_moe_route(
        _ptr(router_logits), S, E, top_k, _ptr(ids), _ptr(weights), _ptr(offsets), _ptr(pair_rows),
        _ptr(n_hit), _ptr(hit), _stream(stream)))


# ---- host n-gram drafter (host pointers; no GPU involved) -------------------------

def sdv_ngram_create(m: int) -> int:
    """A native drafter of order m; returns its opaque handle."""
    h = ctypes.c_void_p()
    _check("sdv_ngram_create", load().sdv_ngram_create(m, ctypes.byref(h)))
    return h.value


def sdv_ngram_destroy(handle: int) -> None:
    _check("sdv_ngram_destroy", load().sdv_ngram_destroy(ctypes.c_void_p(handle)))


def sdv_ngram_append(handle: int, tokens) -> None:
    arr = (ctypes.c_int32 * len(tokens))(*[int(t) for t in tokens])
    _check("sdv_ngram_append", load().sdv_ngram_append(ctypes.c_void_p(handle), arr, len(tokens)))


def sdv_ngram_propose(handle: int, k: int) -> list[int]:
    """Up to k drafts continuing the stream's last m tokens (empty when none)."""
    buf = (ctypes.c_int32 * max(k, 1))()
    count = ctypes.c_int32(0)
    _check("sdv_ngram_propose", load().sdv_ngram_propose(ctypes.c_void_p(handle), k, buf, ctypes.byref(count)))
    return list(buf[:count.value])


# ---- small allocation helpers (torch owns the memory) ---------------------------

def workspace(op: int, n: int, k: int, S: int, E: int = 0, top_k: int = 0, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the size the operation needs."""
    nbytes = max(sdv_workspace_bytes(op, n, k, S, E, top_k), 256)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def quantize(w: torch.Tensor, bits: int) -> QWeight:
    """Quantise an fp32 [n, k] CUDA tensor with sdv_quantize_block32."""
    n, k = w.shape
    codes = torch.empty((n, k if bits == 8 else k // 2), dtype=torch.int8 if bits == 8 else torch.uint8,
                        device=w.device)
    scales = torch.empty((n, k // 32), dtype=torch.float16, device=w.device)
    sdv_quantize_block32(w.contiguous(), bits, codes, scales)
    return QWeight(codes, scales, bits, n, k)

"""Helpers shared by the GPU parity tests: moving seeded inputs to the device,
running the oracle on the same bytes, and the comparison rules.

Comparison rules (from the stated tolerances):
* fp32 outputs of a dequantised GEMM (logits, Y): max |gpu - oracle| <=
  2e-3 * sqrt(K / 256) * RMS(oracle), K the reduction length;
* an argmax (and the accept decisions that read it) must be bit-exact on every
  row whose oracle top-2 gap exceeds 1e-2;
* integer outputs of integer steps (codes, accept on a given argmax) are
  bit-exact.
"""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import quant, verify

GAP = 1e-2


def tol(k: int) -> float:
    return 2e-3 * float(np.sqrt(k / 256.0))


def to_dev_f16(a: np.ndarray, dev="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a.astype(np.float16))
    return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.float16)


def to_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def oracle_weight(w: np.ndarray, bits: int):
    """Oracle quantisation: (unpacked codes, scales fp16, stored codes).

    bits 8 / 4: integer codes (int8); bits 2: FP4 -- the unpacked codes are the
    E2M1 codes, one per byte (uint8, which the oracle's GEMM reads as E2M1),
    the stored codes the packed nibbles."""
    if bits == 2:
        c4, scales = quant.quantize_fp4_block32(w)
        return c4, scales, quant.pack_nibbles(c4)
    codes, scales = quant.quantize_block32(w, bits)
    stored = codes if bits == 8 else quant.pack_int4(codes)
    return codes, scales, stored


def device_weight(stored: np.ndarray, scales: np.ndarray, bits: int, n: int, k: int, dev="cuda"):
    from speculative_decode_verify_sdv_gb300 import sdv
    codes_t = to_dev(stored.view(np.int8) if bits == 8 else stored.view(np.uint8), dev)
    scales_t = torch.from_numpy(np.ascontiguousarray(scales.view(np.int16))).to(dev).view(torch.float16)
    return sdv.QWeight(codes_t, scales_t, bits, n, k)


def assert_gemm_close(y_gpu: np.ndarray, y_orc: np.ndarray, k: int, what: str = "output"):
    y_orc = np.asarray(y_orc, dtype=np.float64)
    rms = float(np.sqrt(np.mean(y_orc ** 2)))
    err = float(np.max(np.abs(np.asarray(y_gpu, dtype=np.float64) - y_orc)))
    bound = tol(k) * rms
    assert err <= bound, f"{what}: max abs error {err:.3e} > {bound:.3e} (rms {rms:.3e})"
    return err / rms if rms > 0 else 0.0


def check_head_outputs(ref: dict, am: np.ndarray, acc: int, nxt: int):
    """argmax exact on eligible rows; accept/next_a0 exact when every row the
    accept scan read (rows 0..accepted) is eligible.  Returns #eligible rows."""
    elig = ref["gap"] > GAP
    np.testing.assert_array_equal(am[elig], ref["argmax"][elig])
    j = ref["accepted"]
    if elig[: j + 1].all():
        assert acc == j, f"accepted {acc} != {j}"
        assert nxt == ref["next_a0"], f"next_a0 {nxt} != {ref['next_a0']}"
    return int(elig.sum())


PATHS = {"mma": 1, "tc": 2, "gemv": 3}


class gemm_path:
    """Context manager selecting the GEMM implementation (sdv_set_gemm_path)."""

    def __init__(self, name: str):
        self.path = PATHS[name] if isinstance(name, str) else int(name)

    def __enter__(self):
        from speculative_decode_verify_sdv_gb300 import sdv
        self.prev = sdv.sdv_set_gemm_path(self.path)
        return self

    def __exit__(self, *a):
        from speculative_decode_verify_sdv_gb300 import sdv
        sdv.sdv_set_gemm_path(self.prev)


def run_head(head, x: np.ndarray, drafts: np.ndarray, n_valid: int, want_logits=True, ws=None):
    from speculative_decode_verify_sdv_gb300 import sdv
    S = x.shape[0]
    dev = head.codes.device
    xt = to_dev_f16(x, dev)
    dt = to_dev(np.asarray(drafts, dtype=np.int32), dev) if S > 1 else torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.full((S, head.n), float("nan"), dtype=torch.float32, device=dev) if want_logits else None
    am = torch.full((S,), -1, dtype=torch.int32, device=dev)
    acc = torch.full((1,), -1, dtype=torch.int32, device=dev)
    nxt = torch.full((1,), -1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = sdv.workspace(sdv.SDV_OP_VERIFY_HEAD, head.n, head.k, S, device=dev)
    sdv.sdv_verify_head(head, xt, S, dt, n_valid, logits, am, acc, nxt, ws)
    assert sdv.sdv_last_device_status(ws) == sdv.SDV_OK
    return (logits.cpu().numpy() if want_logits else None, am.cpu().numpy(), int(acc.item()),
            int(nxt.item()))


GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_windows(prefix: str, name: str, S: int):
    """(header dict, window records) of tests/golden/<prefix>_<name>_s<S>.jsonl, a
    file of the oracle's per-window results written by a committed generator
    that calls only oracle/ (make_head_windows.py, make_mlp_windows.py)."""
    import json
    head, recs = {}, []
    with open(os.path.join(GOLDEN_DIR, f"{prefix}_{name}_s{S}.jsonl")) as f:
        for line in f:
            if line.startswith("#"):
                if ":" in line:
                    k, v = line[1:].split(":", 1)
                    head[k.strip()] = v.strip()
            elif line.strip():
                recs.append(json.loads(line))
    return head, recs

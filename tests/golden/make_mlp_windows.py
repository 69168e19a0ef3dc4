"""Write the oracle's per-window scales of the 27B-shaped SwiGLU projection.

    python tests/golden/make_mlp_windows.py

For every seeded window of the mlp27 workload (gate/up 17408 x 5120 int8,
S = 1, 9, 17) this calls only the oracle (``oracle/``, the plain C++
implementation) on the inputs ``synth`` generates and stores the RMS of the
oracle's float64 gate and up projections g = x G^T and u = x U^T over the
whole [S, 17408] output.  They set the tolerance of the GPU's h = fp16(SiLU(g) u)
in the all-windows parity test, which compares sampled elements of every
window against the oracle evaluated one by one and the whole output on every
tenth window.  Nothing here comes from the GPU.
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from oracle import quant, verify  # noqa: E402
from synth import workloads as W  # noqa: E402

S_LIST = (1, 9, 17)


def path_of(S: int) -> str:
    return os.path.join(HERE, f"mlp_windows_mlp27_s{S}.jsonl")


def main():
    with open(os.path.join(ROOT, "oracle", "src", "oracle.cpp"), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    wl = W.MLP27
    t0 = time.time()
    cg, sg = quant.quantize_block32(W.mlp_weights(wl, "gate"), wl.bits)
    cu, su = quant.quantize_block32(W.mlp_weights(wl, "up"), wl.bits)
    for S in S_LIST:
        lines = [f"# oracle per-window scales: workload mlp27 (gate/up {wl.inter} x {wl.h} int8), S = {S}, "
                 f"{wl.windows} windows: RMS of the float64 g = x G^T and u = x U^T",
                 f"# oracle_sha256: {sha}",
                 "# written by tests/golden/make_mlp_windows.py (calls oracle/ only)"]
        for win in range(wl.windows):
            x = W.activations(wl, win, S)
            g = verify.dequant_gemm64(x, cg, sg)
            u = verify.dequant_gemm64(x, cu, su)
            lines.append(json.dumps({"window": win, "rms_g": float(np.sqrt(np.mean(g * g))),
                                     "rms_u": float(np.sqrt(np.mean(u * u)))}, separators=(",", ":")))
        with open(path_of(S), "w") as f:
            f.write("\n".join(lines) + "\n")
        print(f"mlp27 S={S}: {wl.windows} windows, {time.time() - t0:.0f} s", flush=True)


if __name__ == "__main__":
    main()

"""Write the oracle's per-window results of the full-size verify heads.

    python tests/golden/make_head_windows.py [q4b|a3b ...]

For every seeded window of the Qwen3-4B-shaped head (151936 x 2560 int8, S = 9)
and the 35B-A3B-shaped head (248320 x 2048 int4, S = 1, 2, 9, 17), this calls
only the oracle (``oracle/``, the plain C++ implementation) on the inputs
``synth`` generates, and stores what the GPU parity tests compare against:

* the argmax of every window row (float32 logits, lowest index on ties),
* every row's top-2 gap (float64 logits), which decides whether the row's
  argmax must match exactly (gap > 1e-2),
* the drafts of the window (draft rule: j ~ U{0..S-1}, the first j drafts copy
  the oracle's argmax chain, the rest uniform ids; n_valid = S - 1),
* the accepted count and next a0 of the greedy accept.

One JSON object per window after '#' header lines naming the workload, the
oracle source's sha256 and the generator.  Nothing here comes from the GPU.
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

CASES = {"q4b": (W.Q4B, (9,)), "a3b": (W.A3B, (1, 2, 9, 17))}


def path_of(name: str, S: int) -> str:
    return os.path.join(HERE, f"head_windows_{name}_s{S}.jsonl")


def oracle_sha() -> str:
    with open(os.path.join(ROOT, "oracle", "src", "oracle.cpp"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def quantized(wl):
    w = W.head_weights(wl)
    codes, scales = quant.quantize_block32(w, wl.bits)
    return codes, scales


def window_record(wl, codes, scales, S: int, win: int) -> dict:
    x = W.activations(wl, win, S)
    ref = verify.verify_head(x, codes, scales, np.zeros(max(S - 1, 0), np.int32), 0)
    drafts, n_valid = W.drafts(wl, win, S, ref["argmax"])
    acc, nxt = verify.greedy_accept(ref["argmax"], drafts, n_valid)
    return {"window": win, "argmax": [int(v) for v in ref["argmax"]],
            "gap": [float("%.9g" % g) for g in ref["gap"]], "drafts": [int(d) for d in drafts],
            "n_valid": int(n_valid), "accepted": int(acc), "next_a0": int(nxt)}


def main(names):
    sha = oracle_sha()
    for name in names:
        wl, s_list = CASES[name]
        t0 = time.time()
        codes, scales = quantized(wl)
        for S in s_list:
            lines = [f"# oracle per-window results: workload {wl.name} ({wl.n} x {wl.h}, "
                     f"{'int8' if wl.bits == 8 else 'int4'}), S = {S}, {wl.windows} windows",
                     f"# oracle_sha256: {sha}",
                     "# written by tests/golden/make_head_windows.py (calls oracle/ only)"]
            for win in range(wl.windows):
                lines.append(json.dumps(window_record(wl, codes, scales, S, win), separators=(",", ":")))
            with open(path_of(name, S), "w") as f:
                f.write("\n".join(lines) + "\n")
            print(f"{name} S={S}: {wl.windows} windows, {time.time() - t0:.0f} s", flush=True)


def load(name: str, S: int):
    """(header dict, list of window records) of a stored file."""
    head, recs = {}, []
    with open(path_of(name, S)) as f:
        for line in f:
            if line.startswith("#"):
                if ":" in line and "sha256" in line:
                    k, v = line[1:].split(":", 1)
                    head[k.strip()] = v.strip()
            elif line.strip():
                recs.append(json.loads(line))
    return head, recs


if __name__ == "__main__":
    main(sys.argv[1:] or list(CASES))

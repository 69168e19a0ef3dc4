"""Pins for the oracle's FP4 (E2M1) weight quantisation (CPU only).

* the 16 codes decode to the OCP Microscaling E2M1 values;
* encoding is the nearest E2M1 value by exhaustive search, ties to the even
  mantissa bit, saturating beyond 6, zero always +0;
* hand-worked blocks (tests/golden/fp4_block32_worked.txt);
* per-block scale = fp16(max|w| / 6); the block maximum maps to +-6.
"""
import os

import numpy as np
import pytest

from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp4_block32_worked.txt")


def test_decode_table():
    vals = quant.decode_e2m1(np.arange(16))
    assert vals.tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]


def _brute(r):
    """Nearest E2M1 magnitude by exhaustive search; a tie between neighbours
    goes to the one whose mantissa bit is 0 (even index in the E2M1 table)."""
    a = min(abs(float(r)), 6.0)
    d = np.abs(quant.E2M1 - a)
    cands = [i for i in range(8) if d[i] == d.min()]
    idx = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
    return idx | (8 if float(r) < 0 and idx > 0 else 0)


def test_encode_matches_brute_force():
    rng = np.random.default_rng(0)
    r = np.concatenate([rng.uniform(-8, 8, 20000).astype(np.float32),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, -0.25, -0.75, -5.0,
                                  0.0, -0.0, 1e-30, -1e-30], np.float32)])
    got = quant.encode_e2m1(r)
    want = np.array([_brute(v) for v in r], np.uint8)
    assert np.array_equal(got, want)


def test_round_trip_of_grid_values():
    for s in (np.float16(0.01), np.float16(1.0), np.float16(3.0)):
        c = np.arange(16, dtype=np.uint8)
        c[8] = 0                                  # -0 encodes as +0
        w = (quant.decode_e2m1(c) * float(s)).astype(np.float32)
        r = w / np.float32(s)
        assert np.array_equal(quant.encode_e2m1(r), c)


def _golden():
    blocks, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":") if ":" in line else (line, "", "")
        if line.startswith("block"):
            cur = {"name": line.split()[1]}
            blocks.append(cur)
        else:
            cur[key.strip()] = val.strip()
    return blocks


def test_golden_blocks():
    blocks = _golden()
    assert len(blocks) >= 2
    for b in blocks:
        w = np.array([eval(t) for t in b["w"].split()], dtype=np.float32)[None, :]
        codes, scales = quant.quantize_fp4_block32(w)
        assert int(scales.view(np.uint16)[0, 0]) == int(b["scale"], 16), b["name"]
        assert codes[0].tolist() == [int(t) for t in b["codes"].split()], b["name"]


def test_block_max_maps_to_six():
    rng = np.random.default_rng(1)
    w = rng.normal(0, 0.02, (64, 256)).astype(np.float32)
    codes, scales = quant.quantize_fp4_block32(w)
    v = quant.decode_e2m1(codes).reshape(64, 8, 32)
    assert np.all(np.max(np.abs(v), axis=2) >= 4.0)     # max |w| / s16 is 6 up to the fp16 rounding of s
    err = np.abs(v * scales.astype(np.float64)[:, :, None] - w.reshape(64, 8, 32))
    assert np.all(err <= scales.astype(np.float64)[:, :, None] * 1.0 + 1e-12)   # half the widest E2M1 gap (2)

"""Planted mistakes in the oracle (CPU only).

Each case below puts one plausible bug into the oracle -- a stand-in for one of
its functions, patched into the oracle module for the length of one test -- and
runs the pins of that function (the tests in tests/test_oracle_*.py, called as
they are).  At least one pin must fail on every planted bug: a set of pins that
let one through would not pin the function.  The bugs are the kinds of mistake
that the pins are there to catch: a dropped term or factor, a wrong sign, an
index off by one, a transposed operand or result, a wrong tie rule, a skipped
rounding, a swapped operand pair.
"""
import functools

import numpy as np
import pytest

import tests.test_oracle_accept as pins_accept
import tests.test_oracle_fp4 as pins_fp4
import tests.test_oracle_gemm as pins_gemm
import tests.test_oracle_mlp as pins_mlp
import tests.test_oracle_quant as pins_quant
import tests.test_oracle_sample as pins_sample
import tests.test_oracle_tree as pins_tree
from oracle import mlp, quant, sample, verify

# ---- the dequantised GEMM -----------------------------------------------------------


def gemm_block_off_by_one(real):
    # weight k takes the scale of block k // 32 + 1 (the last block wraps to 0)
    return lambda x, c, s: real(x, c, np.roll(np.asarray(s), -1, axis=1))


def gemm_scale_dropped(real):
    return lambda x, c, s: real(x, c, np.ones_like(np.asarray(s)))


def gemm_sign_flipped(real):
    return lambda x, c, s: -real(x, c, s)


def gemm_last_term_dropped(real):
    def f(x, c, s):
        x2 = np.array(x, copy=True)
        x2[:, -1] = 0
        return real(x2, c, s)
    return f


def gemm_result_transposed(real):
    # y[i, j] written where y[j, i] belongs, read back in the caller's shape
    def f(x, c, s):
        y = real(x, c, s)
        return np.ascontiguousarray(y.T).reshape(y.shape)
    return f


def gemm_row_off_by_one(real):
    # window row i computed from activation row i + 1 (the last row repeated)
    def f(x, c, s):
        x = np.asarray(x)
        idx = np.minimum(np.arange(x.shape[0]) + 1, x.shape[0] - 1)
        return real(np.ascontiguousarray(x[idx]), c, s)
    return f


GEMM_PINS = [pins_gemm.test_integer_gemm_unit_scales_is_exact,
             pins_gemm.test_power_of_two_block_scales_pin_the_block_index,
             pins_gemm.test_one_hot_returns_dequantised_column, pins_gemm.test_operands_not_transposed,
             pins_gemm.test_random_against_exact_rationals, pins_gemm.test_window_equals_single_rows,
             pins_gemm.test_int4_dequant_uses_unpacked_codes]

# ---- argmax -------------------------------------------------------------------------


def argmax_ties_to_last(real):
    def f(l):
        l = np.asarray(l)
        return (l.shape[1] - 1 - np.argmax(l[:, ::-1], axis=1)).astype(np.int32)
    return f


def argmax_tail_dropped(real):
    # the scan stops one entry short of the row's end
    return lambda l: real(np.ascontiguousarray(np.asarray(l)[:, :-1]))


def top2_second_distinct(real):
    # the second largest taken over the values below the maximum, so a
    # duplicated maximum no longer gives a gap of 0
    def f(l):
        l = np.asarray(l, np.float64)
        out = []
        for row in l:
            m = row.max()
            below = row[row < m]
            out.append(m - below.max() if below.size else 0.0)
        return np.array(out)
    return f


ARGMAX_PINS = [pins_gemm.test_argmax_brute_force_and_ties]
TOP2_PINS = [pins_gemm.test_top2_gap]

# ---- greedy accept ------------------------------------------------------------------


def accept_next_off_by_one(real):
    def f(am, d, n_valid):
        j, _ = real(am, d, n_valid)
        am = np.asarray(am)
        return j, int(am[min(j + 1, len(am) - 1)])
    return f


def accept_pads(real):
    # every draft slot treated as real, whatever n_valid says
    def f(am, d, n_valid):
        nd = 0 if d is None else len(d)
        return real(am, d, min(len(np.asarray(am)) - 1, nd))
    return f


def accept_shifted_compare(real):
    # draft i compared with the prediction of row i + 1
    def f(am, d, n_valid):
        am = np.asarray(am)
        j = n_valid
        for i in range(n_valid):
            if i + 1 >= len(am) or int(d[i]) != int(am[i + 1]):
                j = i
                break
        return j, int(am[j])
    return f


def accept_keeps_the_miss(real):
    # the first mismatching draft is counted as accepted
    def f(am, d, n_valid):
        j, _ = real(am, d, n_valid)
        j = min(j + 1, n_valid)
        return j, int(np.asarray(am)[j])
    return f


ACCEPT_PINS = ([functools.partial(pins_accept.test_accept_exhaustive_tiny, s) for s in (2, 3, 4)] +
               [pins_accept.test_all_drafts_match_gives_bonus, pins_accept.test_first_mismatch_at_zero,
                pins_accept.test_pads_are_never_accepted, pins_accept.test_off_by_one_drafter_accepts_nothing])

# ---- tree accept --------------------------------------------------------------------


def tree_as_chain(real):
    # the parent links ignored: node i taken as the child of node i - 1
    def f(am, tokens, parent):
        s = len(np.asarray(am))
        return real(am, tokens, np.array([-1] + list(range(s - 1))) if s > 1 else parent)
    return f


def tree_compares_own_row(real):
    # a node's token compared with its own row's prediction, not its parent's
    def f(am, tokens, parent):
        am = np.asarray(am)
        s = len(am)
        ok, depth = [True] + [False] * (s - 1), [0] * s
        for i in range(1, s):
            p = int(parent[i])
            if 0 <= p < i and ok[p] and int(tokens[i]) == int(am[i]):
                ok[i], depth[i] = True, depth[p] + 1
        best = min((i for i in range(s) if ok[i]), key=lambda i: (-depth[i], i))
        path, j = [], best
        while j != 0:
            path.append(j)
            j = int(parent[j])
        return path[::-1], int(am[best])
    return f


TREE_PINS = [pins_tree.test_random_trees_match_independent_statement, pins_tree.test_deeper_branch_wins,
             functools.partial(pins_tree.test_chain_equals_greedy, 3)]

# ---- SwiGLU and the MoE router ------------------------------------------------------


def silu_sign_error(real):
    return lambda t: np.asarray(t, np.float64) / (1.0 + np.exp(np.asarray(t, np.float64)))


def swiglu_gate_up_swapped(real):
    return lambda x, gq, gs, uq, us: real(x, uq, us, gq, gs)


def route_ties_to_higher_id(real):
    def f(r, k):
        r = np.asarray(r)
        ids, w = real(np.ascontiguousarray(r[:, ::-1]), k)
        return r.shape[1] - 1 - ids, w
    return f


def route_softmax_over_all_experts(real):
    # the top-k weights taken from the softmax over every expert (not renormalised)
    def f(r, k):
        ids, _ = real(r, k)
        r64 = np.asarray(r, np.float64)
        e = np.exp(r64 - r64.max(axis=1, keepdims=True))
        return ids, np.take_along_axis(e / e.sum(axis=1, keepdims=True), ids, axis=1)
    return f


def group_rows_reversed(real):
    # an expert's selections listed in decreasing row order
    def f(ids, e):
        off, rows, slots = real(ids, e)
        rows, slots = rows.copy(), slots.copy()
        for x in range(e):
            a, b = int(off[x]), int(off[x + 1])
            rows[a:b], slots[a:b] = rows[a:b][::-1], slots[a:b][::-1]
        return off, rows, slots
    return f


def group_offsets_inclusive(real):
    # the offsets taken from an inclusive scan of the counts
    def f(ids, e):
        off, rows, slots = real(ids, e)
        return np.append(off[1:], off[-1]).astype(np.int32), rows, slots
    return f


# ---- quantisers ---------------------------------------------------------------------


def quant_ties_away_from_zero(real):
    def f(w, bits):
        codes, scales = real(w, bits)
        q = 127 if bits == 8 else 7
        s = np.repeat(scales.astype(np.float64), 32, axis=1)
        v = np.divide(np.asarray(w, np.float64), s, out=np.zeros_like(s), where=s > 0)
        tie = np.abs(v - np.trunc(v)) == 0.5
        away = np.clip(np.sign(v) * (np.floor(np.abs(v)) + 1), -q, q)
        return np.where(tie, away, codes).astype(np.int8), scales
    return f


def quant_scale_not_rounded_to_fp16(real):
    # the codes divide by the float32 scale; the fp16 scale is stored all the same
    def f(w, bits):
        codes, scales = real(w, bits)
        q = 127 if bits == 8 else 7
        w32 = np.asarray(w, np.float32)
        n, k = w32.shape
        s32 = (np.abs(w32.reshape(n, k // 32, 32)).max(axis=2) / np.float32(q)).astype(np.float32)
        s = np.repeat(s32, 32, axis=1)
        v = np.divide(w32, s, out=np.zeros_like(s), where=s > 0)
        return np.clip(np.rint(v), -q, q).astype(np.int8), scales
    return f


def pack_nibbles_swapped(real):
    def f(c):
        p = real(c)
        return (((p & 0x0F) << 4) | (p >> 4)).astype(np.uint8)
    return f


QUANT_PINS = ([functools.partial(pins_quant.test_worked_blocks, b) for b in pins_quant._load_golden()] +
              [functools.partial(pins_quant.test_exact_rederivation_random_blocks, b) for b in (8, 4)] +
              [pins_quant.test_scale_is_absmax_over_q_rounded_to_fp16, pins_quant.test_block_boundaries_are_along_the_row])

_E2M1_MIDPOINT_UP = {0.25: 1, 0.75: 2, 1.25: 3, 1.75: 4, 2.5: 5, 3.5: 6, 5.0: 7}


def e2m1_ties_up(real):
    # a ratio halfway between two E2M1 values goes to the larger magnitude
    def f(r):
        codes = real(r)
        r = np.asarray(r, np.float32)
        out = codes.copy().reshape(-1)
        for i, v in enumerate(r.reshape(-1)):
            up = _E2M1_MIDPOINT_UP.get(abs(float(v)))
            if up is not None:
                out[i] = up | (8 if float(v) < 0 else 0)
        return out.reshape(codes.shape)
    return f


def e2m1_negative_zero(real):
    # a negative ratio that rounds to zero keeps its sign bit (code 8)
    def f(r):
        codes = real(r)
        neg = np.signbit(np.asarray(r, np.float32))
        return np.where((codes == 0) & neg, 8, codes).astype(np.uint8)
    return f


FP4_PINS = [pins_fp4.test_encode_matches_brute_force, pins_fp4.test_round_trip_of_grid_values]

# ---- sampling verify ----------------------------------------------------------------


def sample_temperature_ignored(real):
    return lambda L, d, n_valid, T, seed, counter: real(L, d, n_valid, 1.0, seed, counter)


def sample_residual_may_return_draft(real):
    # on a rejection the next token is the rejected draft itself
    def f(L, d, n_valid, T, seed, counter):
        r = dict(real(L, d, n_valid, T, seed, counter))
        if r["accepted"] < n_valid:
            r["token"] = int(d[r["accepted"]])
        return r
    return f


def mix_state_off_by_one(real):
    # the finaliser applied to the state before its increment
    return lambda z: real(np.asarray(z, np.uint64) - sample.G)


SAMPLE_PINS = [pins_sample.test_low_temperature_reduces_to_greedy,
               functools.partial(pins_sample.test_first_token_follows_target, 2)]

PLANTS = [
    ("gemm: scale of the next block", verify, "dequant_gemm", gemm_block_off_by_one, GEMM_PINS),
    ("gemm: block scale dropped", verify, "dequant_gemm", gemm_scale_dropped, GEMM_PINS),
    ("gemm: sign flipped", verify, "dequant_gemm", gemm_sign_flipped, GEMM_PINS),
    ("gemm: last term dropped", verify, "dequant_gemm", gemm_last_term_dropped, GEMM_PINS),
    ("gemm: result transposed", verify, "dequant_gemm", gemm_result_transposed, GEMM_PINS),
    ("gemm: activation row off by one", verify, "dequant_gemm", gemm_row_off_by_one, GEMM_PINS),
    ("argmax: ties to the last index", verify, "argmax_rows", argmax_ties_to_last, ARGMAX_PINS),
    ("argmax: last entry not scanned", verify, "argmax_rows", argmax_tail_dropped, ARGMAX_PINS),
    ("top2: second largest below the maximum", verify, "top2_gap", top2_second_distinct, TOP2_PINS),
    ("accept: next token off by one", verify, "greedy_accept", accept_next_off_by_one, ACCEPT_PINS),
    ("accept: pads accepted", verify, "greedy_accept", accept_pads, ACCEPT_PINS),
    ("accept: shifted compare", verify, "greedy_accept", accept_shifted_compare, ACCEPT_PINS),
    ("accept: the miss kept", verify, "greedy_accept", accept_keeps_the_miss, ACCEPT_PINS),
    ("tree: parent links ignored", verify, "tree_accept", tree_as_chain, TREE_PINS),
    ("tree: token vs its own row", verify, "tree_accept", tree_compares_own_row, TREE_PINS),
    ("silu: sign of the exponent", mlp, "silu", silu_sign_error,
     [pins_mlp.test_silu_closed_forms, pins_mlp.test_silu_reflection_identity]),
    ("swiglu: gate and up swapped", mlp, "swiglu64", swiglu_gate_up_swapped, [pins_mlp.test_swiglu_one_hot_closed_form]),
    ("route: ties to the higher id", mlp, "route_topk", route_ties_to_higher_id,
     [pins_mlp.test_route_topk_brute_force_and_ties]),
    ("route: softmax over every expert", mlp, "route_topk", route_softmax_over_all_experts,
     [pins_mlp.test_route_topk_brute_force_and_ties]),
    ("group: rows in decreasing order", mlp, "group_by_expert", group_rows_reversed, [pins_mlp.test_group_by_expert]),
    ("group: inclusive offsets", mlp, "group_by_expert", group_offsets_inclusive, [pins_mlp.test_group_by_expert]),
    ("quant: ties away from zero", quant, "quantize_block32", quant_ties_away_from_zero, QUANT_PINS),
    ("quant: scale not rounded to fp16", quant, "quantize_block32", quant_scale_not_rounded_to_fp16, QUANT_PINS),
    ("int4: nibbles swapped", quant, "pack_int4", pack_nibbles_swapped,
     [pins_quant.test_int4_pack_roundtrip_and_nibble_order]),
    ("e2m1: ties to the larger magnitude", quant, "encode_e2m1", e2m1_ties_up, FP4_PINS),
    ("e2m1: negative zero", quant, "encode_e2m1", e2m1_negative_zero, FP4_PINS),
    ("splitmix: state off by one increment", sample, "mix", mix_state_off_by_one,
     [pins_sample.test_splitmix64_published_stream]),
    ("sample: temperature ignored", sample, "verify_sample", sample_temperature_ignored, SAMPLE_PINS),
    ("sample: residual draw may be the draft", sample, "verify_sample", sample_residual_may_return_draft,
     SAMPLE_PINS),
]


@pytest.mark.parametrize("plant", PLANTS, ids=[p[0] for p in PLANTS])
def test_pins_catch_planted_mistake(plant, monkeypatch):
    _, module, name, make, pins = plant
    monkeypatch.setattr(module, name, make(getattr(module, name)))
    caught = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin of {module.__name__}.{name} caught the planted mistake"


@pytest.mark.parametrize("plant", PLANTS, ids=[p[0] for p in PLANTS])
def test_pins_pass_on_the_oracle_itself(plant):
    # the same pins, unpatched: they fail above only because of the plant
    for pin in plant[4]:
        pin()

"""Pins for the oracle's general fused definition (router weights, input rows
per pair, several adapter slices, output column offset).

Each test ties it to something other than itself: a hand-worked example
(tests/golden/fused_ex_worked_example.json), the pinned one-slice definition
reached by an independent route (a problem reshaped so that every pair is its
own token; slices evaluated one at a time at their own offsets), exact integer
arithmetic, and the scaling law of the router weight.  All run on the CPU.
"""
import json
import os

import numpy as np

import oracle
from lora_moe_gb300 import inputs as gen

from test_oracle_pins import GOLDEN, covered_mask, f2b, small_case


def test_fused_ex_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "fused_ex_worked_example.json")))
    i, want = g["inputs"], g["expected"]
    a = [f2b(s) for s in i["lora_a_slices"]]
    b = [f2b(s) for s in i["lora_b_slices"]]
    args = (f2b(i["x_per_pair"]), a, b, f2b(i["y_in"]), np.array(i["topk_ids"]),
            np.array(i["token_lora_mapping"]), np.array(i["lora_ids"]))
    w = np.array(i["topk_weights"], np.float32)
    for add, key in ((True, "add_inputs_1"), (False, "add_inputs_0")):
        got = oracle.fused_ex(*args, add_inputs=add, topk_weights=w, x_per_pair=True,
                              y_offset=i["y_offset"])
        assert np.array_equal(got, np.array(want[key], np.float64)), key


def test_fused_ex_defaults_equal_one_slice_definition():
    for seed in range(4):
        x, a, b, y, tk, mp, ids = small_case(seed)
        for add in (True, False):
            assert np.array_equal(oracle.fused_ex(x, a, b, y, tk, mp, ids, add_inputs=add),
                                  oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=add))


def test_fused_ex_per_pair_rows_as_tokens():
    """Input rows per pair: the same as the one-slice definition on a reshaped
    problem in which every pair is a token of its own (topk = 1)."""
    for seed in range(4):
        x, a, b, y, tk, mp, ids = small_case(seed)
        M, topk = tk.shape
        K = x.shape[1]
        rng = np.random.default_rng(100 + seed)
        xp = f2b(rng.standard_normal((M * topk, K)).astype(np.float32))
        for add in (True, False):
            got = oracle.fused_ex(xp, a, b, y, tk, mp, ids, add_inputs=add, x_per_pair=True)
            want = oracle.fused(xp, a, b, y.reshape(M * topk, 1, -1), tk.reshape(-1, 1),
                                np.repeat(mp, topk), ids, add_inputs=add)
            assert np.array_equal(got.reshape(M * topk, -1), want.reshape(M * topk, -1))


def test_fused_ex_replicated_pair_rows_equal_token_rows():
    x, a, b, y, tk, mp, ids = small_case(7)
    topk = tk.shape[1]
    xp = np.repeat(x, topk, axis=0)
    assert np.array_equal(oracle.fused_ex(xp, a, b, y, tk, mp, ids, x_per_pair=True),
                          oracle.fused(x, a, b, y, tk, mp, ids))


def test_fused_ex_slices_are_independent_column_blocks():
    """Two slices at an offset: each slice's columns equal the one-slice
    definition with that slice's adapters; the other columns keep y_in."""
    for seed in range(3):
        x, a0, b0, _, tk, mp, ids = small_case(seed)
        _, a1, b1, _, _, _, _ = small_case(seed + 50)
        M, topk = tk.shape
        N = b0.shape[2]
        off, ldy = 8, 8 + 2 * N + 8
        rng = np.random.default_rng(seed)
        y = f2b(rng.standard_normal((M, topk, ldy)).astype(np.float32))
        for add in (True, False):
            got = oracle.fused_ex(x, [a0, a1], [b0, b1], y, tk, mp, ids, add_inputs=add, y_offset=off)
            s0 = oracle.fused(x, a0, b0, np.ascontiguousarray(y[:, :, off:off + N]), tk, mp, ids, add_inputs=add)
            s1 = oracle.fused(x, a1, b1, np.ascontiguousarray(y[:, :, off + N:off + 2 * N]), tk, mp, ids,
                              add_inputs=add)
            assert np.array_equal(got[:, :, off:off + N], s0)
            assert np.array_equal(got[:, :, off + N:off + 2 * N], s1)
            yv = gen.bf16_bits_to_f32(y).astype(np.float64)
            assert np.array_equal(got[:, :, :off], yv[:, :, :off])
            assert np.array_equal(got[:, :, off + 2 * N:], yv[:, :, off + 2 * N:])


def test_fused_ex_router_weight_scales_the_delta_only():
    """out - (add ? y_in : 0) is w[m, k] times the unweighted delta.  Powers of
    two keep the product exact."""
    x, a, b, y, tk, mp, ids = small_case(11)
    M, topk = tk.shape
    rng = np.random.default_rng(5)
    w = np.ldexp(1.0, rng.integers(-3, 4, size=(M, topk))).astype(np.float32)
    w *= rng.choice([-1.0, 1.0], size=(M, topk)).astype(np.float32)
    yv = gen.bf16_bits_to_f32(y).astype(np.float64)
    cov = covered_mask(tk, mp, ids, a.shape[1])
    for add in (True, False):
        base = yv if add else 0.0
        plain = oracle.fused_ex(x, a, b, y, tk, mp, ids, add_inputs=add)
        got = oracle.fused_ex(x, a, b, y, tk, mp, ids, add_inputs=add, topk_weights=w)
        want = np.where(cov[:, :, None], base + w[:, :, None].astype(np.float64) * (plain - base), yv)
        assert np.array_equal(got, want)


def test_fused_ex_integer_case_exact():
    """Two slices, per-pair rows, integer weights and {-1, 0, 1} operands:
    every value is an exact integer, so the result equals integer arithmetic."""
    x, a0, b0, _, tk, mp, ids = small_case(3, K=40, N=12, r=8, values="int")
    _, a1, b1, _, _, _, _ = small_case(4, K=40, N=12, r=8, values="int")
    M, topk = tk.shape
    rng = np.random.default_rng(9)
    xp = f2b(rng.integers(-1, 2, size=(M * topk, 40)).astype(np.float32))
    w = rng.integers(-3, 4, size=(M, topk)).astype(np.float32)
    ldy, off = 32, 4
    y = f2b(rng.integers(-4, 5, size=(M, topk, ldy)).astype(np.float32))
    got = oracle.fused_ex(xp, [a0, a1], [b0, b1], y, tk, mp, ids, add_inputs=True,
                          topk_weights=w, x_per_pair=True, y_offset=off)
    Xi = gen.bf16_bits_to_f32(xp).astype(np.int64)
    Yi = gen.bf16_bits_to_f32(y).astype(np.int64)
    cov = covered_mask(tk, mp, ids, a0.shape[1])
    for m in range(M):
        for k in range(topk):
            f = m * topk + k
            want = Yi[m, k].copy()
            if cov[m, k]:
                l, e = mp[m], tk[m, k]
                for s, (A, B) in enumerate(((a0, b0), (a1, b1))):
                    Ai = gen.bf16_bits_to_f32(A).astype(np.int64)[l, e]
                    Bi = gen.bf16_bits_to_f32(B).astype(np.int64)[l, e]
                    want[off + s * 12:off + (s + 1) * 12] += int(w[m, k]) * (Bi @ (Ai @ Xi[f]))
            assert np.array_equal(got[m, k], want.astype(np.float64))


def test_fused_ex_selected_pairs_equal_full():
    x, a0, b0, y, tk, mp, ids = small_case(2)
    _, a1, b1, _, _, _, _ = small_case(12)
    M, topk = tk.shape
    N = b0.shape[2]
    rng = np.random.default_rng(1)
    y2 = f2b(rng.standard_normal((M, topk, 2 * N + 8)).astype(np.float32))
    w = rng.standard_normal((M, topk)).astype(np.float32)
    full = oracle.fused_ex(x, [a0, a1], [b0, b1], y2, tk, mp, ids, topk_weights=w, y_offset=8)
    pairs = rng.choice(M * topk, 10, replace=False)
    sel = oracle.fused_ex(x, [a0, a1], [b0, b1], y2, tk, mp, ids, topk_weights=w, y_offset=8, pairs=pairs)
    assert np.array_equal(sel, full.reshape(M * topk, -1)[pairs])

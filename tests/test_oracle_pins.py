"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties the oracle to a fact fixed by the pages or by mathematics:
hand-worked examples (tests/golden), an independent brute force that uses a
different algorithm (a stable sort instead of count/prefix/scatter), exhaustive
enumeration of tiny inputs, invariants of the output, closed forms (zero B,
one-hot adapters, linearity, permutation) and a dense special case computed by
numpy.matmul.  All run on the CPU.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from lora_moe_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f2b(a):
    return gen.f32_to_bf16_bits(np.asarray(a, np.float32))


# ----------------------------------------------------------------------------
# Align: brute force by a different algorithm
# ----------------------------------------------------------------------------

def brute_align(topk_ids, mapping, lora_ids, E, block_size, adapter_enabled=None):
    """Stable sort of the covered pairs by (expert, flat index), then padding.

    Returns {l: (ntpp, sorted_prefix, expert_prefix)} for every active l."""
    M, topk = topk_ids.shape
    S = M * topk
    out = {}
    for l in lora_ids:
        l = int(l)
        if adapter_enabled is not None and not adapter_enabled[l]:
            out[l] = (0, [], [])
            continue
        keyed = sorted((int(topk_ids[m, k]), m * topk + k)
                       for m in range(M) for k in range(topk)
                       if mapping[m] == l and 0 <= topk_ids[m, k] < E)
        seq, experts = [], []
        for e, grp in itertools.groupby(keyed, key=lambda t: t[0]):
            fs = [f for _, f in grp]
            nblk = -(-len(fs) // block_size)
            seq += fs + [S] * (nblk * block_size - len(fs))
            experts += [e] * nblk
        out[l] = (len(seq), seq, experts)
    return out


def check_align_against_brute(topk_ids, mapping, lora_ids, E, L, bs, adapter_enabled=None):
    st, s, e, n = oracle.align(topk_ids, mapping, lora_ids, E, L, bs,
                               adapter_enabled=adapter_enabled)
    want = brute_align(topk_ids, mapping, lora_ids, E, bs, adapter_enabled)
    for l, (ntpp, seq, experts) in want.items():
        assert n[l] == ntpp
        assert list(s[l, :ntpp]) == seq
        assert list(e[l, :ntpp // bs]) == experts
    # nothing outside the defined region is written
    for l in range(L):
        if l not in want:
            assert n[l] == -7 and (s[l] == -7).all() and (e[l] == -7).all()
        else:
            assert (s[l, want[l][0]:] == -7).all()
            assert (e[l, want[l][0] // bs:] == -7).all()
    return st


def test_align_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "align_worked_example.json")))
    i, x = g["inputs"], g["expected"]
    st, s, e, n = oracle.align(np.array(i["topk_ids"]), np.array(i["token_lora_mapping"]),
                               np.array(i["lora_ids"]), i["num_experts"], i["max_loras"],
                               i["block_size"])
    assert st == 0
    assert list(n) == x["num_tokens_post_padded"]
    for l in range(i["max_loras"]):
        nt = x["num_tokens_post_padded"][l]
        assert list(s[l, :nt]) == x["sorted_token_ids"][l]
        assert list(e[l, :nt // i["block_size"]]) == x["expert_ids"][l]


def test_align_exhaustive_tiny_distinct_experts():
    """Every topk assignment (distinct experts per token) and every mapping over
    {-1, 0, 1}, for M=3, topk=2, E=3, all block sizes 1, 2, 4."""
    E, topk, M, L = 3, 2, 3, 2
    rows = list(itertools.permutations(range(E), topk))
    maps = list(itertools.product([-1, 0, 1], repeat=M))
    rng = np.random.default_rng(1)
    assigns = list(itertools.product(rows, repeat=M))
    for bs in (1, 2, 4):
        for ti, tk in enumerate(assigns):
            topk_ids = np.array(tk, np.int32)
            # all maps for a subset of assignments, a random map otherwise
            chosen = maps if ti % 9 == 0 else [maps[rng.integers(len(maps))]]
            for mp in chosen:
                check_align_against_brute(topk_ids, np.array(mp, np.int32),
                                          np.array([0, 1], np.int32), E, L, bs)


def test_align_exhaustive_tiny_with_repeats():
    """Repeated experts within a token (not produced by a router, but the
    definition covers them): every assignment for M=2, topk=2, E=2."""
    E, topk, M = 2, 2, 2
    for tk in itertools.product(range(E), repeat=M * topk):
        for mp in itertools.product([-1, 0, 1], repeat=M):
            for bs in (1, 2, 4):
                for lora_ids in ([0], [1], [0, 1], [1, 0]):
                    check_align_against_brute(np.array(tk, np.int32).reshape(M, topk),
                                              np.array(mp, np.int32),
                                              np.array(lora_ids, np.int32), E, 2, bs)


@pytest.mark.parametrize("seed", range(12))
def test_align_random_against_brute(seed):
    rng = np.random.default_rng(100 + seed)
    M = int(rng.integers(1, 40))
    E = int(rng.integers(1, 40))
    topk = int(rng.integers(1, min(E, 8) + 1))
    L = int(rng.integers(1, 6))
    nact = int(rng.integers(1, L + 1))
    bs = int(rng.choice([1, 2, 4, 16, 64]))
    lora_ids = rng.choice(L, nact, replace=False).astype(np.int32)
    topk_ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    mapping = rng.integers(-1, L, size=M).astype(np.int32)
    enabled = (rng.random(L) < 0.8).astype(np.int32) if seed % 3 == 0 else None
    st = check_align_against_brute(topk_ids, mapping, lora_ids, E, L, bs, enabled)
    assert st == 0


def test_align_invariants_on_workloads():
    for name in ("tiny", "decode_qwen3_w13", "decode_gptoss_w2", "prefill_mixtral_w13",
                 "large_e_nact4"):
        w = gen.WORKLOADS[name]
        inp = gen.make_inputs(w, with_tensors=False)
        st, s, e, n = oracle.align(inp.topk_ids, inp.token_lora_mapping, inp.lora_ids,
                                   w.E, w.max_loras, w.block_size)
        assert st == 0
        S = w.M * w.topk
        seen = []
        for l in inp.lora_ids:
            nt = int(n[l])
            assert nt % w.block_size == 0                        # segments padded to bs
            seg, blk = s[l, :nt], e[l, :nt // w.block_size]
            # closed form: ntpp = sum_e ceil(cnt/bs)*bs
            mask = inp.token_lora_mapping == l
            cnt = np.bincount(inp.topk_ids[mask].ravel(), minlength=w.E)
            assert nt == int((-(-cnt // w.block_size) * w.block_size).sum())
            assert (np.diff(blk) >= 0).all()                     # ascending experts, one run each
            for ex in np.unique(blk):                            # a segment ascends across its blocks
                seg_e = seg[np.repeat(blk == ex, w.block_size)]
                assert (np.diff(seg_e[seg_e != S]) > 0).all()
            for b in range(nt // w.block_size):
                ids = seg[b * w.block_size:(b + 1) * w.block_size]
                real = ids[ids != S]
                # padding only at the end of a block, and each block has a real pair
                assert len(real) > 0 and (ids[:len(real)] != S).all()
                assert (np.diff(real) > 0).all()                # ascending flat index
                assert (inp.topk_ids.ravel()[real] == blk[b]).all()   # block's expert
                assert (inp.token_lora_mapping[real // w.topk] == l).all()
            seen += list(seg[seg != S])
        seen = np.array(sorted(seen))
        covered = [f for f in range(S) if inp.token_lora_mapping[f // w.topk] in inp.lora_ids]
        assert list(seen) == covered                            # each covered pair exactly once
        # tokens with LoRA -1 are dropped
        none = np.where(inp.token_lora_mapping == -1)[0]
        assert not np.isin(seen // w.topk, none).any()


def test_align_single_lora_is_plain_moe_align():
    """One LoRA owning every token reduces to the non-LoRA align: a stable sort
    of pairs by expert (numpy argsort, kind='stable') plus block padding."""
    rng = np.random.default_rng(7)
    M, topk, E, bs = 50, 4, 16, 8
    topk_ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    st, s, e, n = oracle.align(topk_ids, np.zeros(M, np.int32), np.array([0], np.int32),
                               E, 1, bs)
    order = np.argsort(topk_ids.ravel(), kind="stable")
    keys = topk_ids.ravel()[order]
    seq, blocks = [], []
    for ex in range(E):
        fs = order[keys == ex]
        if len(fs) == 0:
            continue
        nb = -(-len(fs) // bs)
        seq += list(fs) + [M * topk] * (nb * bs - len(fs))
        blocks += [ex] * nb
    assert st == 0 and n[0] == len(seq)
    assert list(s[0, :n[0]]) == seq and list(e[0, :n[0] // bs]) == blocks


@pytest.mark.parametrize("seed,M,topk,E,bs", [(1, 50, 4, 16, 8), (2, 3, 1, 1, 16), (3, 200, 8, 64, 64),
                                               (4, 0, 2, 4, 16), (5, 33, 6, 6, 128)])
def test_align_plain_is_stable_sort_by_expert(seed, M, topk, E, bs):
    """The plain align (no LoRA): a stable sort of all pairs by expert
    (numpy argsort, kind='stable'), padded per expert to block_size with the
    sentinel M*topk; experts without pairs get no block."""
    rng = np.random.default_rng(seed)
    topk_ids = rng.integers(0, E, size=(M, topk)).astype(np.int32)
    st, s, e, n = oracle.align_plain(topk_ids, E, bs)
    order = np.argsort(topk_ids.ravel(), kind="stable")
    keys = topk_ids.ravel()[order]
    seq, blocks = [], []
    for ex in range(E):
        fs = order[keys == ex]
        if len(fs) == 0:
            continue
        nb = -(-len(fs) // bs)
        seq += list(fs) + [M * topk] * (nb * bs - len(fs))
        blocks += [ex] * nb
    assert st == 0 and n[0] == len(seq)
    assert list(s[:n[0]]) == seq and list(e[:n[0] // bs]) == blocks
    assert (s[n[0]:] == -7).all() and (e[n[0] // bs:] == -7).all()


def test_align_reports_bad_ids():
    topk_ids = np.array([[0, 5], [1, 2]], np.int32)   # 5 is out of range for E=3
    st, s, e, n = oracle.align(topk_ids, np.array([0, 0], np.int32), np.array([0], np.int32), 3, 1, 2)
    assert st & oracle.STATUS_BAD_EXPERT_ID
    assert list(s[0, :n[0]]) == [0, 4, 2, 4, 3, 4]   # the bad pair (f=1) is dropped
    st, *_ = oracle.align(topk_ids[:, :1], np.array([0, 0], np.int32), np.array([3], np.int32), 3, 2, 2)
    assert st & oracle.STATUS_BAD_LORA_ID


def test_align_disabled_adapter_and_inactive_slot():
    topk_ids = np.array([[0], [1], [0]], np.int32)
    mapping = np.array([0, 1, 2], np.int32)
    st, s, e, n = oracle.align(topk_ids, mapping, np.array([0, 1], np.int32), 2, 3, 1,
                               adapter_enabled=np.array([1, 0, 1], np.int32))
    assert st == 0 and n[0] == 1 and n[1] == 0 and n[2] == -7   # slot 2 not active: untouched


# ----------------------------------------------------------------------------
# Fused: closed forms, special cases and a library cross-check
# ----------------------------------------------------------------------------

def small_case(seed, M=9, topk=3, E=5, K=24, N=16, r=4, L=3, nact=2, values="normal"):
    rng = np.random.default_rng(seed)
    lora_ids = np.sort(rng.choice(L, nact, replace=False)).astype(np.int32)
    topk_ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    mapping = rng.integers(-1, L, size=M).astype(np.int32)
    if values == "int":
        draw = lambda *s: rng.integers(-1, 2, size=s).astype(np.float32)
    else:
        draw = lambda *s: rng.standard_normal(s).astype(np.float32)
    x = f2b(draw(M, K))
    a = f2b(draw(L, E, r, K) if values == "int" else draw(L, E, r, K) / np.sqrt(K))
    b = f2b(draw(L, E, N, r))
    y = f2b(draw(M, topk, N))
    return x, a, b, y, topk_ids, mapping, lora_ids


def covered_mask(topk_ids, mapping, lora_ids, E, enabled=None):
    M, topk = topk_ids.shape
    cov = np.zeros((M, topk), bool)
    for m in range(M):
        l = mapping[m]
        if l < 0 or l not in lora_ids or (enabled is not None and not enabled[l]):
            continue
        cov[m] = (topk_ids[m] >= 0) & (topk_ids[m] < E)
    return cov


def test_fused_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "fused_worked_example.json")))
    i, x = g["inputs"], g["expected"]
    args = [f2b(i["x"]), f2b(i["lora_a"]), f2b(i["lora_b"]), f2b(i["y_in"]),
            np.array(i["topk_ids"]), np.array(i["token_lora_mapping"]), np.array(i["lora_ids"])]
    assert np.array_equal(oracle.fused(*args, add_inputs=True), np.array(x["add_inputs_1"]))
    assert np.array_equal(oracle.fused(*args, add_inputs=False), np.array(x["add_inputs_0"]))


def test_fused_matches_grouped_matmul():
    """Cross-check with a different computation route: gather each (lora, expert)
    segment's x rows into a matrix and apply numpy.matmul twice in float64."""
    for seed in range(6):
        x, a, b, y, tk, mp, ids = small_case(seed)
        E = a.shape[1]
        for add in (True, False):
            ref = oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=add)
            X = gen.bf16_bits_to_f32(x).astype(np.float64)
            A = gen.bf16_bits_to_f32(a).astype(np.float64)
            B = gen.bf16_bits_to_f32(b).astype(np.float64)
            Y = gen.bf16_bits_to_f32(y).astype(np.float64)
            want = Y.copy()
            cov = covered_mask(tk, mp, ids, E)
            for l in ids:
                for e in range(E):
                    sel = [(m, k) for m in range(tk.shape[0]) for k in range(tk.shape[1])
                           if cov[m, k] and mp[m] == l and tk[m, k] == e]
                    if not sel:
                        continue
                    rows = np.array([m for m, _ in sel])
                    delta = np.matmul(np.matmul(X[rows], A[l, e].T), B[l, e].T)
                    for i, (m, k) in enumerate(sel):
                        want[m, k] = (Y[m, k] if add else 0.0) + delta[i]
            np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-12)


def test_fused_integer_case_exact():
    """x, A, B in {-1, 0, 1}: every product and partial sum is an exact integer,
    so the oracle must equal integer arithmetic exactly."""
    x, a, b, y, tk, mp, ids = small_case(3, K=40, N=12, r=8, values="int")
    ref = oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=False)
    Xi = gen.bf16_bits_to_f32(x).astype(np.int64)
    Ai = gen.bf16_bits_to_f32(a).astype(np.int64)
    Bi = gen.bf16_bits_to_f32(b).astype(np.int64)
    Yi = gen.bf16_bits_to_f32(y).astype(np.float64)
    cov = covered_mask(tk, mp, ids, a.shape[1])
    for m in range(tk.shape[0]):
        for k in range(tk.shape[1]):
            if not cov[m, k]:
                assert np.array_equal(ref[m, k], Yi[m, k])
                continue
            l, e = mp[m], tk[m, k]
            t = Ai[l, e] @ Xi[m]
            assert np.array_equal(ref[m, k], (Bi[l, e] @ t).astype(np.float64))


def test_fused_zero_b_gives_zero_delta():
    x, a, b, y, tk, mp, ids = small_case(4)
    b0 = np.zeros_like(b)
    Y = gen.bf16_bits_to_f32(y).astype(np.float64)
    cov = covered_mask(tk, mp, ids, a.shape[1])
    assert np.array_equal(oracle.fused(x, a, b0, y, tk, mp, ids, add_inputs=True), Y)
    out0 = oracle.fused(x, a, b0, y, tk, mp, ids, add_inputs=False)
    assert (out0[cov] == 0).all() and np.array_equal(out0[~cov], Y[~cov])


def test_fused_one_hot_adapters_copy_x():
    """A[l,e][j][k] = 1 iff k == c[j]; B[l,e][n][j] = 1 iff j == d[n]:
    the delta at column n is x[m][c[d[n]]]."""
    x, a, b, y, tk, mp, ids = small_case(5, K=16, N=10, r=4)
    L, E, r, K = a.shape
    N = b.shape[2]
    rng = np.random.default_rng(11)
    c = rng.integers(0, K, size=(L, E, r))
    d = rng.integers(0, r, size=(L, E, N))
    A = np.zeros((L, E, r, K), np.float32)
    B = np.zeros((L, E, N, r), np.float32)
    for l in range(L):
        for e in range(E):
            A[l, e, np.arange(r), c[l, e]] = 1
            B[l, e, np.arange(N), d[l, e]] = 1
    out = oracle.fused(x, f2b(A), f2b(B), y, tk, mp, ids, add_inputs=False)
    X = gen.bf16_bits_to_f32(x)
    cov = covered_mask(tk, mp, ids, E)
    for m in range(tk.shape[0]):
        for k in range(tk.shape[1]):
            if cov[m, k]:
                l, e = mp[m], tk[m, k]
                assert np.array_equal(out[m, k], X[m, c[l, e][d[l, e]]].astype(np.float64))


def test_fused_linearity_in_b():
    x, a, b, y, tk, mp, ids = small_case(6)
    b2 = f2b(gen.bf16_bits_to_f32(b) * 2)     # exact: a power-of-two scale of bf16
    d1 = oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=False)
    d2 = oracle.fused(x, a, b2, y, tk, mp, ids, add_inputs=False)
    cov = covered_mask(tk, mp, ids, a.shape[1])
    assert np.array_equal(d2[cov], 2 * d1[cov])


def test_fused_token_permutation():
    x, a, b, y, tk, mp, ids = small_case(7)
    perm = np.random.default_rng(3).permutation(x.shape[0])
    base = oracle.fused(x, a, b, y, tk, mp, ids)
    permuted = oracle.fused(x[perm], a, b, y[perm], tk[perm], mp[perm], ids)
    assert np.array_equal(permuted, base[perm])


def test_fused_dense_special_case():
    """E = 1, one LoRA, every token covered: y = y_in + (x A^T) B^T, a plain
    dense product computed by numpy.matmul in float64."""
    rng = np.random.default_rng(9)
    M, K, N, r = 33, 72, 40, 8
    x = f2b(rng.standard_normal((M, K)))
    a = f2b(rng.standard_normal((1, 1, r, K)) / np.sqrt(K))
    b = f2b(rng.standard_normal((1, 1, N, r)) / np.sqrt(r))
    y = f2b(rng.standard_normal((M, 1, N)))
    ref = oracle.fused(x, a, b, y, np.zeros((M, 1), np.int32), np.zeros(M, np.int32),
                       np.array([0], np.int32))
    X = gen.bf16_bits_to_f32(x).astype(np.float64)
    A = gen.bf16_bits_to_f32(a)[0, 0].astype(np.float64)
    B = gen.bf16_bits_to_f32(b)[0, 0].astype(np.float64)
    want = gen.bf16_bits_to_f32(y)[:, 0].astype(np.float64) + np.matmul(np.matmul(X, A.T), B.T)
    np.testing.assert_allclose(ref[:, 0], want, rtol=1e-12, atol=1e-12)


def test_fused_uncovered_pairs_untouched_and_poison_unread():
    """Inactive slots hold NaN; -1 tokens, tokens of inactive or disabled slots
    and out-of-range experts keep y_in exactly, and no NaN reaches the output."""
    x, a, b, y, tk, mp, ids = small_case(8, L=4, nact=2)
    L = a.shape[0]
    inactive = [l for l in range(L) if l not in ids]
    a = a.copy(); b = b.copy()
    a[inactive] = gen.BF16_QNAN
    b[inactive] = gen.BF16_QNAN
    tk = tk.copy(); tk[0, 0] = 99                   # out of range expert
    enabled = np.ones(L, np.int32); enabled[ids[0]] = 0
    a[ids[0]] = gen.BF16_QNAN                       # disabled slot is never read either
    for add in (True, False):
        out = oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=add, adapter_enabled=enabled)
        assert np.isfinite(out).all()
        cov = covered_mask(tk, mp, ids, a.shape[1], enabled)
        Y = gen.bf16_bits_to_f32(y).astype(np.float64)
        assert np.array_equal(out[~cov], Y[~cov])
        assert cov.any() and (~cov).any()


def test_fused_sampled_equals_full():
    x, a, b, y, tk, mp, ids = small_case(10)
    full = oracle.fused(x, a, b, y, tk, mp, ids)
    pairs = np.array([0, 5, 7, 26], np.int32)
    cols = np.array([0, 3, 15], np.int32)
    samp = oracle.fused_sampled(x, a, b, y, tk, mp, ids, pairs, cols)
    flat = full.reshape(-1, full.shape[2])
    assert np.array_equal(samp, flat[pairs][:, cols])


def test_fused_add_modes_agree():
    x, a, b, y, tk, mp, ids = small_case(12, values="int")
    one = oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=True)
    zero = oracle.fused(x, a, b, y, tk, mp, ids, add_inputs=False)
    cov = covered_mask(tk, mp, ids, a.shape[1])
    Y = gen.bf16_bits_to_f32(y).astype(np.float64)
    np.testing.assert_allclose(one[cov] - Y[cov], zero[cov], rtol=1e-12, atol=1e-12)

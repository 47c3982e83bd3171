"""Property-based pins of the oracle (hypothesis; skipped where it is not
installed).  Over generated routings and shapes, the align output satisfies
what the definition fixes: every covered pair appears exactly once, in its
expert's segment, in ascending flat index; segments are block_size multiples
in ascending expert order and padded with the sentinel; tokens mapped to -1
or to an unlisted slot are dropped.  The fused definition gives a zero delta
for a zero B and does not depend on the order of lora_ids."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from lora_moe_gb300 import inputs as gen  # noqa: E402


@st.composite
def routings(draw):
    E = draw(st.integers(1, 12))
    topk = draw(st.integers(1, min(E, 4)))
    M = draw(st.integers(0, 24))
    L = draw(st.integers(1, 4))
    nact = draw(st.integers(1, L))
    bs = draw(st.sampled_from([16, 32, 64, 128]))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    lora_ids = rng.permutation(L)[:nact].astype(np.int32)
    topk_ids = (np.stack([rng.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
                if M else np.zeros((0, topk), np.int32))
    mapping = rng.integers(-1, L, size=M).astype(np.int32)
    return topk_ids, mapping, lora_ids, E, L, bs


@settings(max_examples=200, deadline=None)
@given(routings())
def test_align_properties(r):
    topk_ids, mapping, lora_ids, E, L, bs = r
    M, topk = topk_ids.shape
    P = M * topk
    st_, s, e, n = oracle.align(topk_ids, mapping, lora_ids, E, L, bs)
    assert st_ == 0
    for l in range(L):
        if l not in set(lora_ids.tolist()):
            assert n[l] == -7            # unlisted rows are not written
            continue
        ntpp = int(n[l])
        assert ntpp % bs == 0
        seq, experts = s[l, :ntpp], e[l, :ntpp // bs]
        # the covered pairs of this slot, each exactly once
        want = sorted(m * topk + k for m in range(M) for k in range(topk) if mapping[m] == l)
        real = sorted(int(f) for f in seq if f != P)
        assert real == want
        assert all(0 <= f <= P for f in seq)
        # segments: one expert per block, experts ascending, pairs ascending and
        # belonging to the block's expert, padding only at a segment's end
        assert all(experts[i] <= experts[i + 1] for i in range(len(experts) - 1))
        for b in range(ntpp // bs):
            ex = int(experts[b])
            blk = [int(f) for f in seq[b * bs:(b + 1) * bs]]
            reals = [f for f in blk if f != P]
            assert all(topk_ids.reshape(-1)[f] == ex for f in reals)
            assert reals == sorted(reals)
            first_pad = next((i for i, f in enumerate(blk) if f == P), bs)
            assert all(f == P for f in blk[first_pad:])
            if b + 1 < ntpp // bs and experts[b + 1] == ex:
                assert first_pad == bs           # only the last block of a segment pads
        # each expert's pairs in ascending flat index across its blocks
        for ex in set(int(v) for v in experts):
            fs = [int(f) for b in range(ntpp // bs) if experts[b] == ex for f in seq[b * bs:(b + 1) * bs] if f != P]
            assert fs == sorted(fs)
        # padding is minimal: ceil(count / bs) blocks per expert
        for ex in range(E):
            cnt = sum(1 for f in want if topk_ids.reshape(-1)[f] == ex)
            assert int((experts == ex).sum()) == -(-cnt // bs)


@st.composite
def fused_cases(draw):
    topk_ids, mapping, lora_ids, E, L, bs = draw(routings())
    K = 8 * draw(st.integers(1, 6))
    N = 8 * draw(st.integers(1, 4))
    r = draw(st.sampled_from([1, 2, 4, 8]))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return topk_ids, mapping, lora_ids, E, L, K, N, r, seed


def _tensors(M, topk, E, L, K, N, r, seed):
    rng = np.random.default_rng(seed)
    f2b = gen.f32_to_bf16_bits
    x = f2b(rng.standard_normal((M, K)).astype(np.float32))
    a = f2b(rng.standard_normal((L, E, r, K)).astype(np.float32))
    b = f2b(rng.standard_normal((L, E, N, r)).astype(np.float32))
    y = f2b(rng.standard_normal((M, topk, N)).astype(np.float32))
    return x, a, b, y


@settings(max_examples=100, deadline=None)
@given(fused_cases())
def test_fused_zero_b_and_slot_order(c):
    topk_ids, mapping, lora_ids, E, L, K, N, r, seed = c
    M, topk = topk_ids.shape
    x, a, b, y = _tensors(M, topk, E, L, K, N, r, seed)
    yv = gen.bf16_bits_to_f32(y).astype(np.float64)
    # a zero B: accumulate keeps y_in, overwrite writes zeros on covered pairs only
    zb = np.zeros_like(b)
    keep = oracle.fused(x, a, zb, y, topk_ids, mapping, lora_ids, add_inputs=True)
    assert np.array_equal(keep, yv)
    over = oracle.fused(x, a, zb, y, topk_ids, mapping, lora_ids, add_inputs=False)
    listed = set(lora_ids.tolist())
    for m in range(M):
        want = np.zeros((topk, N)) if int(mapping[m]) in listed else yv[m]
        assert np.array_equal(over[m], want)
    # the order of lora_ids does not matter
    ref = oracle.fused(x, a, b, y, topk_ids, mapping, lora_ids)
    assert np.array_equal(ref, oracle.fused(x, a, b, y, topk_ids, mapping, lora_ids[::-1].copy()))

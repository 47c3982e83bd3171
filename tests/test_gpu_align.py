"""GPU parity of moe_lora_align against the CPU oracle: bit-exact on every
defined entry, every other entry left untouched, both variants."""
import numpy as np
import pytest

from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

VARIANTS = [B.ALIGN_SMEM, B.ALIGN_GLOBAL, B.ALIGN_CLUSTER]
WORKLOADS = ["tiny", "decode_qwen3_w13", "decode_gptoss_w2", "prefill_mixtral_w13",
             "large_e_nact1", "large_e_nact4", "large_e_nact8"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("variant", VARIANTS + [B.ALIGN_AUTO])
@pytest.mark.parametrize("name", WORKLOADS)
def test_align_workloads(name, variant):
    from helpers import assert_align_equal
    w = gen.WORKLOADS[name]
    inp = gen.make_inputs(w, with_tensors=False)
    assert_align_equal(inp.topk_ids, inp.token_lora_mapping, inp.lora_ids, w.E, w.max_loras, w.block_size,
                       variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("seed", range(16))
def test_align_random_shapes(seed, variant):
    from helpers import assert_align_equal
    rng = np.random.default_rng(1000 + seed)
    M = int(rng.choice([1, 3, 17, 64, 257, 1000, 3001]))
    E = int(rng.choice([1, 2, 8, 33, 128, 255, 256, 600, 1024]))
    topk = int(rng.integers(1, min(E, 8) + 1))
    L = int(rng.integers(1, 9))
    nact = int(rng.integers(1, L + 1))
    bs = int(rng.choice([16, 32, 64, 128]))
    lora_ids = rng.choice(L, nact, replace=False).astype(np.int32)
    topk_ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    mapping = rng.integers(-1, L, size=M).astype(np.int32)
    enabled = (rng.random(L) < 0.75).astype(np.int32) if seed % 4 == 0 else None
    assert_align_equal(topk_ids, mapping, lora_ids, E, L, bs, variant, enabled)


@pytest.mark.parametrize("variant", VARIANTS)
def test_align_edge_cases(variant):
    from helpers import assert_align_equal
    # every token without an adapter
    assert_align_equal(np.array([[0, 1]] * 5, np.int32), np.full(5, -1, np.int32), np.array([0, 1], np.int32),
                       4, 2, 16, variant)
    # a single pair
    assert_align_equal(np.array([[3]], np.int32), np.array([0], np.int32), np.array([0], np.int32), 4, 1, 16,
                       variant)
    # M = 0
    assert_align_equal(np.zeros((0, 2), np.int32), np.zeros(0, np.int32), np.array([1, 0], np.int32), 4, 2, 32,
                       variant)
    # tokens mapped to slots that are not listed are dropped; E = 1; topk = E
    assert_align_equal(np.zeros((40, 1), np.int32), np.arange(40, dtype=np.int32) % 3, np.array([2], np.int32),
                       1, 3, 16, variant)
    assert_align_equal(np.tile(np.arange(8, dtype=np.int32), (33, 1)), np.zeros(33, np.int32),
                       np.array([0], np.int32), 8, 1, 64, variant)
    # lora ids listed out of order
    rng = np.random.default_rng(5)
    topk_ids = np.stack([rng.choice(64, 4, replace=False) for _ in range(200)]).astype(np.int32)
    assert_align_equal(topk_ids, rng.integers(0, 4, 200).astype(np.int32), np.array([3, 0, 2], np.int32), 64, 4,
                       16, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_align_bad_ids_flagged_and_dropped(variant):
    from helpers import assert_align_equal
    topk_ids = np.array([[0, 9], [1, -3], [2, 3]], np.int32)     # 9 and -3 are outside [0, 4)
    assert_align_equal(topk_ids, np.array([0, 0, 0], np.int32), np.array([0], np.int32), 4, 1, 16, variant)
    # an out-of-range slot id is flagged and its slot skipped
    s, e, n, err, _ = __import__("helpers").gpu_align(
        (np.array([[0]], np.int32), np.array([0], np.int32), np.array([5], np.int32)), 4, 2, 16, variant)
    assert err & B.DEVERR_LORA_ID
    assert (n == 0x7FFFFFFF).all()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,topk,E", [(20000, 8, 64), (4097, 1, 1024), (9000, 7, 256)])
def test_align_long_pair_lists(M, topk, E, variant):
    """Pair lists long enough for 8-CTA clusters and, past 256 pairs a warp,
    the walks that reread the routing; ragged ranges per CTA and per warp."""
    from helpers import assert_align_equal
    rng = np.random.default_rng(M + E)
    topk_ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    mapping = rng.integers(-1, 3, size=M).astype(np.int32)
    assert_align_equal(topk_ids, mapping, np.array([2, 0], np.int32), E, 3, 64, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_align_deterministic_repeats(variant):
    """The same inputs give identical outputs on repeated runs (no order left to
    the scheduler)."""
    from helpers import gpu_align
    w = gen.WORKLOADS["large_e_nact8"]
    inp = gen.make_inputs(w, with_tensors=False)
    first = gpu_align((inp.topk_ids, inp.token_lora_mapping, inp.lora_ids), w.E, w.max_loras, w.block_size,
                      variant)
    for _ in range(20):
        again = gpu_align((inp.topk_ids, inp.token_lora_mapping, inp.lora_ids), w.E, w.max_loras, w.block_size,
                          variant)
        for a, b in zip(first[:3], again[:3]):
            assert np.array_equal(a, b)

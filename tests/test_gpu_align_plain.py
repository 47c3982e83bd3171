"""GPU parity of the plain (non-LoRA) MoE align, moe_align_block_size: the
single-slot case of the LoRA align, bit-exact against the oracle on the
defined entries, every other entry left untouched, in both variants."""
import numpy as np
import pytest

import oracle
from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

VARIANTS = [B.ALIGN_SMEM, B.ALIGN_GLOBAL, B.ALIGN_CLUSTER, B.ALIGN_AUTO]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_plain(topk_ids, E, bs, variant):
    import torch
    from helpers import POISON, dev_i32
    M, topk = topk_ids.shape
    cap = B.max_num_tokens_padded(M, topk, E, bs)
    capb = B.max_num_m_blocks(M, topk, E, bs)
    s = torch.full((cap,), POISON, dtype=torch.int32, device="cuda")
    e = torch.full((capb,), POISON, dtype=torch.int32, device="cuda")
    n = torch.full((1,), POISON, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    nbytes = B.align_workspace_bytes(M, topk, E, 1, bs, variant)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    B.moe_align_block_size(dev_i32(topk_ids), E, bs, s, e, n, workspace=ws, variant=variant, err_flag=err)
    torch.cuda.synchronize()
    ost, os_, oe, on = oracle.align_plain(topk_ids, E, bs, max_num_tokens_padded=cap, max_num_m_blocks=capb,
                                          fill=POISON)
    assert np.array_equal(n.cpu().numpy(), on)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(e.cpu().numpy(), oe)
    want_err = B.DEVERR_EXPERT_ID if ost & oracle.STATUS_BAD_EXPERT_ID else 0
    assert int(err.item()) == want_err


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "decode_qwen3_w13", "decode_gptoss_w2", "prefill_mixtral_w13",
                                  "large_e_nact8"])
def test_plain_align_workloads(name, variant):
    w = gen.WORKLOADS[name]
    inp = gen.make_inputs(w, with_tensors=False)
    run_plain(inp.topk_ids, w.E, w.block_size, variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("seed", range(8))
def test_plain_align_random_shapes(seed, variant):
    rng = np.random.default_rng(300 + seed)
    E = int(rng.integers(1, 1025)) if seed % 2 else int(rng.integers(1, 64))
    M = int(rng.integers(0, 3000))
    topk = int(rng.integers(1, min(E, 8) + 1))
    bs = int(rng.choice([16, 32, 64, 128]))
    topk_ids = rng.integers(0, E, size=(M, topk)).astype(np.int32)
    run_plain(topk_ids, E, bs, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_plain_align_bad_expert_ids_dropped(variant):
    rng = np.random.default_rng(5)
    topk_ids = rng.integers(0, 16, size=(40, 4)).astype(np.int32)
    topk_ids[3, 1] = -1
    topk_ids[7, 0] = 16
    run_plain(topk_ids, 16, 16, variant)

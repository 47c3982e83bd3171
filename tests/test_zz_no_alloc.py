"""moe_lora_align_static_workspace: the align entry point for callers that
cannot allocate device memory (its workspace is a buffer built into the
library).  Its results must equal moe_lora_align's, call after call, because
the built-in buffer is shared by every call and keeps the previous call's
contents.

This file is collected last so that a run that stops at the first failure has
already run every other test; it also passes when run alone."""
import numpy as np
import pytest

from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _outputs(w, inp, fn, **kw):
    import torch
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    buf = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size,
                         variant=B.ALIGN_GLOBAL)
    for t in (buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded):
        t.fill_(0x7FFFFFFF)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn(dev(inp.topk_ids), dev(inp.token_lora_mapping), dev(inp.lora_ids), w.E, w.max_loras, w.block_size,
       buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded, err_flag=err, **kw)
    torch.cuda.synchronize()
    return (buf.sorted_token_ids.cpu().numpy(), buf.expert_ids.cpu().numpy(),
            buf.num_tokens_post_padded.cpu().numpy(), int(err.item()))


@pytest.mark.parametrize("names", [("large_e_nact8", "decode_qwen3_w13"), ("decode_gptoss_w2", "large_e_nact4")])
def test_static_workspace_matches_workspace_entry_point(names):
    """Two calls in a row (different inputs, so the second call finds the first
    call's data in the shared buffer); each must equal moe_lora_align on a
    caller-allocated workspace, bit for bit."""
    for name in names:
        w = gen.WORKLOADS[name]
        inp = gen.make_inputs(w, with_tensors=False)
        ref_buf = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size,
                                 variant=B.ALIGN_GLOBAL)
        want = _outputs(w, inp, B.moe_lora_align, workspace=ref_buf.workspace, variant=B.ALIGN_GLOBAL)
        got = _outputs(w, inp, B.moe_lora_align_static_workspace)
        for a, b in zip(got[:3], want[:3]):
            assert np.array_equal(a, b)
        assert got[3] == want[3] == 0


def test_static_workspace_rejects_sizes_beyond_its_buffer():
    """A problem whose workspace exceeds the built-in 4 MiB is refused with
    MOE_LORA_ERR_WORKSPACE before anything is enqueued."""
    import torch
    M, topk, E, L, bs = 65536, 8, 1024, 8, 16
    need = B.align_workspace_bytes(M, topk, E, L, bs, B.ALIGN_GLOBAL)
    assert need > B.STATIC_WORKSPACE_BYTES
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = B.lib().moe_lora_align_static_workspace(
        z.data_ptr(), z.data_ptr(), z.data_ptr(), None, M, topk, E, L, L, bs, z.data_ptr(), z.data_ptr(),
        z.data_ptr(), B.max_num_tokens_padded(M, topk, E, bs), B.max_num_m_blocks(M, topk, E, bs), None, None)
    assert st == 4   # MOE_LORA_ERR_WORKSPACE

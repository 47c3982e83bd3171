"""The kernels' on-chip waits are bounded: a wait that runs out reports
MOE_LORA_DEVERR_TIMEOUT and the call returns, leaving the device usable.

moe_lora_test_withheld_copy runs the naive fused call with every CTA's
B-slice copy withheld and a 1 ms wait limit, so the wait for that copy is a
flag that nothing sets.  No copy is in flight when a CTA gives up (the
withheld one was never issued).  The test checks the error bit, that the call
returned promptly, that uncovered pairs were not touched, and that the next
ordinary call on the same device is correct."""
import time

import numpy as np
import pytest

import oracle
from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_withheld_copy_times_out_and_the_device_stays_usable():
    import torch
    from helpers import check_close, covered, dev_bf16, dev_i32, host_bf16_bits
    w = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(w)
    x, a, b = dev_bf16(inp.x), dev_bf16(inp.lora_a), dev_bf16(inp.lora_b)
    tk, mp, ids = dev_i32(inp.topk_ids), dev_i32(inp.token_lora_mapping), dev_i32(inp.lora_ids)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = dev_bf16(inp.y_in)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    B.moe_lora_test_withheld_copy(x, a, b, y, tk, mp, ids, w.max_loras, wait_limit_ns=1_000_000, err_flag=err)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) & B.DEVERR_TIMEOUT, int(err.item())
    assert elapsed < 2.0, elapsed                      # 1 ms limits, not the default 4 s
    cov = covered(inp).reshape(-1)
    got = host_bf16_bits(y).reshape(w.M * w.topk, w.N)
    yin = inp.y_in.reshape(w.M * w.topk, w.N)
    assert np.array_equal(got[~cov], yin[~cov])        # uncovered pairs untouched

    # the same device, the ordinary call: correct
    err.zero_()
    y2 = dev_bf16(inp.y_in)
    B.moe_lora_fused_shrink_expand_naive(x, a, b, y2, tk, mp, ids, w.max_loras, add_inputs=True,
                                         path=B.PATH_CUDA_CORE_CLUSTER, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.fused(inp.x, inp.lora_a, inp.lora_b, inp.y_in, inp.topk_ids, inp.token_lora_mapping,
                       inp.lora_ids)
    check_close(host_bf16_bits(y2).reshape(ref.shape), ref, "after a timed-out call")


def test_withheld_copy_rejects_limits_out_of_range():
    import torch
    from helpers import dev_bf16, dev_i32
    w = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(w)
    args = (dev_bf16(inp.x), dev_bf16(inp.lora_a), dev_bf16(inp.lora_b), dev_bf16(inp.y_in),
            dev_i32(inp.topk_ids), dev_i32(inp.token_lora_mapping), dev_i32(inp.lora_ids), w.max_loras)
    for bad in (0, 999, 5_000_000_000):
        with pytest.raises(B.MoeLoraError):
            B.moe_lora_test_withheld_copy(*args, wait_limit_ns=bad)
    torch.cuda.synchronize()

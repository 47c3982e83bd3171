"""GPU parity of the general fused call (moe_lora_fused_shrink_expand_ex)
against the oracle's general definition: router weights (mul_routed_weight),
input rows per pair (the w2 stage), several adapter slices (w13's separate
gate and up adapters) written at an output column offset.

Bar: |gpu - ref| <= 1e-2 + 1e-2 |ref| on every written element; uncovered
pairs and the columns no slice writes stay bit-identical.  Every fused kernel
is forced where the shapes allow; ragged K and N tails, 1 to 4 slices."""
import numpy as np
import pytest

import oracle
from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

from test_gpu_fused import ALL_PATHS, skip_unsupported, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_ex(ex, path, add_inputs=True, pairs=None, adapter_enabled=None):
    """Align + general fused on the device; compare with the oracle (all pairs,
    or the sampled `pairs` at full size).  Returns the largest error."""
    import torch
    from helpers import dev_bf16, dev_i32, host_bf16_bits, check_close
    inp, w = ex.base, ex.base.w
    buf = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    en = dev_i32(adapter_enabled) if adapter_enabled is not None else None
    lora_ids = dev_i32(inp.lora_ids)
    B.moe_lora_align(dev_i32(inp.topk_ids), dev_i32(inp.token_lora_mapping), lora_ids, w.E, w.max_loras,
                     w.block_size, buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded,
                     adapter_enabled=en, workspace=buf.workspace, err_flag=err)
    y = dev_bf16(ex.y_in)
    wts = None if ex.topk_weights is None else torch.from_numpy(ex.topk_weights).cuda()
    B.moe_lora_fused_shrink_expand_ex(
        dev_bf16(ex.x), [dev_bf16(a) for a in ex.lora_a], [dev_bf16(b) for b in ex.lora_b], y,
        buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded, lora_ids, w.topk, w.block_size,
        add_inputs=add_inputs, adapter_enabled=en, topk_weights=wts, x_per_pair=ex.x_per_pair,
        y_offset=ex.y_offset, path=path, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = host_bf16_bits(y).reshape(w.M * w.topk, -1)
    yin = ex.y_in.reshape(w.M * w.topk, -1)
    ref = oracle.fused_ex(ex.x, ex.lora_a, ex.lora_b, ex.y_in, inp.topk_ids, inp.token_lora_mapping,
                          inp.lora_ids, add_inputs=add_inputs, adapter_enabled=adapter_enabled,
                          topk_weights=ex.topk_weights, x_per_pair=ex.x_per_pair, y_offset=ex.y_offset,
                          pairs=pairs)
    rows = np.arange(w.M * w.topk) if pairs is None else np.asarray(pairs)
    got, yin, ref = got[rows], yin[rows], ref.reshape(len(rows), -1)
    S, N = len(ex.lora_a), w.N
    lo, hi = ex.y_offset, ex.y_offset + S * N
    # columns no slice writes are never touched
    assert np.array_equal(got[:, :lo], yin[:, :lo]) and np.array_equal(got[:, hi:], yin[:, hi:])
    from helpers import covered
    cov = covered(inp, adapter_enabled).reshape(-1)[rows]
    assert np.array_equal(got[~cov], yin[~cov]), "uncovered pairs were modified"
    return check_close(got[:, lo:hi], ref[:, lo:hi], "%s path=%d" % (w.name, path))


OPTIONS = {
    "w13_two_slices": dict(num_slices=2),
    "w2_per_pair_weighted": dict(x_per_pair=True, routed_weights=True),
    "weighted_offset": dict(routed_weights=True, y_offset=16, extra=24),
    "three_slices_offset_per_pair": dict(num_slices=3, x_per_pair=True, y_offset=8, extra=8),
    "four_slices_weighted": dict(num_slices=4, routed_weights=True),
}


def make_ex(w, num_slices=1, x_per_pair=False, routed_weights=False, y_offset=0, extra=0):
    ldy = y_offset + num_slices * w.N + extra
    return gen.make_ex_inputs(w, num_slices=num_slices, x_per_pair=x_per_pair, routed_weights=routed_weights,
                              y_offset=y_offset, ldy=ldy)


@pytest.mark.parametrize("add_inputs", [True, False])
@pytest.mark.parametrize("path", ALL_PATHS + [B.PATH_AUTO])
@pytest.mark.parametrize("opt", sorted(OPTIONS))
@pytest.mark.parametrize("name", ["tiny", "decode_qwen3_w13"])
def test_fused_ex_small_workloads(name, opt, path, add_inputs):
    w = gen.WORKLOADS[name]
    skip_unsupported(w, path)
    run_ex(make_ex(w, **OPTIONS[opt]), path, add_inputs)


@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("seed", range(6))
def test_fused_ex_random_shapes(seed, path):
    """Ragged K and N, every block size, ranks 8..128, with a random mix of the
    options."""
    w = small_workload(200 + seed)
    skip_unsupported(w, path)
    rng = np.random.default_rng(seed)
    opt = dict(num_slices=int(rng.integers(1, 5)), x_per_pair=bool(rng.integers(0, 2)),
               routed_weights=bool(rng.integers(0, 2)), y_offset=8 * int(rng.integers(0, 3)),
               extra=8 * int(rng.integers(0, 3)))
    run_ex(make_ex(w, **opt), path, add_inputs=bool(seed % 2))


@pytest.mark.parametrize("seed", range(6))
def test_fused_ex_random_shapes_cluster_stream(seed):
    """The cluster streaming kernel with a random mix of the options, at its
    ranks (powers of two, 8 .. 128)."""
    w = small_workload(700 + seed, rank=[8, 16, 32, 64, 128][seed % 5])
    rng = np.random.default_rng(seed)
    opt = dict(num_slices=int(rng.integers(1, 5)), x_per_pair=bool(rng.integers(0, 2)),
               routed_weights=bool(rng.integers(0, 2)), y_offset=8 * int(rng.integers(0, 3)),
               extra=8 * int(rng.integers(0, 3)))
    run_ex(make_ex(w, **opt), B.PATH_CUDA_CORE_STREAM, add_inputs=bool(seed % 2))


@pytest.mark.parametrize("rank", [4, 12])
def test_fused_ex_small_ranks_cuda_core(rank):
    w = small_workload(77, rank=rank, K=136, N=264)
    run_ex(make_ex(w, num_slices=2, x_per_pair=True, routed_weights=True, y_offset=8), B.PATH_CUDA_CORE_CLUSTER)


@pytest.mark.parametrize("path", ALL_PATHS)
def test_fused_ex_disabled_adapter(path):
    w = gen.WORKLOADS["tiny"]
    skip_unsupported(w, path)
    ex = make_ex(w, num_slices=2, routed_weights=True)
    enabled = np.ones(w.max_loras, np.int32)
    enabled[int(ex.base.lora_ids[0])] = 0
    run_ex(ex, path, adapter_enabled=enabled)


def test_fused_ex_one_slice_equals_plain_call():
    """The plain entry point is the one-slice case of the general one: same
    bits on the same inputs."""
    import torch
    from helpers import DeviceInputs, gpu_step, dev_bf16
    inp = gen.make_inputs(gen.WORKLOADS["decode_qwen3_w13"])
    d = DeviceInputs(inp)
    y_plain, err = gpu_step(d)
    assert err == 0
    y = d.y_in.clone()
    w = inp.w
    B.moe_lora_fused_shrink_expand_ex(d.x, [d.a], [d.b], y.view(w.M, w.topk, w.N), d.buf.sorted_token_ids,
                                      d.buf.expert_ids, d.buf.num_tokens_post_padded, d.lora_ids, w.topk,
                                      w.block_size)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16))


def test_fused_ex_gptoss_w2_full():
    """The w2 stage as the model runs it: one input row per pair and router
    weights, at the gpt-oss decode size, every pair compared."""
    w = gen.WORKLOADS["decode_gptoss_w2"]
    run_ex(make_ex(w, x_per_pair=True, routed_weights=True), B.PATH_AUTO)


def test_fused_ex_prefill_w13_two_slices_every_element():
    """w13 with separate gate and up adapters at the Mixtral prefill size
    (output rows 2 x 28672 wide), every covered pair and column against the
    oracle."""
    import torch
    from helpers import compare_every_pair, dev_bf16, dev_i32, host_bf16_bits
    w = gen.WORKLOADS["prefill_mixtral_w13"]
    ex = make_ex(w, num_slices=2)
    inp = ex.base
    buf = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lora_ids = dev_i32(inp.lora_ids)
    B.moe_lora_align(dev_i32(inp.topk_ids), dev_i32(inp.token_lora_mapping), lora_ids, w.E, w.max_loras,
                     w.block_size, buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded,
                     workspace=buf.workspace, err_flag=err)
    y = dev_bf16(ex.y_in)
    B.moe_lora_fused_shrink_expand_ex(
        dev_bf16(ex.x), [dev_bf16(a) for a in ex.lora_a], [dev_bf16(b) for b in ex.lora_b], y,
        buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded, lora_ids, w.topk, w.block_size,
        add_inputs=True, path=B.PATH_AUTO, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = host_bf16_bits(y).reshape(w.M * w.topk, -1)
    del y, buf
    torch.cuda.empty_cache()
    compare_every_pair(ex, {"auto": got})

"""GPU parity of the fused call with naive block assignment (no align: one
work item per pair) against the oracle's general definition, and its
agreement, bit for bit, with the sorted cluster kernel (the same per-pair
arithmetic).  Early exit (tokens without an adapter), zero grid, disabled
adapters and out-of-range ids are covered."""
import numpy as np
import pytest

import oracle
from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

from test_gpu_fused import small_workload
from test_gpu_fused_ex import OPTIONS, make_ex

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


NAIVE_PATHS = [B.PATH_CUDA_CORE_CLUSTER, B.PATH_CUDA_CORE_STREAM]


def skip_naive(w, path):
    if path == B.PATH_CUDA_CORE_STREAM and w.rank not in (8, 16, 32, 64, 128):
        pytest.skip("the cluster streaming kernel needs a power-of-two rank of 8 .. 128")


def run_naive(ex, add_inputs=True, adapter_enabled=None, topk_ids=None, mapping=None, lora_ids=None,
              want_err=0, pairs=None, path=B.PATH_CUDA_CORE_CLUSTER):
    import torch
    from helpers import dev_bf16, dev_i32, host_bf16_bits, check_close
    inp, w = ex.base, ex.base.w
    topk_ids = inp.topk_ids if topk_ids is None else topk_ids
    mapping = inp.token_lora_mapping if mapping is None else mapping
    lora_ids = inp.lora_ids if lora_ids is None else lora_ids
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = dev_bf16(ex.y_in)
    wts = None if ex.topk_weights is None else torch.from_numpy(ex.topk_weights).cuda()
    B.moe_lora_fused_shrink_expand_naive(
        dev_bf16(ex.x), [dev_bf16(a) for a in ex.lora_a], [dev_bf16(b) for b in ex.lora_b], y, dev_i32(topk_ids),
        dev_i32(mapping), dev_i32(lora_ids), w.max_loras, add_inputs=add_inputs,
        adapter_enabled=None if adapter_enabled is None else dev_i32(adapter_enabled), topk_weights=wts,
        x_per_pair=ex.x_per_pair, y_offset=ex.y_offset, path=path, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == want_err
    got = host_bf16_bits(y).reshape(w.M * w.topk, -1)
    ref = oracle.fused_ex(ex.x, ex.lora_a, ex.lora_b, ex.y_in, topk_ids, mapping, lora_ids, add_inputs=add_inputs,
                          adapter_enabled=adapter_enabled, topk_weights=ex.topk_weights, x_per_pair=ex.x_per_pair,
                          y_offset=ex.y_offset, pairs=pairs)
    rows = np.arange(w.M * w.topk) if pairs is None else np.asarray(pairs)
    got, ref = got[rows], ref.reshape(len(rows), -1)
    yin = ex.y_in.reshape(w.M * w.topk, -1)[rows]
    lo, hi = ex.y_offset, ex.y_offset + len(ex.lora_a) * w.N
    assert np.array_equal(got[:, :lo], yin[:, :lo]) and np.array_equal(got[:, hi:], yin[:, hi:])
    # uncovered pairs keep y_in bit for bit (the oracle returns y_in there)
    yv = gen.bf16_bits_to_f32(yin).astype(np.float64)
    unc = np.all(ref == yv, axis=1)
    assert np.array_equal(got[unc], yin[unc])
    check_close(got[:, lo:hi], ref[:, lo:hi], "%s naive" % w.name)
    return y


@pytest.mark.parametrize("path", NAIVE_PATHS)
@pytest.mark.parametrize("add_inputs", [True, False])
@pytest.mark.parametrize("opt", sorted(OPTIONS) + ["plain"])
@pytest.mark.parametrize("name", ["tiny", "decode_qwen3_w13", "decode_gptoss_w2"])
def test_naive_workloads(name, opt, add_inputs, path):
    w = gen.WORKLOADS[name]
    ex = make_ex(w, **OPTIONS.get(opt, {}))
    run_naive(ex, add_inputs, path=path)


@pytest.mark.parametrize("path", NAIVE_PATHS)
@pytest.mark.parametrize("seed", range(6))
def test_naive_random_shapes(seed, path):
    w = small_workload(400 + seed, M=int(np.random.default_rng(seed).integers(1, 40)))
    skip_naive(w, path)
    rng = np.random.default_rng(seed)
    opt = dict(num_slices=int(rng.integers(1, 4)), x_per_pair=bool(rng.integers(0, 2)),
               routed_weights=bool(rng.integers(0, 2)), y_offset=8 * int(rng.integers(0, 2)))
    run_naive(make_ex(w, **opt), add_inputs=bool(seed % 2), path=path)


@pytest.mark.parametrize("seed", range(5))
def test_naive_random_shapes_cluster_stream(seed):
    w = small_workload(800 + seed, M=int(np.random.default_rng(seed).integers(1, 40)),
                       rank=[8, 16, 32, 64, 128][seed])
    rng = np.random.default_rng(seed)
    opt = dict(num_slices=int(rng.integers(1, 4)), x_per_pair=bool(rng.integers(0, 2)),
               routed_weights=bool(rng.integers(0, 2)), y_offset=8 * int(rng.integers(0, 2)))
    run_naive(make_ex(w, **opt), add_inputs=bool(seed % 2), path=B.PATH_CUDA_CORE_STREAM)


@pytest.mark.parametrize("rank", [4, 12, 20])
def test_naive_small_ranks(rank):
    w = small_workload(77, rank=rank, K=136, N=264)
    run_naive(make_ex(w, num_slices=2, routed_weights=True))


@pytest.mark.parametrize("path", NAIVE_PATHS)
def test_naive_early_exit_and_zero_grid(path):
    """No token has an adapter: every program exits early and y is unchanged.
    No active slot (zero grid): nothing is launched."""
    import torch
    from helpers import dev_bf16, dev_i32, host_bf16_bits
    w = gen.WORKLOADS["tiny"]
    ex = make_ex(w, num_slices=2)
    run_naive(ex, mapping=np.full(w.M, -1, np.int32), path=path)
    y = dev_bf16(ex.y_in)
    B.moe_lora_fused_shrink_expand_naive(dev_bf16(ex.x), [dev_bf16(a) for a in ex.lora_a],
                                         [dev_bf16(b) for b in ex.lora_b], y, dev_i32(ex.base.topk_ids),
                                         dev_i32(ex.base.token_lora_mapping), dev_i32(np.zeros(0, np.int32)),
                                         w.max_loras, path=path)
    torch.cuda.synchronize()
    assert np.array_equal(host_bf16_bits(y).reshape(ex.y_in.shape), ex.y_in)


@pytest.mark.parametrize("path", NAIVE_PATHS)
def test_naive_disabled_adapter_and_bad_ids(path):
    w = gen.WORKLOADS["decode_qwen3_w13"]
    ex = make_ex(w, routed_weights=True)
    enabled = np.ones(w.max_loras, np.int32)
    enabled[int(ex.base.lora_ids[0])] = 0
    run_naive(ex, adapter_enabled=enabled, path=path)
    topk = ex.base.topk_ids.copy()
    act = set(int(v) for v in ex.base.lora_ids)
    m_cov = [m for m in range(w.M) if int(ex.base.token_lora_mapping[m]) in act]
    topk[m_cov[0], 0] = w.E          # a covered pair with an expert id out of range: flagged, skipped
    topk[m_cov[-1], 1] = -3
    run_naive(ex, topk_ids=topk, want_err=B.DEVERR_EXPERT_ID, path=path)
    ids = np.array(list(ex.base.lora_ids) + [w.max_loras + 2], np.int32)   # bad slot id: flagged
    run_naive(ex, lora_ids=ids, want_err=B.DEVERR_LORA_ID, path=path)


@pytest.mark.parametrize("opt", ["plain", "w2_per_pair_weighted", "three_slices_offset_per_pair"])
@pytest.mark.parametrize("name", ["tiny", "decode_qwen3_w13", "decode_gptoss_w2"])
def test_naive_equals_sorted_cluster_bits(name, opt):
    """Naive and sorted assignment run the same per-pair arithmetic on the
    cluster kernel: with the same cluster size their outputs agree bit for
    bit.  Blocks whose adapters exceed 8 x 12 KB take 12-CTA clusters on the
    sorted path and 8 on the naive one (the K and N slices, hence the fp32
    summation order, differ): there both stay within the oracle's tolerance
    of each other."""
    import torch
    from helpers import dev_bf16, dev_i32
    w = gen.WORKLOADS[name]
    ex = make_ex(w, **OPTIONS.get(opt, {}))
    y_naive = run_naive(ex)
    inp = ex.base
    buf = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size)
    lora_ids = dev_i32(inp.lora_ids)
    B.moe_lora_align(dev_i32(inp.topk_ids), dev_i32(inp.token_lora_mapping), lora_ids, w.E, w.max_loras,
                     w.block_size, buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded,
                     workspace=buf.workspace)
    y = dev_bf16(ex.y_in)
    wts = None if ex.topk_weights is None else torch.from_numpy(ex.topk_weights).cuda()
    B.moe_lora_fused_shrink_expand_ex(
        dev_bf16(ex.x), [dev_bf16(a) for a in ex.lora_a], [dev_bf16(b) for b in ex.lora_b], y,
        buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded, lora_ids, w.topk, w.block_size,
        topk_weights=wts, x_per_pair=ex.x_per_pair, y_offset=ex.y_offset, path=B.PATH_CUDA_CORE_CLUSTER)
    torch.cuda.synchronize()
    twelve = (w.K + w.N) * w.rank * 2 > 8 * 12 * 1024 and w.K // 8 >= 12 and w.N // 8 >= 12
    if not twelve:
        assert torch.equal(y.view(torch.int16), y_naive.view(torch.int16))
    else:
        a, b = y.float(), y_naive.float()
        assert torch.all((a - b).abs() <= 1e-2 + 1e-2 * b.abs())

"""GPU parity of the fused shrink+expand against the CPU oracle.

Every output element must satisfy |gpu - ref| <= 1e-2 + 1e-2 |ref| against the
oracle's unrounded fp64 value; pairs the path does not cover must be left
bit-identical.  Both paths (CUDA cores, tcgen05) are forced where the shapes
allow, on the five workloads, on random shapes with ragged K and N tails, on
exact-integer inputs (bit-exact) and with NaN-poisoned inactive slots."""
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


ALL_PATHS = [B.PATH_CUDA_CORE_CLUSTER, B.PATH_CUDA_CORE_STREAM, B.PATH_TCGEN05]


def skip_unsupported(w, path):
    """The tensor-core kernel needs rank % 8 == 0, the cluster streaming kernel
    a rank of 8, 16, 32, 64 or 128."""
    if path == B.PATH_TCGEN05 and w.rank % 8:
        pytest.skip("path needs rank % 8 == 0")
    if path == B.PATH_CUDA_CORE_STREAM and w.rank not in (8, 16, 32, 64, 128):
        pytest.skip("path needs a power-of-two rank of 8 .. 128")


def run_and_compare_full(inp, path, add_inputs=True, adapter_enabled=None, variant=B.ALIGN_AUTO):
    from helpers import DeviceInputs, gpu_step, host_bf16_bits, check_close, covered
    d = DeviceInputs(inp, variant)
    y, err = gpu_step(d, add_inputs=add_inputs, path=path, variant=variant, adapter_enabled=adapter_enabled)
    assert err == 0, err
    got = host_bf16_bits(y).reshape(inp.y_in.shape)
    ref = oracle.fused(inp.x, inp.lora_a, inp.lora_b, inp.y_in, inp.topk_ids, inp.token_lora_mapping,
                       inp.lora_ids, add_inputs=add_inputs, adapter_enabled=adapter_enabled)
    cov = covered(inp, adapter_enabled)
    assert np.array_equal(got[~cov], inp.y_in[~cov]), "uncovered pairs were modified"
    return check_close(got, ref, "%s path=%d" % (inp.w.name, path))


@pytest.mark.parametrize("add_inputs", [True, False])
@pytest.mark.parametrize("path", ALL_PATHS + [B.PATH_CUDA_CORE, B.PATH_AUTO])
@pytest.mark.parametrize("name", ["tiny", "decode_qwen3_w13", "decode_gptoss_w2"])
def test_fused_small_workloads_full(name, path, add_inputs):
    skip_unsupported(gen.WORKLOADS[name], path)
    inp = gen.make_inputs(gen.WORKLOADS[name])
    run_and_compare_full(inp, path, add_inputs)


def small_workload(seed, **kw):
    rng = np.random.default_rng(seed)
    base = dict(name="rand%d" % seed, M=int(rng.integers(1, 200)), K=8 * int(rng.integers(1, 120)),
                N=8 * int(rng.integers(1, 150)), E=int(rng.integers(1, 40)), topk=1, max_loras=int(rng.integers(1, 5)),
                num_active_loras=1, rank=8 * int(rng.integers(1, 17)), block_size=int(rng.choice([16, 32, 64, 128])),
                mapping="uniform_with_none", experts="uniform", seed=seed)
    base["topk"] = int(rng.integers(1, min(base["E"], 8) + 1))
    base["num_active_loras"] = int(rng.integers(1, base["max_loras"] + 1))
    base.update(kw)
    return gen.Workload(**base)


@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("seed", range(12))
def test_fused_random_shapes(seed, path):
    """Ragged K (not a multiple of the 64-wide K tile) and N (not a multiple of
    the 128-wide N tile), every block size, ranks 8..128."""
    skip_unsupported(small_workload(seed), path)
    inp = gen.make_inputs(small_workload(seed))
    run_and_compare_full(inp, path, add_inputs=bool(seed % 2))


@pytest.mark.parametrize("seed", range(12))
def test_fused_random_shapes_cluster_stream(seed):
    """The cluster streaming kernel on random shapes with its ranks (8 .. 128,
    powers of two): ragged K and N, every block size, both add modes."""
    rank = [8, 16, 32, 64, 128][seed % 5]
    inp = gen.make_inputs(small_workload(600 + seed, rank=rank))
    run_and_compare_full(inp, B.PATH_CUDA_CORE_STREAM, add_inputs=bool(seed % 2))


@pytest.mark.parametrize("rank", [4, 12, 20])
def test_fused_small_ranks_cuda_core(rank):
    inp = gen.make_inputs(small_workload(77, rank=rank, K=136, N=264))
    run_and_compare_full(inp, B.PATH_CUDA_CORE_CLUSTER)


@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("rank", [8, 16, 64, 128])
def test_fused_ranks(rank, path):
    w = small_workload(5, rank=rank, M=96, K=520, N=392, E=6, topk=2, block_size=32)
    skip_unsupported(w, path)
    inp = gen.make_inputs(w)
    run_and_compare_full(inp, path)


@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("rank,nnz", [(8, 16), (16, 8), (64, 2), (128, 1)])
def test_fused_exact_integer_case(path, rank, nnz):
    """x, B in {-1, 0, 1}; each row of A has nnz entries in {-1, 1}; y_in in
    [-4, 4].  Then |t| <= nnz and |ref| <= rank * nnz + 4 <= 260 with every
    partial sum an integer, exact in fp32 and in bf16 up to 256 -- the GPU must
    equal the oracle bit for bit.  K = 264 spans five 64-wide K tiles with a
    ragged tail and N = 392 four 128-wide N tiles (also ragged), so this pins the
    tensor-core operand layouts, the K accumulation, the cluster reduction and
    the tails."""
    from helpers import DeviceInputs, gpu_step, host_bf16_bits
    w = gen.Workload("int", M=70, K=264, N=392, E=3, topk=2, max_loras=2, num_active_loras=2, rank=rank,
                     block_size=64, mapping="uniform_with_none",
                     experts="uniform", seed=3)
    inp = gen.make_inputs(w)
    rng = np.random.default_rng(8)
    f2b = gen.f32_to_bf16_bits
    inp.x = f2b(rng.integers(-1, 2, size=inp.x.shape).astype(np.float32))
    a = np.zeros(inp.lora_a.shape, np.float32)
    for idx in np.ndindex(*a.shape[:3]):
        cols = rng.choice(w.K, nnz, replace=False)
        a[idx][cols] = rng.choice([-1.0, 1.0], nnz)
    inp.lora_a = f2b(a)
    inp.lora_b = f2b(rng.integers(-1, 2, size=inp.lora_b.shape).astype(np.float32))
    inp.y_in = f2b(rng.integers(-4, 5, size=inp.y_in.shape).astype(np.float32))
    for add in (True, False):
        d = DeviceInputs(inp)
        y, err = gpu_step(d, add_inputs=add, path=path)
        assert err == 0
        got = gen.bf16_bits_to_f32(host_bf16_bits(y).reshape(inp.y_in.shape)).astype(np.float64)
        ref = oracle.fused(inp.x, inp.lora_a, inp.lora_b, inp.y_in, inp.topk_ids, inp.token_lora_mapping,
                           inp.lora_ids, add_inputs=add)
        assert np.abs(ref).max() <= 256 or rank * nnz + 4 > 256
        bad = got != ref
        assert not bad.any(), "first mismatch at %s: got %r ref %r" % (
            tuple(np.argwhere(bad)[0]), got[bad][0], ref[bad][0])


@pytest.mark.parametrize("path", ALL_PATHS)
def test_fused_disabled_adapter_and_poison(path):
    """Inactive and disabled slots hold NaN in A and B; the output stays finite
    and their tokens keep y_in."""
    w = gen.Workload("poison", M=120, K=256, N=256, E=8, topk=2, max_loras=4, num_active_loras=3, rank=16,
                     block_size=16, mapping="uniform_with_none", experts="uniform", seed=11)
    inp = gen.make_inputs(w)
    enabled = np.ones(4, np.int32)
    enabled[inp.lora_ids[0]] = 0
    inp.lora_a[inp.lora_ids[0]] = gen.BF16_QNAN
    inp.lora_b[inp.lora_ids[0]] = gen.BF16_QNAN
    run_and_compare_full(inp, path, adapter_enabled=enabled)


@pytest.mark.parametrize("path", ALL_PATHS)
def test_fused_no_covered_pairs(path):
    from helpers import DeviceInputs, gpu_step, host_bf16_bits
    w = gen.Workload("none", M=40, K=64, N=128, E=4, topk=2, max_loras=2, num_active_loras=2, rank=8,
                     block_size=16, mapping="uniform_with_none", experts="uniform", seed=1)
    inp = gen.make_inputs(w)
    inp.token_lora_mapping[:] = -1
    d = DeviceInputs(inp)
    y, err = gpu_step(d, path=path)
    assert err == 0 and np.array_equal(host_bf16_bits(y).reshape(inp.y_in.shape), inp.y_in)


@pytest.mark.parametrize("shape", ["two_pairs_clusters", "one_pair"])
def test_fused_stream_units_in_turn(shape):
    """More aligned blocks than the streaming kernel's list builder counts in
    one pass (1280): it takes the units in turn instead of the balanced list.
    Two pairs per item over 4-CTA clusters (pairs beyond the (LoRA, expert)
    pairs), and one pair per item (pairs no more than those).  Every element
    against the oracle."""
    if shape == "two_pairs_clusters":
        w = gen.Workload("stream_in_turn_2", M=4096, K=128, N=128, E=64, topk=8, max_loras=2, num_active_loras=2,
                         rank=16, block_size=16, mapping="uniform", experts="uniform", seed=5)
    else:
        w = gen.Workload("stream_in_turn_1", M=2048, K=64, N=64, E=1024, topk=8, max_loras=16, num_active_loras=16,
                         rank=16, block_size=16, mapping="uniform", experts="uniform", seed=6)
    plan = B.fused_plan(w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras, w.block_size,
                        path=B.PATH_CUDA_CORE_STREAM, sm_count=152, max_smem_per_block=232448)
    assert plan["pairs_per_group"] == (2 if shape == "two_pairs_clusters" else 1), plan
    inp = gen.make_inputs(w)
    # the routing really has more blocks than one counting pass covers
    per_slot = [np.bincount(inp.topk_ids.reshape(-1)[np.repeat(inp.token_lora_mapping, w.topk) == l],
                            minlength=w.E) for l in inp.lora_ids]
    blocks = sum(int(np.sum((c + w.block_size - 1) // w.block_size)) for c in per_slot)
    assert blocks > 1280, blocks
    run_and_compare_full(inp, B.PATH_CUDA_CORE_STREAM, add_inputs=True)


def test_fused_stream_flags_out_of_layout_block():
    """A block whose pair follows a sentinel (a layout moe_lora_align never
    writes): the streaming kernel's balanced list counts each block's pairs up
    to its first sentinel, so it flags the block (DEVERR_PAIR_ID) instead of
    dropping the pair silently."""
    import torch
    from helpers import DeviceInputs
    w = gen.Workload("stream_layout", M=16, K=64, N=64, E=64, topk=2, max_loras=2, num_active_loras=2, rank=16,
                     block_size=16, mapping="uniform", experts="uniform", seed=3)
    assert B.fused_plan(w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras, w.block_size,
                        path=B.PATH_CUDA_CORE_STREAM, sm_count=152, max_smem_per_block=232448)["pairs_per_group"] == 1
    inp = gen.make_inputs(w)
    d = DeviceInputs(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_lora_align(d.topk_ids, d.mapping, d.lora_ids, w.E, w.max_loras, w.block_size, d.buf.sorted_token_ids,
                     d.buf.expert_ids, d.buf.num_tokens_post_padded, workspace=d.buf.workspace, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the first block of the first slot: swap its first pair with the sentinel after it
    l = int(inp.lora_ids[0])
    row = d.buf.sorted_token_ids[l]
    sentinel = w.M * w.topk
    blk = row[:w.block_size].clone()
    n_real = int((blk < sentinel).sum().item())
    assert 1 <= n_real < w.block_size
    row[n_real - 1], row[n_real] = sentinel, int(blk[n_real - 1].item())
    y = d.y_in.clone()
    B.moe_lora_fused_shrink_expand(d.x, d.a, d.b, y, d.buf.sorted_token_ids, d.buf.expert_ids,
                                   d.buf.num_tokens_post_padded, d.lora_ids, w.topk, w.block_size, add_inputs=True,
                                   path=B.PATH_CUDA_CORE_STREAM, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_PAIR_ID


@pytest.mark.parametrize("variant", [B.ALIGN_SMEM, B.ALIGN_GLOBAL, B.ALIGN_CLUSTER])
def test_fused_after_either_align_variant(variant):
    inp = gen.make_inputs(gen.WORKLOADS["decode_gptoss_w2"])
    run_and_compare_full(inp, B.PATH_AUTO, variant=variant)


# ---------------------------------------------------------------- full size

def full_size_outputs(inp, paths, add_inputs=True):
    """Run align + fused at full size once per path; return host copies of y
    ([M*topk, N] uint16) keyed by path."""
    import torch
    from helpers import DeviceInputs, gpu_step, host_bf16_bits
    w = inp.w
    d = DeviceInputs(inp)
    outs = {}
    for path in paths:
        y, err = gpu_step(d, add_inputs=add_inputs, path=path)
        assert err == 0, (path, err)
        outs["path%d" % path] = host_bf16_bits(y).reshape(w.M * w.topk, w.N)
        del y
    del d
    torch.cuda.empty_cache()
    return outs


@pytest.mark.parametrize("name", ["prefill_mixtral_w13", "large_e_nact1", "large_e_nact4", "large_e_nact8"])
def test_fused_full_size_every_element(name):
    """Full-size workloads on the kernel AUTO picks (the tensor-core kernel:
    the persistent work split, its rings and its straddled units only occur
    at these sizes), every covered pair and every column against the oracle.
    On the prefill shape the CUDA-core cluster kernel runs too."""
    from helpers import as_ex, compare_every_pair
    inp = gen.make_inputs(gen.WORKLOADS[name])
    w = inp.w
    assert B.fused_resolve_path(w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras, w.block_size, 1,
                                B.PATH_AUTO) == B.PATH_TCGEN05
    paths = [B.PATH_AUTO] + ([B.PATH_CUDA_CORE_CLUSTER] if name.startswith("prefill") else [])
    outs = full_size_outputs(inp, paths)
    compare_every_pair(as_ex(inp), outs)


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("N,rank", [(28672, 64), (14336, 128)])
def test_fused_long_rows_small_batch_auto(M, N, rank):
    """Small batches whose adapter rows are too long for the cluster kernel's
    shared memory (one Mixtral-sized w13 token at rank 64 or 128): AUTO sends
    them to the tensor-core kernel.  Every element against the oracle."""
    from helpers import as_ex, compare_every_pair
    w = gen.Workload("long_rows_m%d_n%d_r%d" % (M, N, rank), M=M, K=4096, N=N, E=8, topk=2, max_loras=2,
                     num_active_loras=2, rank=rank, block_size=16, mapping="uniform", experts="uniform", seed=21)
    assert B.fused_resolve_path(M, w.topk, w.E, w.K, N, rank, w.num_active_loras, w.block_size, 1,
                                B.PATH_AUTO) == B.PATH_TCGEN05
    inp = gen.make_inputs(w)
    for add in (True, False):
        outs = full_size_outputs(inp, [B.PATH_AUTO], add_inputs=add)
        compare_every_pair(as_ex(inp), outs, add_inputs=add)

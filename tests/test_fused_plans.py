"""The launch plans of the fused kernels on a GB300 (152 SMs, 227 KB of
opt-in shared memory per block), computed on the host: pinned for the
benchmark workloads (a change to the shared-memory layout that costs ring
depth shows up here, not only in a benchmark), and checked for invariants
over a sweep of shapes."""
import itertools

import pytest

from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

GB300 = dict(sm_count=152, max_smem_per_block=232448)


def plan_of(w, **kw):
    return B.fused_plan(w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras, w.block_size, **kw, **GB300)


# (kernel, shrink stages, lag, expand stages, T buffers, TMEM columns) for the
# tensor-core kernel; (kernel, CTAs per cluster, pairs per group) for the
# CUDA-core kernels.  These are the plans the measured numbers were taken with.
PINNED = {
    "decode_gptoss_w2": (B.PATH_CUDA_CORE_STREAM, 1, 1),
    "prefill_mixtral_w13": (B.PATH_TCGEN05, 10, 4, 6, 1, 256),
    "large_e_nact1": (B.PATH_TCGEN05, 4, 1, 2, 1, 256),
    "large_e_nact8": (B.PATH_TCGEN05, 4, 1, 2, 1, 256),
    "decode_qwen3_w13": (B.PATH_CUDA_CORE_CLUSTER, 12, 8),
    "tiny": (B.PATH_CUDA_CORE_CLUSTER, 1, 8),
}


@pytest.mark.parametrize("name", sorted(PINNED))
def test_benchmark_plans_pinned(name):
    p = plan_of(gen.WORKLOADS[name])
    want = PINNED[name]
    if want[0] == B.PATH_TCGEN05:
        got = (p["kernel"], p["s_sh"], p["lag"], p["s_ex"], p["t_bufs"], p["tmem_cols"])
    else:
        got = (p["kernel"], p["cluster"], p["pairs_per_group"])
    assert got == want, p


SHAPES = list(itertools.product([16, 256, 4096], [2, 8], [8, 128, 256], [1024, 4096, 7168], [1536, 4096, 28672],
                                [8, 16, 64, 128], [16, 64, 128]))


@pytest.mark.parametrize("path", [B.PATH_TCGEN05, B.PATH_CUDA_CORE_CLUSTER, B.PATH_CUDA_CORE_STREAM])
def test_plan_invariants(path):
    checked = 0
    for M, topk, E, K, N, r, bs in SHAPES:
        if topk > E:
            continue
        try:
            p = B.fused_plan(M, topk, E, K, N, r, 2, bs, path=path, **GB300)
        except B.MoeLoraError:
            continue
        checked += 1
        assert p["kernel"] == path
        assert 0 < p["smem_bytes"] <= GB300["max_smem_per_block"]
        if path == B.PATH_TCGEN05:
            # a next B tile loads under the MMA -- except at block size 128 with
            # rank > 64, where two expand stages (64 KB each) do not fit beside the
            # 32 KB shrink stages and the 64 KB T buffer
            if not (bs == 128 and r > 64):
                assert p["s_ex"] >= 2, (M, topk, E, K, N, r, bs, p)
            assert p["s_sh"] >= 2 * p["lag"] + 1, p                       # the shrink producers cannot deadlock
            assert p["tmem_cols"] in (32, 64, 128, 256, 512)
            per_sm = max(1, (228 * 1024) // (p["smem_bytes"] + 1024))
            assert per_sm * p["tmem_cols"] <= 512, p                      # co-resident CTAs fit in TMEM
            assert p["threads"] == 416 and 1 <= p["grid"] <= 152 * per_sm
        elif path == B.PATH_CUDA_CORE_STREAM:
            # clusters of 1..8 CTAs, one per SM; each CTA holds at least one
            # 8-wide chunk of K and of N; a ring of at least 4 stages
            C = p["cluster"]
            assert C in (1, 2, 4, 8) and C <= min(K // 8, N // 8), (K, N, p)
            assert p["grid"] % C == 0 and 1 <= p["grid"] <= 2 * 152, p
            assert p["s_sh"] >= 4 and p["threads"] == 320, p
            assert p["smem_bytes"] <= 113 * 1024, p
            # one pair per item where the pairs are no more than the (LoRA,
            # expert) pairs, else two over clusters of up to 4 CTAs
            single = M * topk <= E * 2   # nact = 2 in these plans
            assert p["pairs_per_group"] == (1 if single else 2), p
            assert C == 1 if single else C <= 4, p
            assert r * p["s_ex"] * 2 <= 16384 and p["t_bufs"] * r * 2 <= 16384, p   # A box, B rows per stage
        else:
            assert 1 <= p["cluster"] <= 16 and p["pairs_per_group"] in (1, 2, 8)
    assert checked > 100


def test_cluster_never_leaves_a_cta_without_columns():
    """Every CTA of a cluster holds at least one 8-element chunk of K and of N
    (so each adapter copy is at least 16 bytes), down to the smallest rows."""
    checked = rejected = 0
    for K, N, r in itertools.product([8, 16, 24, 40, 64, 136, 1024], [8, 16, 24, 40, 64, 136, 1024],
                                     [4, 8, 12, 16, 64, 128]):
        try:
            p = B.fused_plan(16, 2, 8, K, N, r, 2, 16, path=B.PATH_CUDA_CORE_CLUSTER, **GB300)
        except B.MoeLoraError:
            # only when even the largest cluster leaves a CTA more A and B rows
            # than shared memory holds
            C = min(16, K // 8, N // 8)
            kslice, nslice = -(-(K // 8) // C) * 8, -(-(N // 8) // C) * 8
            assert r * (kslice + 8) * 2 + nslice * r * 2 > GB300["max_smem_per_block"], (K, N, r)
            rejected += 1
            continue
        assert 1 <= p["cluster"] <= min(16, K // 8, N // 8), (K, N, r, p)
        checked += 1
    assert checked + rejected == 7 * 7 * 6 and rejected <= 2


def test_auto_sends_rows_too_long_for_the_cluster_kernel_to_tensor_cores():
    """One-token decode with w13-sized rows: N * rank beyond what 16 cluster
    CTAs hold in shared memory goes to the tensor-core kernel; short rows stay
    on the cluster kernel."""
    R = B.fused_resolve_path
    assert R(1, 1, 8, 4096, 28672, 64, 1, 16) == B.PATH_TCGEN05
    assert R(1, 2, 8, 4096, 14336, 128, 1, 16) == B.PATH_TCGEN05
    assert R(1, 1, 8, 4096, 1536, 64, 1, 16) == B.PATH_CUDA_CORE_CLUSTER
    with pytest.raises(B.MoeLoraError):   # the cluster kernel itself cannot hold these rows
        B.fused_plan(1, 1, 8, 4096, 28672, 64, 1, 16, path=B.PATH_CUDA_CORE_CLUSTER, **GB300)
    assert B.fused_plan(1, 1, 8, 4096, 28672, 64, 1, 16, **GB300)["kernel"] == B.PATH_TCGEN05


def test_auto_plans_every_shape_with_a_full_k_tile():
    """AUTO finds a kernel for every supported shape with K >= 64, N >= 32
    and rank % 8 == 0, from one-token decode to prefill batches."""
    n = 0
    for M, topk, E, K, N, r, bs, nact in itertools.product(
            [1, 16, 200, 4096], [1, 8], [8, 256], [64, 1024, 7168], [32, 1536, 14336, 28672], [8, 64, 128],
            [16, 128], [1, 4]):
        if topk > E:
            continue
        p = B.fused_plan(M, topk, E, K, N, r, nact, bs, **GB300)
        assert p["kernel"] in (B.PATH_TCGEN05, B.PATH_CUDA_CORE_CLUSTER, B.PATH_CUDA_CORE_STREAM)
        if p["kernel"] == B.PATH_CUDA_CORE_STREAM:   # decode batches with large adapters only
            assert M * topk < 1024 and r in (8, 16, 32, 64, 128)
        if M * topk >= 1024:
            assert p["kernel"] == B.PATH_TCGEN05
        n += 1
    assert n > 1000


def test_auto_streams_large_decode_adapters():
    """Decode batches whose adapters, by the block bound, exceed 48 MB go to
    the cluster streaming kernel (the gpt-oss-shaped w2 decode); small
    adapters stay on the one-cluster-per-block kernel (the Qwen3-shaped w13
    decode); prefill-sized batches go to tensor cores."""
    R = B.fused_resolve_path
    assert R(64, 4, 128, 2880, 2880, 64, 6, 16) == B.PATH_CUDA_CORE_STREAM
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16) == B.PATH_CUDA_CORE_CLUSTER
    assert R(8192, 2, 8, 4096, 28672, 16, 4, 64) == B.PATH_TCGEN05
    assert R(64, 4, 128, 2880, 2880, 72, 6, 16) == B.PATH_TCGEN05          # rank the streaming kernel lacks


def test_plan_rejects_what_the_kernel_cannot_run():
    with pytest.raises(B.MoeLoraError):
        B.fused_plan(64, 4, 128, 2880, 2880, 12, 6, 16, path=B.PATH_TCGEN05, **GB300)   # rank % 8 != 0
    with pytest.raises(B.MoeLoraError):
        B.fused_plan(64, 4, 128, 2880, 2880, 12, 6, 16, path=B.PATH_CUDA_CORE_STREAM, **GB300)  # rank % 8 != 0


def test_cluster_stream_plan_gptoss_decode():
    """The cluster streaming kernel on the gpt-oss decode shape: 256 pairs
    against 768 (LoRA, expert) pairs, so one pair per work item on CTAs of
    their own (one per pair), two CTAs of 10 warps per SM, each with a ring of
    six 16.25 KB stages (A boxes of 64 ranks x 128 columns, B pieces of 128
    rows x 64 ranks, each with the pair's x or y_in piece).  A prefill batch of
    the same shape takes two pairs per item over clusters of 4 CTAs."""
    p = B.fused_plan(64, 4, 128, 2880, 2880, 64, 6, 16, path=B.PATH_CUDA_CORE_STREAM, **GB300)
    assert p["kernel"] == B.PATH_CUDA_CORE_STREAM
    assert p["cluster"] == 1 and p["pairs_per_group"] == 1 and p["grid"] == 256
    assert p["s_sh"] == 6 and p["threads"] == 320                        # ring stages, threads
    assert p["s_ex"] == 128 and p["t_bufs"] == 128                      # A columns, B rows per stage
    assert p["smem_bytes"] <= 113 * 1024                                # two CTAs share an SM
    q = B.fused_plan(2048, 8, 128, 2880, 2880, 64, 6, 16, path=B.PATH_CUDA_CORE_STREAM, **GB300)
    assert q["cluster"] == 4 and q["pairs_per_group"] == 2 and q["grid"] == 304

"""Seeded synthetic inputs for the multi-LoRA MoE adapter path.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It draws inputs only; it holds none of the
method's arithmetic (no counting, padding, scatter or contraction).

Workloads are shaped like the models the vLLM pages benchmark (vLLM PR #29257
"Lora MoE Align Improvements", gpt-oss-120b serving run; vLLM PR #29708
"[LoRA] Support FusedMoE LoRA Triton kernel for mxfp4", gpt-oss-20b serving
run; the prhub.com.cn summary of vLLM PR #42290, section "Implementation
breakdown", step 4, which benchmarks qwen3moe-shaped inputs).  No dataset or
trained weight is used: every value comes from numpy's PCG64 generator.

Routing is drawn from one stream, `numpy.random.default_rng(seed)`, in the
order

    active LoRA set -> topk_ids -> token_lora_mapping

Tensors are drawn in chunks of 2**24 elements, chunk c of a tensor from its
own stream `numpy.random.default_rng([seed, tag, slice, slot, c])`, so that
the value of every element is fixed by definition whatever the tensor size,
and chunks can be drawn on several host threads at once.  Tags: 1 x,
2 A, 3 B, 4 y_in, 5 x with one row per pair, 6 a wide y_in (output offset or
row stride); `slice` is the adapter slice (0 for the plain call) and `slot`
the LoRA slot of an adapter (0 for x and y_in).  Router weights come from
`default_rng([seed, 7])`.

Value distributions: x ~ N(0,1); A[l,e] ~ N(0, 1/K) (K = input dim of the
adapter); B[l,e] ~ N(0, 1/r); y_in ~ N(0,1); router weights a softmax over
each token's top-k of N(0,1) draws (float32, positive, summing to 1 per token,
like a router's top-k probabilities).  Normals are drawn as float32 and
rounded to bf16 with round-to-nearest-even.  Adapter slots that are not in the
active set are filled with a bf16 quiet NaN (0x7FC0) so that any read of an
inactive slot shows up in the output.

bf16 values are carried as numpy uint16 arrays holding the raw bit patterns.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
import threading
from typing import Optional

import numpy as np

BF16_QNAN = np.uint16(0x7FC0)
# Tensors are drawn in chunks of this many elements, each chunk from its own
# keyed stream.
_CHUNK = 1 << 24


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution parameters of one synthetic workload."""

    name: str
    M: int              # tokens
    K: int              # adapter input dim (hidden size for w13, intermediate for w2)
    N: int              # adapter output dim
    E: int              # experts
    topk: int
    max_loras: int
    num_active_loras: int
    rank: int
    block_size: int
    mapping: str        # "uniform_with_none" | "none10" | "uniform"
    experts: str        # "uniform" | "zipf"
    zipf_s: float = 0.0
    seed: int = 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the specification, named by what they are.
WORKLOADS = {
    # Tiny: every step is checked against the oracle on all outputs.
    "tiny": Workload("tiny", M=16, K=256, N=512, E=8, topk=2, max_loras=2,
                     num_active_loras=2, rank=8, block_size=16,
                     mapping="uniform_with_none", experts="uniform"),
    # Decode, Qwen3-MoE-30B-A3B-shaped w13 LoRA (gate_up = 2 x 768).
    "decode_qwen3_w13": Workload("decode_qwen3_w13", M=16, K=2048, N=1536, E=128,
                                 topk=8, max_loras=4, num_active_loras=2, rank=16,
                                 block_size=16, mapping="uniform_with_none",
                                 experts="zipf", zipf_s=1.1),
    # Decode, gpt-oss-120b-shaped w2 LoRA.
    "decode_gptoss_w2": Workload("decode_gptoss_w2", M=64, K=2880, N=2880, E=128,
                                 topk=4, max_loras=6, num_active_loras=6, rank=64,
                                 block_size=16, mapping="none10", experts="uniform"),
    # Prefill, Mixtral-8x7B-shaped w13 LoRA (gate_up = 2 x 14336).
    "prefill_mixtral_w13": Workload("prefill_mixtral_w13", M=8192, K=4096, N=28672,
                                    E=8, topk=2, max_loras=4, num_active_loras=4,
                                    rank=16, block_size=64, mapping="uniform",
                                    experts="uniform"),
    # Large expert count, rank 128 (the one-shot rank limit), 1/4/8 active.
    "large_e_nact1": Workload("large_e_nact1", M=4096, K=7168, N=4096, E=256, topk=8,
                              max_loras=8, num_active_loras=1, rank=128, block_size=64,
                              mapping="uniform_with_none", experts="zipf", zipf_s=1.2),
    "large_e_nact4": Workload("large_e_nact4", M=4096, K=7168, N=4096, E=256, topk=8,
                              max_loras=8, num_active_loras=4, rank=128, block_size=64,
                              mapping="uniform_with_none", experts="zipf", zipf_s=1.2),
    "large_e_nact8": Workload("large_e_nact8", M=4096, K=7168, N=4096, E=256, topk=8,
                              max_loras=8, num_active_loras=8, rank=128, block_size=64,
                              mapping="uniform_with_none", experts="zipf", zipf_s=1.2),
    # Profiling-sized cases.  A full ncu capture replays each launch dozens of
    # times and saves device memory between replays, so it runs on inputs of a
    # few GB at most: the prefill shape at a quarter of the tokens (y still
    # larger than L2), and the rank-128 large-E shape with one adapter slot
    # allocated (the same active work as large_e_nact1 without the 5 GB of
    # inactive slots).
    "prefill_mixtral_w13_m2048": Workload("prefill_mixtral_w13_m2048", M=2048, K=4096, N=28672, E=8, topk=2,
                                          max_loras=4, num_active_loras=4, rank=16, block_size=64,
                                          mapping="uniform", experts="uniform"),
    "large_e_l1": Workload("large_e_l1", M=4096, K=7168, N=4096, E=256, topk=8, max_loras=1,
                           num_active_loras=1, rank=128, block_size=64, mapping="uniform_with_none",
                           experts="zipf", zipf_s=1.2),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return raw bits.

    Inputs must be finite (they are normals here)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_TAG_X, _TAG_A, _TAG_B, _TAG_Y, _TAG_X_PAIR, _TAG_Y_WIDE, _TAG_WEIGHTS = 1, 2, 3, 4, 5, 6, 7

_pool = None
_pool_lock = threading.Lock()
_scratch = threading.local()


def _executor() -> concurrent.futures.ThreadPoolExecutor:
    global _pool
    with _pool_lock:
        if _pool is None:
            try:
                n = len(os.sched_getaffinity(0))
            except AttributeError:
                n = os.cpu_count() or 1
            _pool = concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(32, n)))
    return _pool


def _draw_chunk(out: np.ndarray, key, scale: float) -> None:
    """out[:] = bf16(scale * N(0,1) draws of stream `key`), float32 draws."""
    n = out.size
    buf = getattr(_scratch, "f32", None)
    if buf is None or buf.size < n:
        buf = _scratch.f32 = np.empty(_CHUNK, np.float32)
        _scratch.u32 = np.empty(_CHUNK, np.uint32)
    v = buf[:n]
    np.random.default_rng(key).standard_normal(dtype=np.float32, out=v)
    if scale != 1.0:
        v *= np.float32(scale)
    # round to nearest even, in place: (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    u = v.view(np.uint32)
    t = _scratch.u32[:n]
    np.right_shift(u, np.uint32(16), out=t)
    t &= np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    out[...] = t


def _normal_bf16_into(out: np.ndarray, seed: int, tag: int, sl: int, slot: int, scale: float) -> None:
    """Fill the contiguous uint16 array `out` chunk by chunk, chunk c from the
    stream [seed, tag, sl, slot, c] (chunks drawn on the host threads)."""
    flat = out.reshape(-1)
    n = flat.size
    jobs = [_executor().submit(_draw_chunk, flat[s:min(n, s + _CHUNK)], [seed, tag, sl, slot, s // _CHUNK], scale)
            for s in range(0, n, _CHUNK)]
    for j in jobs:
        j.result()


def _normal_bf16(shape, seed: int, tag: int, sl: int, slot: int, scale: float) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    _normal_bf16_into(out, seed, tag, sl, slot, scale)
    return out


def _adapters(w: "Workload", lora_ids, sl: int):
    """A [L, E, r, K] and B [L, E, N, r] of slice `sl`: N(0, 1/K) and N(0, 1/r)
    in the listed slots, bf16 NaN elsewhere."""
    L, E, r, K, N = w.max_loras, w.E, w.rank, w.K, w.N
    a = np.full((L, E, r, K), BF16_QNAN, dtype=np.uint16)
    b = np.full((L, E, N, r), BF16_QNAN, dtype=np.uint16)
    for l in lora_ids:
        _normal_bf16_into(a[l], w.seed, _TAG_A, sl, int(l), 1.0 / np.sqrt(K))
        _normal_bf16_into(b[l], w.seed, _TAG_B, sl, int(l), 1.0 / np.sqrt(r))
    return a, b


@dataclasses.dataclass
class Inputs:
    """One batch of inputs; arrays are numpy, bf16 as uint16 bit patterns."""

    w: Workload
    lora_ids: np.ndarray            # int32 [num_active_loras], sorted active slots
    topk_ids: np.ndarray            # int32 [M, topk]
    token_lora_mapping: np.ndarray  # int32 [M], -1 = no adapter
    x: Optional[np.ndarray]         # uint16 [M, K]
    lora_a: Optional[np.ndarray]    # uint16 [max_loras, E, r, K]
    lora_b: Optional[np.ndarray]    # uint16 [max_loras, E, N, r]
    y_in: Optional[np.ndarray]      # uint16 [M, topk, N]


def expert_probabilities(w: Workload) -> Optional[np.ndarray]:
    """Router distribution over experts: None = uniform; bounded Zipf p(e) ~ (e+1)^-s."""
    if w.experts == "uniform":
        return None
    if w.experts == "zipf":
        p = np.arange(1, w.E + 1, dtype=np.float64) ** (-w.zipf_s)
        return p / p.sum()
    raise ValueError(w.experts)


def draw_routing(w: Workload, rng: np.random.Generator):
    """Active set, topk_ids and token_lora_mapping, in the fixed draw order."""
    L, nact = w.max_loras, w.num_active_loras
    if nact == L:
        lora_ids = np.arange(L, dtype=np.int32)
    else:
        lora_ids = np.sort(rng.choice(L, nact, replace=False)).astype(np.int32)
    p = expert_probabilities(w)
    topk_ids = np.empty((w.M, w.topk), dtype=np.int32)
    for m in range(w.M):
        topk_ids[m] = rng.choice(w.E, w.topk, replace=False, p=p)
    if w.mapping == "uniform_with_none":
        choices = np.concatenate([np.array([-1], np.int32), lora_ids])
        mapping = choices[rng.integers(0, len(choices), size=w.M)].astype(np.int32)
    elif w.mapping == "none10":
        none = rng.random(w.M) < 0.1
        slot = rng.integers(0, L, size=w.M)
        mapping = np.where(none, -1, slot).astype(np.int32)
    elif w.mapping == "uniform":
        mapping = lora_ids[rng.integers(0, nact, size=w.M)].astype(np.int32)
    else:
        raise ValueError(w.mapping)
    return lora_ids, topk_ids, mapping


def make_inputs(w: Workload, with_tensors: bool = True) -> Inputs:
    """Draw one batch.  with_tensors=False draws the routing only (align inputs)."""
    rng = np.random.default_rng(w.seed)
    lora_ids, topk_ids, mapping = draw_routing(w, rng)
    if not with_tensors:
        return Inputs(w, lora_ids, topk_ids, mapping, None, None, None, None)
    x = _normal_bf16((w.M, w.K), w.seed, _TAG_X, 0, 0, 1.0)
    a, b = _adapters(w, lora_ids, 0)
    y = _normal_bf16((w.M, w.topk, w.N), w.seed, _TAG_Y, 0, 0, 1.0)
    return Inputs(w, lora_ids, topk_ids, mapping, x, a, b, y)


@dataclasses.dataclass
class ExInputs:
    """Inputs of the general fused call: slices, rows per pair, weights, offset."""

    base: Inputs                        # routing; slice 0's adapters are base.lora_a / base.lora_b
    x: np.ndarray                       # uint16 [M, K], or [M*topk, K] when x_per_pair
    lora_a: list                        # per slice: uint16 [max_loras, E, r, K]
    lora_b: list                        # per slice: uint16 [max_loras, E, N, r]
    topk_weights: Optional[np.ndarray]  # float32 [M, topk] or None
    y_in: np.ndarray                    # uint16 [M, topk, ldy]
    x_per_pair: bool
    y_offset: int


def make_ex_inputs(w: Workload, num_slices: int = 1, x_per_pair: bool = False, routed_weights: bool = False,
                   y_offset: int = 0, ldy: Optional[int] = None) -> ExInputs:
    base = make_inputs(w)
    N = w.N
    if ldy is None:
        ldy = y_offset + num_slices * N
    x = base.x
    if x_per_pair:
        x = _normal_bf16((w.M * w.topk, w.K), w.seed, _TAG_X_PAIR, 0, 0, 1.0)
    lora_a, lora_b = [base.lora_a], [base.lora_b]
    for sl in range(1, num_slices):
        a, b = _adapters(w, base.lora_ids, sl)
        lora_a.append(a)
        lora_b.append(b)
    weights = None
    if routed_weights:
        g = np.random.default_rng([w.seed, _TAG_WEIGHTS]).standard_normal((w.M, w.topk), dtype=np.float32)
        g = np.exp(g - g.max(axis=1, keepdims=True))
        weights = (g / g.sum(axis=1, keepdims=True)).astype(np.float32)
    if ldy == N and y_offset == 0:
        y = base.y_in
    else:
        y = _normal_bf16((w.M, w.topk, ldy), w.seed, _TAG_Y_WIDE, 0, 0, 1.0)
    return ExInputs(base, x, lora_a, lora_b, weights, y, x_per_pair, y_offset)

"""Thin Python binding of libmoe_lora.so (include/moe_lora.h).

Argument marshalling only: each function checks tensor dtypes / devices,
passes raw pointers and sizes to the C ABI of the same name and raises
MoeLoraError on a non-zero status.  Every step of the computation runs in
the library's CUDA kernels; there is no other implementation to fall back to,
so a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MOE_LORA_OK = 0
ALIGN_AUTO, ALIGN_SMEM, ALIGN_GLOBAL, ALIGN_CLUSTER = 0, 1, 2, 3
PATH_AUTO, PATH_CUDA_CORE, PATH_TCGEN05, PATH_CUDA_CORE_CLUSTER, PATH_CUDA_CORE_STREAM = 0, 1, 2, 3, 4
DEVERR_EXPERT_ID, DEVERR_LORA_ID, DEVERR_CAPACITY, DEVERR_PAIR_ID, DEVERR_TIMEOUT = 1, 2, 4, 8, 16

_lib = None
_lock = threading.Lock()


class MoeLoraError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libmoe_lora.so (building it with nvcc if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libmoe_lora.so is missing: " + path)
            L = ctypes.CDLL(path)
            I, P, S = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            L.moe_lora_version.restype = I
            L.moe_lora_version.argtypes = []
            L.moe_lora_status_string.restype = ctypes.c_char_p
            L.moe_lora_status_string.argtypes = [I]
            L.moe_lora_max_num_tokens_padded.restype = I
            L.moe_lora_max_num_tokens_padded.argtypes = [I, I, I, I]
            L.moe_lora_max_num_m_blocks.restype = I
            L.moe_lora_max_num_m_blocks.argtypes = [I, I, I, I]
            L.moe_lora_align_resolve_variant.restype = I
            L.moe_lora_align_resolve_variant.argtypes = [I, I, I, I]
            L.moe_lora_align_workspace_bytes.restype = S
            L.moe_lora_align_workspace_bytes.argtypes = [I, I, I, I, I, I]
            L.moe_lora_align.restype = I
            L.moe_lora_align.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, I, I, P, S, I, P, P]
            L.moe_lora_align_static_workspace.restype = I
            L.moe_lora_align_static_workspace.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, I, I, P, P]
            L.moe_lora_fused_shrink_expand.restype = I
            L.moe_lora_fused_shrink_expand.argtypes = [P, P, P, P, P, P, P, P, P,
                                                       I, I, I, I, I, I, I, I, I, I, I, I, I, P, P]
            L.moe_lora_fused_shrink_expand_ex.restype = I
            L.moe_lora_fused_shrink_expand_ex.argtypes = [P, I, ctypes.POINTER(P), ctypes.POINTER(P), I, P, I, I, P,
                                                          P, P, P, P, P,
                                                          I, I, I, I, I, I, I, I, I, I, I, I, I, P, P]
            L.moe_align_block_size.restype = I
            L.moe_align_block_size.argtypes = [P, I, I, I, I, P, P, P, I, I, P, S, I, P, P]
            L.moe_lora_fused_shrink_expand_naive.restype = I
            L.moe_lora_fused_shrink_expand_naive.argtypes = [P, I, ctypes.POINTER(P), ctypes.POINTER(P), I, P, I, I,
                                                             P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P,
                                                             P]
            L.moe_lora_test_withheld_copy.restype = I
            L.moe_lora_test_withheld_copy.argtypes = [P, I, ctypes.POINTER(P), ctypes.POINTER(P), I, P, I, I, P, P,
                                                      P, P, P, I, I, I, I, I, I, I, I, I, ctypes.c_ulonglong, P, P]
            L.moe_lora_fused_plan.restype = I
            L.moe_lora_fused_plan.argtypes = [I] * 12 + [P]
            L.moe_lora_fused_resolve_path.restype = I
            L.moe_lora_fused_resolve_path.argtypes = [I] * 10
            L.moe_lora_fused_naive_resolve_path.restype = I
            L.moe_lora_fused_naive_resolve_path.argtypes = [I] * 9
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_lora_status_string(int(status)).decode()


def max_num_tokens_padded(M: int, topk: int, num_experts: int, block_size: int) -> int:
    return lib().moe_lora_max_num_tokens_padded(M, topk, num_experts, block_size)


def max_num_m_blocks(M: int, topk: int, num_experts: int, block_size: int) -> int:
    return lib().moe_lora_max_num_m_blocks(M, topk, num_experts, block_size)


def align_resolve_variant(M, topk, num_experts, variant=ALIGN_AUTO) -> int:
    """The align variant a call with these sizes runs (ALIGN_SMEM, ALIGN_GLOBAL
    or ALIGN_CLUSTER)."""
    v = lib().moe_lora_align_resolve_variant(M, topk, num_experts, variant)
    if v < 0:
        raise MoeLoraError(-v, "moe_lora_align_resolve_variant")
    return v


def align_workspace_bytes(M, topk, num_experts, num_active_loras, block_size, variant=ALIGN_AUTO) -> int:
    return lib().moe_lora_align_workspace_bytes(M, topk, num_experts, num_active_loras, block_size, variant)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status, what):
    if status != MOE_LORA_OK:
        raise MoeLoraError(status, what)


def moe_lora_align(topk_ids, token_lora_mapping, lora_ids, num_experts, max_loras, block_size,
                   sorted_token_ids, expert_ids, num_tokens_post_padded, adapter_enabled=None,
                   workspace=None, variant=ALIGN_AUTO, err_flag=None, stream=None):
    """moe_lora_align on device tensors; outputs are written in place."""
    M, topk = topk_ids.shape
    nact = lora_ids.numel()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().moe_lora_align(
        _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(token_lora_mapping, torch.int32, "token_lora_mapping"),
        _ptr(lora_ids, torch.int32, "lora_ids"), _ptr(adapter_enabled, torch.int32, "adapter_enabled"),
        M, topk, num_experts, max_loras, nact, block_size,
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(num_tokens_post_padded, torch.int32, "num_tokens_post_padded"),
        sorted_token_ids.shape[-1], expert_ids.shape[-1],
        _ptr(workspace, None, "workspace"), ws_bytes, variant,
        _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_lora_align")


STATIC_WORKSPACE_BYTES = 4 << 20


def moe_align_block_size(topk_ids, num_experts, block_size, sorted_token_ids, expert_ids, num_tokens_post_padded,
                         workspace=None, variant=ALIGN_AUTO, err_flag=None, stream=None):
    """The plain (non-LoRA) MoE align on device tensors: outputs are
    sorted_token_ids [cap], expert_ids [capb], num_tokens_post_padded [1]."""
    M, topk = topk_ids.shape
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().moe_align_block_size(
        _ptr(topk_ids, torch.int32, "topk_ids"), M, topk, num_experts, block_size,
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(num_tokens_post_padded, torch.int32, "num_tokens_post_padded"),
        sorted_token_ids.numel(), expert_ids.numel(), _ptr(workspace, name="workspace"), nbytes, variant,
        _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_align_block_size")


def moe_lora_align_static_workspace(topk_ids, token_lora_mapping, lora_ids, num_experts, max_loras, block_size,
                                    sorted_token_ids, expert_ids, num_tokens_post_padded, adapter_enabled=None,
                                    err_flag=None, stream=None):
    """moe_lora_align (global variant) on the library's built-in scratch buffer,
    for callers that cannot allocate device memory; see include/moe_lora.h."""
    M, topk = topk_ids.shape
    st = lib().moe_lora_align_static_workspace(
        _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(token_lora_mapping, torch.int32, "token_lora_mapping"),
        _ptr(lora_ids, torch.int32, "lora_ids"), _ptr(adapter_enabled, torch.int32, "adapter_enabled"),
        M, topk, num_experts, max_loras, lora_ids.numel(), block_size,
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(num_tokens_post_padded, torch.int32, "num_tokens_post_padded"),
        sorted_token_ids.shape[-1], expert_ids.shape[-1],
        _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_lora_align_static_workspace")


def moe_lora_fused_shrink_expand(x, lora_a, lora_b, y, sorted_token_ids, expert_ids, num_tokens_post_padded,
                                 lora_ids, topk, block_size, add_inputs=True, adapter_enabled=None,
                                 path=PATH_AUTO, err_flag=None, stream=None):
    """moe_lora_fused_shrink_expand on device tensors; y is updated in place."""
    M, K = x.shape
    L, E, r, K2 = lora_a.shape
    N = lora_b.shape[2]
    if K2 != K or tuple(lora_b.shape) != (L, E, N, r) or y.numel() != M * topk * N:
        raise ValueError("inconsistent shapes")
    bf = torch.bfloat16
    st = lib().moe_lora_fused_shrink_expand(
        _ptr(x, bf, "x"), _ptr(lora_a, bf, "lora_a"), _ptr(lora_b, bf, "lora_b"), _ptr(y, bf, "y"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(num_tokens_post_padded, torch.int32, "num_tokens_post_padded"),
        _ptr(lora_ids, torch.int32, "lora_ids"), _ptr(adapter_enabled, torch.int32, "adapter_enabled"),
        M, topk, E, K, N, r, L, lora_ids.numel(), block_size,
        sorted_token_ids.shape[-1], expert_ids.shape[-1], int(bool(add_inputs)), path,
        _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_lora_fused_shrink_expand")


def fused_naive_resolve_path(M, topk, num_experts, K, N, rank, num_active_loras, num_slices=1, path=PATH_AUTO) -> int:
    """The kernel a naive-assignment call with these sizes runs
    (PATH_CUDA_CORE_CLUSTER or PATH_CUDA_CORE_STREAM)."""
    v = lib().moe_lora_fused_naive_resolve_path(M, topk, num_experts, K, N, rank, num_active_loras, num_slices, path)
    if v < 0:
        raise MoeLoraError(-v, "moe_lora_fused_naive_resolve_path")
    return v


def fused_resolve_path(M, topk, num_experts, K, N, rank, num_active_loras, block_size, num_slices=1,
                       path=PATH_AUTO) -> int:
    """The kernel a fused call with these sizes runs (PATH_TCGEN05,
    PATH_CUDA_CORE_CLUSTER or PATH_CUDA_CORE_STREAM)."""
    v = lib().moe_lora_fused_resolve_path(M, topk, num_experts, K, N, rank, num_active_loras, block_size,
                                          num_slices, path)
    if v < 0:
        raise MoeLoraError(-v, "moe_lora_fused_resolve_path")
    return v


PLAN_FIELDS = ("kernel", "grid", "threads", "smem_bytes", "s_sh", "lag", "s_ex", "t_bufs", "tmem_cols", "cluster",
               "pairs_per_group")


def fused_plan(M, topk, num_experts, K, N, rank, num_active_loras, block_size, num_slices=1, path=PATH_AUTO,
               sm_count=152, max_smem_per_block=232448) -> dict:
    """The launch plan a plain fused call would use on a device with these
    properties (host arithmetic only)."""
    out = (ctypes.c_int32 * len(PLAN_FIELDS))()
    st = lib().moe_lora_fused_plan(M, topk, num_experts, K, N, rank, num_active_loras, block_size, num_slices, path,
                                   sm_count, max_smem_per_block, ctypes.cast(out, ctypes.c_void_p))
    _check(st, "moe_lora_fused_plan")
    return dict(zip(PLAN_FIELDS, list(out)))


def moe_lora_fused_shrink_expand_ex(x, lora_a, lora_b, y, sorted_token_ids, expert_ids, num_tokens_post_padded,
                                    lora_ids, topk, block_size, add_inputs=True, adapter_enabled=None,
                                    topk_weights=None, x_per_pair=False, y_offset=0,
                                    path=PATH_AUTO, err_flag=None, stream=None):
    """moe_lora_fused_shrink_expand_ex on device tensors; y is updated in place.

    lora_a / lora_b: a tensor (one slice) or a list of per-slice tensors
    ([L, E, r, K] / [L, E, N, r]).  x: [M, K], or [M*topk, K] with x_per_pair.
    y: [M, topk, ldy]; slice s writes columns y_offset + s*N .. + N.
    topk_weights: float32 [M, topk] or None."""
    if isinstance(lora_a, torch.Tensor):
        lora_a, lora_b = [lora_a], [lora_b]
    S = len(lora_a)
    if S < 1 or len(lora_b) != S:
        raise ValueError("lora_a and lora_b need the same number of slices")
    L, E, r, K = lora_a[0].shape
    N = lora_b[0].shape[2]
    for a, b in zip(lora_a, lora_b):
        if tuple(a.shape) != (L, E, r, K) or tuple(b.shape) != (L, E, N, r):
            raise ValueError("inconsistent slice shapes")
    if y.dim() != 3:
        raise ValueError("y must be [M, topk, ldy]")
    M = y.shape[0]
    ldy = y.shape[2]
    if y.shape[1] != topk or tuple(x.shape) != ((M * topk if x_per_pair else M), K):
        raise ValueError("inconsistent shapes")
    if topk_weights is not None and topk_weights.numel() != M * topk:
        raise ValueError("topk_weights must be [M, topk]")
    bf = torch.bfloat16
    a_ptrs = (ctypes.c_void_p * S)(*[_ptr(a, bf, "lora_a") for a in lora_a])
    b_ptrs = (ctypes.c_void_p * S)(*[_ptr(b, bf, "lora_b") for b in lora_b])
    st = lib().moe_lora_fused_shrink_expand_ex(
        _ptr(x, bf, "x"), int(bool(x_per_pair)), a_ptrs, b_ptrs, S, _ptr(y, bf, "y"), ldy, y_offset,
        _ptr(topk_weights, torch.float32, "topk_weights"),
        _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"), _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(num_tokens_post_padded, torch.int32, "num_tokens_post_padded"),
        _ptr(lora_ids, torch.int32, "lora_ids"), _ptr(adapter_enabled, torch.int32, "adapter_enabled"),
        M, topk, E, K, N, r, L, lora_ids.numel(), block_size,
        sorted_token_ids.shape[-1], expert_ids.shape[-1], int(bool(add_inputs)), path,
        _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_lora_fused_shrink_expand_ex")


def moe_lora_fused_shrink_expand_naive(x, lora_a, lora_b, y, topk_ids, token_lora_mapping, lora_ids, max_loras,
                                       add_inputs=True, adapter_enabled=None, topk_weights=None, x_per_pair=False,
                                       y_offset=0, path=PATH_AUTO, err_flag=None, stream=None):
    """moe_lora_fused_shrink_expand_naive (no align: one work item per pair) on
    device tensors; y [M, topk, ldy] is updated in place.  lora_a / lora_b: a
    tensor or a list of per-slice tensors.  path: PATH_AUTO, PATH_CUDA_CORE,
    PATH_CUDA_CORE_CLUSTER or PATH_CUDA_CORE_STREAM."""
    if isinstance(lora_a, torch.Tensor):
        lora_a, lora_b = [lora_a], [lora_b]
    S = len(lora_a)
    if S < 1 or len(lora_b) != S:
        raise ValueError("lora_a and lora_b need the same number of slices")
    L, E, r, K = lora_a[0].shape
    N = lora_b[0].shape[2]
    for a, b in zip(lora_a, lora_b):
        if tuple(a.shape) != (L, E, r, K) or tuple(b.shape) != (L, E, N, r):
            raise ValueError("inconsistent slice shapes")
    M, topk = topk_ids.shape
    if y.dim() != 3 or y.shape[0] != M or y.shape[1] != topk:
        raise ValueError("y must be [M, topk, ldy]")
    if tuple(x.shape) != ((M * topk if x_per_pair else M), K) or token_lora_mapping.numel() != M:
        raise ValueError("inconsistent shapes")
    if topk_weights is not None and topk_weights.numel() != M * topk:
        raise ValueError("topk_weights must be [M, topk]")
    if max_loras != L:
        raise ValueError("max_loras must equal the adapters' first dimension")
    bf = torch.bfloat16
    a_ptrs = (ctypes.c_void_p * S)(*[_ptr(a, bf, "lora_a") for a in lora_a])
    b_ptrs = (ctypes.c_void_p * S)(*[_ptr(b, bf, "lora_b") for b in lora_b])
    st = lib().moe_lora_fused_shrink_expand_naive(
        _ptr(x, bf, "x"), int(bool(x_per_pair)), a_ptrs, b_ptrs, S, _ptr(y, bf, "y"), y.shape[2], y_offset,
        _ptr(topk_weights, torch.float32, "topk_weights"), _ptr(topk_ids, torch.int32, "topk_ids"),
        _ptr(token_lora_mapping, torch.int32, "token_lora_mapping"), _ptr(lora_ids, torch.int32, "lora_ids"),
        _ptr(adapter_enabled, torch.int32, "adapter_enabled"), M, topk, E, K, N, r, L, lora_ids.numel(),
        int(bool(add_inputs)), int(path), _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_lora_fused_shrink_expand_naive")


def moe_lora_test_withheld_copy(x, lora_a, lora_b, y, topk_ids, token_lora_mapping, lora_ids, max_loras,
                                wait_limit_ns, add_inputs=True, err_flag=None, stream=None):
    """moe_lora_test_withheld_copy (a test of the bounded waits): the naive call
    with every CTA's B-slice copy withheld and its wait limited to
    wait_limit_ns; y [M, topk, N], one slice."""
    if isinstance(lora_a, torch.Tensor):
        lora_a, lora_b = [lora_a], [lora_b]
    S = len(lora_a)
    L, E, r, K = lora_a[0].shape
    N = lora_b[0].shape[2]
    M, topk = topk_ids.shape
    bf = torch.bfloat16
    a_ptrs = (ctypes.c_void_p * S)(*[_ptr(a, bf, "lora_a") for a in lora_a])
    b_ptrs = (ctypes.c_void_p * S)(*[_ptr(b, bf, "lora_b") for b in lora_b])
    st = lib().moe_lora_test_withheld_copy(
        _ptr(x, bf, "x"), 0, a_ptrs, b_ptrs, S, _ptr(y, bf, "y"), y.shape[2], 0, None,
        _ptr(topk_ids, torch.int32, "topk_ids"), _ptr(token_lora_mapping, torch.int32, "token_lora_mapping"),
        _ptr(lora_ids, torch.int32, "lora_ids"), None, M, topk, E, K, N, r, L, lora_ids.numel(),
        int(bool(add_inputs)), int(wait_limit_ns), _ptr(err_flag, torch.int32, "err_flag"), _stream(stream))
    _check(st, "moe_lora_test_withheld_copy")


class AlignBuffers:
    """Device output buffers (and workspace) for one align configuration."""

    def __init__(self, M, topk, num_experts, max_loras, num_active_loras, block_size, device="cuda",
                 variant=ALIGN_AUTO):
        cap = max_num_tokens_padded(M, topk, num_experts, block_size)
        capb = max_num_m_blocks(M, topk, num_experts, block_size)
        self.sorted_token_ids = torch.empty((max_loras, cap), dtype=torch.int32, device=device)
        self.expert_ids = torch.empty((max_loras, capb), dtype=torch.int32, device=device)
        self.num_tokens_post_padded = torch.empty((max_loras,), dtype=torch.int32, device=device)
        nbytes = align_workspace_bytes(M, topk, num_experts, num_active_loras, block_size, variant)
        self.workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=device) if nbytes else None

"""ctypes wrapper of the C oracle (moe_lora_oracle.c).  Test infrastructure only.

Arrays are numpy; bf16 tensors are uint16 arrays of raw bit patterns.  The
arithmetic lives in the C file; this wrapper only marshals arguments.
"""
import ctypes
import threading

import numpy as np

from . import build as _build

STATUS_BAD_EXPERT_ID = 1
STATUS_BAD_LORA_ID = 2
STATUS_CAPACITY = 4

_lib = None
_lock = threading.Lock()

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_build.build())
            I = ctypes.c_int
            opt_i32 = ctypes.c_void_p
            lib.oracle_moe_lora_align.restype = I
            lib.oracle_moe_lora_align.argtypes = [
                _i32p, _i32p, _i32p, opt_i32, I, I, I, I, I, I,
                _i32p, _i32p, _i32p, I, I]
            lib.oracle_moe_lora_fused.restype = I
            lib.oracle_moe_lora_fused.argtypes = [
                _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, opt_i32,
                I, I, I, I, I, I, I, I, I, _f64p]
            lib.oracle_moe_lora_fused_sampled.restype = I
            lib.oracle_moe_lora_fused_sampled.argtypes = [
                _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, opt_i32,
                I, I, I, I, I, I, I, I, I, _i32p, I, _i32p, I, _f64p]
            lib.oracle_moe_lora_fused_ex.restype = I
            lib.oracle_moe_lora_fused_ex.argtypes = [
                _u16p, I, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), I,
                _u16p, I, I, ctypes.c_void_p, _i32p, _i32p, _i32p, opt_i32,
                I, I, I, I, I, I, I, I, I, ctypes.c_void_p, I, _f64p]
            _lib = lib
    return _lib


def capacity_tokens(M, topk, E, block_size):
    """Length of one LoRA row of sorted_token_ids: every pair, plus up to
    block_size-1 padding slots per expert."""
    return M * topk + E * (block_size - 1)


def capacity_blocks(M, topk, E, block_size):
    return -(-capacity_tokens(M, topk, E, block_size) // block_size)


def _c32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _opt(a):
    if a is None:
        return None, None
    a = _c32(a)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def align(topk_ids, token_lora_mapping, lora_ids, num_experts, max_loras, block_size,
          adapter_enabled=None, max_num_tokens_padded=None, max_num_m_blocks=None,
          fill=-7):
    """Run the align oracle.  Undefined output entries keep `fill`.

    Returns (status, sorted_token_ids [L, cap], expert_ids [L, capb], ntpp [L])."""
    topk_ids = _c32(topk_ids)
    M, topk = topk_ids.shape
    lora_ids = _c32(lora_ids)
    mapping = _c32(token_lora_mapping)
    cap = max_num_tokens_padded or capacity_tokens(M, topk, num_experts, block_size)
    capb = max_num_m_blocks or capacity_blocks(M, topk, num_experts, block_size)
    sorted_ids = np.full((max_loras, cap), fill, np.int32)
    expert_ids = np.full((max_loras, capb), fill, np.int32)
    ntpp = np.full((max_loras,), fill, np.int32)
    keep, en = _opt(adapter_enabled)
    st = _load().oracle_moe_lora_align(
        topk_ids.reshape(-1), mapping, lora_ids, en, M, topk, num_experts, max_loras,
        len(lora_ids), block_size, sorted_ids.reshape(-1), expert_ids.reshape(-1), ntpp,
        cap, capb)
    del keep
    return st, sorted_ids, expert_ids, ntpp


def align_plain(topk_ids, num_experts, block_size, max_num_tokens_padded=None, max_num_m_blocks=None,
                fill=-7):
    """The plain (non-LoRA) MoE align: the single-slot case of align(), every
    token owned by slot 0.

    Returns (status, sorted_token_ids [cap], expert_ids [capb], ntpp [1])."""
    topk_ids = _c32(topk_ids)
    M = topk_ids.shape[0]
    st, s, e, n = align(topk_ids, np.zeros(M, np.int32), np.array([0], np.int32), num_experts, 1, block_size,
                        max_num_tokens_padded=max_num_tokens_padded, max_num_m_blocks=max_num_m_blocks, fill=fill)
    return st, s[0], e[0], n


def fused(x, lora_a, lora_b, y_in, topk_ids, token_lora_mapping, lora_ids,
          add_inputs=True, adapter_enabled=None):
    """Run the fused oracle over every pair.  Returns float64 [M, topk, N]."""
    x = np.ascontiguousarray(x, np.uint16)
    lora_a = np.ascontiguousarray(lora_a, np.uint16)
    lora_b = np.ascontiguousarray(lora_b, np.uint16)
    y_in = np.ascontiguousarray(y_in, np.uint16)
    topk_ids = _c32(topk_ids)
    M, K = x.shape
    L, E, r, K2 = lora_a.shape
    N = lora_b.shape[2]
    topk = topk_ids.shape[1]
    assert K2 == K and lora_b.shape == (L, E, N, r) and y_in.shape == (M, topk, N)
    lora_ids = _c32(lora_ids)
    ref = np.empty((M, topk, N), np.float64)
    keep, en = _opt(adapter_enabled)
    st = _load().oracle_moe_lora_fused(
        x.reshape(-1), lora_a.reshape(-1), lora_b.reshape(-1), y_in.reshape(-1),
        topk_ids.reshape(-1), _c32(token_lora_mapping), lora_ids, en,
        M, topk, E, K, N, r, L, len(lora_ids), int(bool(add_inputs)), ref.reshape(-1))
    del keep
    assert st == 0
    return ref


def fused_sampled(x, lora_a, lora_b, y_in, topk_ids, token_lora_mapping, lora_ids,
                  pairs, columns, add_inputs=True, adapter_enabled=None):
    """The fused definition at sampled pairs (flat index m*topk+k) and columns.

    Returns float64 [len(pairs), len(columns)]."""
    x = np.ascontiguousarray(x, np.uint16)
    lora_a = np.ascontiguousarray(lora_a, np.uint16)
    lora_b = np.ascontiguousarray(lora_b, np.uint16)
    y_in = np.ascontiguousarray(y_in, np.uint16)
    topk_ids = _c32(topk_ids)
    M, K = x.shape
    L, E, r, _ = lora_a.shape
    N = lora_b.shape[2]
    topk = topk_ids.shape[1]
    pairs = _c32(pairs)
    columns = _c32(columns)
    out = np.empty((len(pairs), len(columns)), np.float64)
    keep, en = _opt(adapter_enabled)
    st = _load().oracle_moe_lora_fused_sampled(
        x.reshape(-1), lora_a.reshape(-1), lora_b.reshape(-1), y_in.reshape(-1),
        topk_ids.reshape(-1), _c32(token_lora_mapping), _c32(lora_ids), en,
        M, topk, E, K, N, r, L, len(lora_ids), int(bool(add_inputs)),
        pairs, len(pairs), columns, len(columns), out.reshape(-1))
    del keep
    assert st == 0
    return out


def fused_ex(x, lora_a, lora_b, y_in, topk_ids, token_lora_mapping, lora_ids,
             add_inputs=True, adapter_enabled=None, topk_weights=None,
             x_per_pair=False, y_offset=0, pairs=None):
    """The fused definition with its options: router weights, input rows per
    pair, several adapter slices and an output column offset.

    lora_a / lora_b: one array per slice ([L, E, r, K] / [L, E, N, r]), or a
    single array for one slice.  x: [M*topk, K] if x_per_pair else [M, K].
    y_in: [M, topk, ldy].  topk_weights: float32 [M, topk] or None.
    pairs: flat pair indices to evaluate (None: every pair).

    Returns float64 [M, topk, ldy], or [len(pairs), ldy] when pairs is given."""
    if not isinstance(lora_a, (list, tuple)):
        lora_a, lora_b = [lora_a], [lora_b]
    lora_a = [np.ascontiguousarray(a, np.uint16) for a in lora_a]
    lora_b = [np.ascontiguousarray(b, np.uint16) for b in lora_b]
    S = len(lora_a)
    assert S >= 1 and len(lora_b) == S
    x = np.ascontiguousarray(x, np.uint16)
    y_in = np.ascontiguousarray(y_in, np.uint16)
    topk_ids = _c32(topk_ids)
    M, topk = topk_ids.shape
    L, E, r, K = lora_a[0].shape
    N = lora_b[0].shape[2]
    for a, b in zip(lora_a, lora_b):
        assert a.shape == (L, E, r, K) and b.shape == (L, E, N, r)
    assert x.shape == ((M * topk if x_per_pair else M), K)
    ldy = y_in.shape[-1]
    assert y_in.shape == (M, topk, ldy) and 0 <= y_offset and y_offset + S * N <= ldy
    a_ptrs = (ctypes.c_void_p * S)(*[a.ctypes.data for a in lora_a])
    b_ptrs = (ctypes.c_void_p * S)(*[b.ctypes.data for b in lora_b])
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, np.float32)
    if w is not None:
        assert w.shape == (M, topk)
    sel = None if pairs is None else _c32(pairs)
    out = np.empty(((M, topk, ldy) if sel is None else (len(sel), ldy)), np.float64)
    keep, en = _opt(adapter_enabled)
    st = _load().oracle_moe_lora_fused_ex(
        x.reshape(-1), int(bool(x_per_pair)), a_ptrs, b_ptrs, S, y_in.reshape(-1), ldy, y_offset,
        None if w is None else w.ctypes.data, topk_ids.reshape(-1), _c32(token_lora_mapping),
        _c32(lora_ids), en, M, topk, E, K, N, r, L, len(lora_ids), int(bool(add_inputs)),
        None if sel is None else sel.ctypes.data, 0 if sel is None else len(sel), out.reshape(-1))
    del keep
    assert st == 0
    return out

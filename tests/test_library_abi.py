"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/moe_lora.h declares, sizes its buffers as documented
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from lora_moe_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_lora.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_lora_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_two_stages():
    names = declared_functions()
    assert "moe_lora_align" in names and "moe_lora_fused_shrink_expand" in names


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    # exported with C linkage (no C++ mangling)
    out = os.popen("nm -D --defined-only %s" % B.library_path()).read()
    for name in declared_functions():
        assert re.search(r"\bT %s$" % name, out, flags=re.M), name


def test_capacities():
    assert B.max_num_tokens_padded(16, 2, 8, 16) == 16 * 2 + 8 * 15
    assert B.max_num_m_blocks(16, 2, 8, 16) == -(-(16 * 2 + 8 * 15) // 16)
    assert B.max_num_tokens_padded(4096, 8, 256, 64) == 48896
    assert B.max_num_m_blocks(4096, 8, 256, 64) == 764
    assert B.max_num_tokens_padded(-1, 2, 8, 16) == -1


def test_workspace_sizes():
    # the shared-memory variant needs none
    assert B.align_workspace_bytes(16, 2, 8, 2, 16, B.ALIGN_SMEM) == 0
    # the global variant: per slot a warps x E table plus E offsets
    n = B.align_workspace_bytes(4096, 8, 256, 8, 64, B.ALIGN_GLOBAL)
    assert n > 0 and n % (8 * 4) == 0
    assert B.align_workspace_bytes(4096, 8, 256, 4, 64, B.ALIGN_GLOBAL) * 2 == n
    assert B.align_workspace_bytes(4096, 8, 256, 8, 64, B.ALIGN_AUTO) == n   # AUTO picks global at E=256


def test_version():
    assert B.lib().moe_lora_version() >= 100


def test_status_strings():
    for st in range(7):
        assert B.status_string(st)
    assert B.status_string(99) == "unknown status"


def _align(**kw):
    args = dict(topk_ids=None, mapping=None, lora_ids=None, enabled=None, M=16, topk=2, E=8, L=2, nact=2, bs=16,
                sorted=None, experts=None, ntpp=None, cap=16 * 2 + 8 * 15, capb=10, ws=None, ws_bytes=0,
                variant=0, err=None, stream=None)
    args.update(kw)
    return B.lib().moe_lora_align(*args.values())


def _fused(**kw):
    args = dict(x=None, a=None, b=None, y=None, sorted=None, experts=None, ntpp=None, lora_ids=None,
                enabled=None, M=16, topk=2, E=8, K=256, N=512, r=8, L=2, nact=2, bs=16, cap=152, capb=10,
                add=1, path=0, err=None, stream=None)
    args.update(kw)
    return B.lib().moe_lora_fused_shrink_expand(*args.values())


def test_align_argument_errors():
    assert _align(E=1025) == 2                    # num_experts > 1024
    assert _align(topk=9) == 2                    # topk > num_experts
    assert _align(bs=8) == 2                      # block size not in {16, 32, 64, 128}
    assert _align(nact=3) == 1                    # more active slots than max_loras
    assert _align(cap=100) == 1                   # capacity too small
    assert _align(M=-1) == 1
    assert _align(variant=7) == 1
    assert _align(nact=0) == 0                    # zero grid: nothing to do
    assert _align() == 1                          # NULL buffers


def test_fused_argument_errors():
    assert _fused(r=132) == 2                     # rank > 128
    assert _fused(r=6) == 2                       # rank % 4 != 0
    assert _fused(K=260) == 3                     # rows not 16-byte multiples
    assert _fused(N=100) == 3
    assert _fused(path=2, r=12) == 2              # tensor-core path needs rank % 8 == 0
    assert _fused(path=5) == 1
    assert _fused(nact=0) == 0                    # zero grid
    assert _fused(M=0) == 0                       # empty batch
    assert _fused() == 1                          # NULL buffers
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    p1 = ((p + 15) & ~15) + 2                     # misaligned on purpose (host memory, never dereferenced)
    assert _fused(x=p1, a=p1, b=p1, y=p1, sorted=p1, experts=p1, ntpp=p1, lora_ids=p1) == 3

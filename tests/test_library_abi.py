"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/moe_lora.h declares, sizes its buffers as documented
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from lora_moe_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_lora.h")


def _header_code():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return "\n".join(l for l in text.splitlines() if not l.lstrip().startswith("#"))


def declared_functions():
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", _header_code())))


def test_header_declares_the_two_stages():
    names = declared_functions()
    assert "moe_lora_align" in names and "moe_lora_fused_shrink_expand" in names
    assert "moe_align_block_size" in names


def test_every_header_declaration_is_parsed():
    """One name per function declaration: a declaration whose name the parser
    missed would escape the export check below."""
    code = _header_code().replace('extern "C" {', "").replace("}", "};")
    decls = [d for d in code.split(";") if "(" in d]
    assert len(decls) == len(declared_functions()), decls


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
    assert B.align_workspace_bytes(4096, 8, 256, 8, 64, B.ALIGN_AUTO) == 0   # AUTO picks the cluster variant at E=256
    assert B.align_workspace_bytes(4096, 8, 256, 8, 64, B.ALIGN_CLUSTER) == 0


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


def test_static_workspace_checks_arguments_before_size():
    """moe_lora_align_static_workspace reports moe_lora_align's argument errors
    first, then MOE_LORA_ERR_WORKSPACE for problems beyond its built-in buffer,
    both before touching a device (the dummy pointers are never read)."""
    lib = B.lib()
    fn = lib.moe_lora_align_static_workspace
    M, topk, E, bs = 65536, 8, 1024, 16          # workspace far beyond 4 MiB
    cap, capb = B.max_num_tokens_padded(M, topk, E, bs), B.max_num_m_blocks(M, topk, E, bs)
    d = ctypes.c_void_p(16)
    # more active slots than max_loras: an argument error, not a size error
    assert fn(d, d, d, None, M, topk, E, 8, 9, bs, d, d, d, cap, capb, None, None) == 1
    # capacity smaller than required
    assert fn(d, d, d, None, M, topk, E, 8, 8, bs, d, d, d, cap - 1, capb, None, None) == 1
    # NULL outputs
    assert fn(d, d, d, None, M, topk, E, 8, 8, bs, None, d, d, cap, capb, None, None) == 1
    # valid arguments, workspace beyond the built-in buffer
    assert B.align_workspace_bytes(M, topk, E, 8, bs, B.ALIGN_GLOBAL) > 4 << 20
    assert fn(d, d, d, None, M, topk, E, 8, 8, bs, d, d, d, cap, capb, None, None) == 4


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


def _fused_ex(slices=1, a_ptrs=None, b_ptrs=None, **kw):
    P = ctypes.c_void_p
    if a_ptrs is None:
        a_ptrs = (P * max(slices, 1))()
    if b_ptrs is None:
        b_ptrs = (P * max(slices, 1))()
    args = dict(x=None, x_per_pair=0, a=a_ptrs, b=b_ptrs, S=slices, y=None, ldy=512, y_off=0, w=None,
                sorted=None, experts=None, ntpp=None, lora_ids=None, enabled=None, M=16, topk=2, E=8, K=256,
                N=512, r=8, L=2, nact=2, bs=16, cap=152, capb=10, add=1, path=0, err=None, stream=None)
    args.update(kw)
    return B.lib().moe_lora_fused_shrink_expand_ex(*args.values())


def test_fused_ex_argument_errors():
    assert _fused_ex(slices=0) == 1                   # no slice
    assert _fused_ex(slices=5, ldy=5 * 512) == 1      # more than MOE_LORA_MAX_SLICES
    assert _fused_ex(slices=2, ldy=512) == 1          # slices do not fit the row
    assert _fused_ex(y_off=8, ldy=512) == 1           # offset pushes the slice past the row
    assert _fused_ex(y_off=-8, ldy=1024) == 1
    assert _fused_ex(ldy=1028, y_off=0) == 3          # row stride not a 16-byte multiple
    assert _fused_ex(ldy=1024, y_off=4) == 3          # offset not a 16-byte multiple
    assert _fused_ex(a=None) == 1                     # no slice pointer arrays
    assert _fused_ex(r=12, path=4) == 2               # streaming kernel needs rank % 8 == 0
    assert _fused_ex(slices=2, ldy=1024, nact=0) == 0 # zero grid
    assert _fused_ex(slices=3, ldy=3 * 512, M=0) == 0 # empty batch
    assert _fused_ex(slices=2, ldy=1024) == 1         # NULL buffers
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    p0 = (p + 15) & ~15
    P = ctypes.c_void_p
    ok = dict(x=p0, y=p0, sorted=p0, experts=p0, ntpp=p0, lora_ids=p0)
    # misaligned slice pointer or weights (host memory, never dereferenced)
    assert _fused_ex(slices=2, ldy=1024, a_ptrs=(P * 2)(p0, p0 + 2), b_ptrs=(P * 2)(p0, p0), **ok) == 3
    assert _fused_ex(slices=1, w=p0 + 2, a_ptrs=(P * 1)(p0), b_ptrs=(P * 1)(p0), **ok) == 3
    assert _fused_ex(slices=2, ldy=1024, a_ptrs=(P * 2)(p0, None), b_ptrs=(P * 2)(p0, p0), **ok) == 1


def test_fused_resolve_path():
    R = B.lib().moe_lora_fused_resolve_path
    # decode-sized, small adapters -> cluster kernel; many pairs -> tensor cores
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16, 1, 0) == 3
    assert R(8192, 2, 8, 4096, 28672, 16, 4, 64, 1, 0) == 2
    # few pairs but large adapters (block bound x (K + N) x r x 2 bytes > 48 MB) -> cluster
    # streaming kernel, or tensor cores for a rank it does not take
    assert R(64, 4, 128, 2880, 2880, 64, 6, 16, 1, 0) == 4
    assert R(64, 4, 128, 2880, 2880, 72, 6, 16, 1, 0) == 2
    # rank % 8 != 0 keeps the CUDA cores
    assert R(8192, 2, 8, 4096, 28672, 12, 4, 64, 1, 0) == 3
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16, 1, 1) == 3   # CUDA_CORE -> cluster
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16, 1, 4) == 4
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16, 1, 2) == 2
    assert R(16, 8, 128, 2048, 1536, 12, 2, 16, 1, 2) == -2  # tensor cores need rank % 8 == 0
    assert R(16, 8, 128, 2048, 1536, 24, 2, 16, 1, 4) == -2  # streaming: ranks 8, 16, 32, 64, 128
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16, 5, 0) == -1  # too many slices
    assert R(16, 8, 128, 2048, 1536, 16, 2, 16, 1, 9) == -1


def test_naive_resolve_path():
    """The naive assignment's kernel: the streaming kernel when the pairs'
    adapters exceed 48 MB (gpt-oss-shaped w2 decode), else the
    one-cluster-per-pair kernel (Qwen3-shaped decode); forced paths kept."""
    R = B.lib().moe_lora_fused_naive_resolve_path
    # (M, topk, E, K, N, rank, num_active_loras, num_slices, path)
    assert R(64, 4, 128, 2880, 2880, 64, 6, 1, 0) == 4
    assert R(64, 4, 128, 2880, 2880, 64, 129, 1, 0) == 3      # more slots than the streaming list indexes
    assert R(16, 8, 128, 2048, 1536, 16, 2, 1, 0) == 3
    assert R(16, 8, 128, 2048, 1536, 16, 2, 1, 1) == 3        # CUDA_CORE -> cluster
    assert R(16, 8, 128, 2048, 1536, 16, 2, 1, 4) == 4
    assert R(16, 8, 128, 2048, 1536, 24, 2, 1, 4) == -2       # streaming: ranks 8, 16, 32, 64, 128
    assert R(16, 8, 128, 2048, 1536, 16, 2, 1, 2) == -1       # no tensor-core naive path
    assert R(16, 8, 128, 2048, 1536, 16, 2, 5, 0) == -1       # too many slices
    assert B.fused_naive_resolve_path(64, 4, 128, 2880, 2880, 64, 6) == B.PATH_CUDA_CORE_STREAM


def test_align_resolve_variant():
    R = B.lib().moe_lora_align_resolve_variant
    assert R(16, 8, 128, 0) in (1, 2, 3)          # AUTO resolves to a concrete variant
    for v in (1, 2, 3):
        assert R(16, 8, 128, v) == v               # forced variants are kept
    assert R(16, 8, 1025, 0) == -2                 # num_experts > 1024
    assert R(16, 8, 128, 4) == -1                  # no such variant
    assert R(-1, 8, 128, 0) == -1


def test_plain_align_argument_errors():
    f = B.lib().moe_align_block_size
    # (topk_ids, M, topk, E, bs, sorted, experts, ntpp, cap, capb, ws, ws_bytes, variant, err, stream)
    assert f(None, 16, 2, 1025, 16, None, None, None, 10000, 1000, None, 0, 0, None, None) == 2
    assert f(None, 16, 2, 8, 8, None, None, None, 10000, 1000, None, 0, 0, None, None) == 2
    assert f(None, 16, 2, 8, 16, None, None, None, 10, 1, None, 0, 0, None, None) == 1     # capacity too small
    assert f(None, 16, 2, 8, 16, None, None, None, 152, 10, None, 0, 7, None, None) == 1   # bad variant
    assert f(None, 16, 2, 8, 16, None, None, None, 152, 10, None, 0, 0, None, None) == 1   # NULL buffers
    assert B.align_workspace_bytes(4096, 8, 256, 1, 64, B.ALIGN_GLOBAL) > 0


def test_fused_naive_argument_errors():
    P = ctypes.c_void_p

    def naive(slices=1, **kw):
        args = dict(x=None, x_per_pair=0, a=(P * max(slices, 1))(), b=(P * max(slices, 1))(), S=slices, y=None,
                    ldy=512, y_off=0, w=None, topk_ids=None, mapping=None, lora_ids=None, enabled=None, M=16,
                    topk=2, E=8, K=256, N=512, r=8, L=2, nact=2, add=1, path=0, err=None, stream=None)
        args.update(kw)
        return B.lib().moe_lora_fused_shrink_expand_naive(*args.values())

    assert naive(E=1025) == 2
    assert naive(topk=9) == 2
    assert naive(nact=3) == 1
    assert naive(r=132) == 2
    assert naive(K=260) == 3
    assert naive(slices=0) == 1
    assert naive(nact=0) == 0          # zero grid
    assert naive(M=0) == 0
    assert naive() == 1                # NULL buffers
    assert naive(path=2) == 1          # the tensor-core kernel has no naive assignment
    assert naive(path=9) == 1
    assert naive(path=4, r=12) == 2    # the cluster streaming kernel takes ranks 8, 16, 32, 64, 128
    assert naive(path=4, r=24) == 2


def test_plain_c_consumer(tmp_path):
    """The header compiles as C11 under -Wall -Wextra -pedantic, and a C
    program links against the library and calls its host-only functions."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib_dir = os.path.dirname(B.library_path())
    src = tmp_path / "consumer.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "moe_lora.h"
int main(void) {
  int32_t plan[11];
  if (moe_lora_version() <= 0) return 1;
  if (moe_lora_max_num_tokens_padded(16, 8, 128, 16) != 16 * 8 + 128 * 15) return 2;
  if (moe_lora_max_num_m_blocks(16, 8, 128, 16) != (16 * 8 + 128 * 15 + 15) / 16) return 3;
  if (strlen(moe_lora_status_string(MOE_LORA_ERR_INVALID_ARG)) == 0) return 4;
  if (moe_lora_fused_resolve_path(16, 8, 128, 2048, 1536, 16, 2, 16, 1, MOE_LORA_PATH_AUTO)
      != MOE_LORA_PATH_CUDA_CORE_CLUSTER) return 5;
  if (moe_lora_fused_plan(8192, 2, 8, 4096, 28672, 16, 4, 64, 1, MOE_LORA_PATH_AUTO, 152, 232448, plan) != 0)
    return 6;
  if (plan[0] != MOE_LORA_PATH_TCGEN05) return 7;
  /* every device entry point links from C; argument errors return before any CUDA call */
  {
    const moe_lora_bf16 *a[1] = {NULL}, *b[1] = {NULL};
    if (moe_lora_align(NULL, NULL, NULL, NULL, 16, 0, 8, 2, 2, 16, NULL, NULL, NULL, 152, 10, NULL, 0,
                       MOE_LORA_ALIGN_AUTO, NULL, NULL) != MOE_LORA_ERR_INVALID_ARG) return 8;
    if (moe_align_block_size(NULL, 16, 2, 8, 8, NULL, NULL, NULL, 152, 10, NULL, 0, MOE_LORA_ALIGN_AUTO, NULL,
                             NULL) != MOE_LORA_ERR_UNSUPPORTED) return 9;
    if (moe_lora_align_static_workspace(NULL, NULL, NULL, NULL, 16, 0, 8, 2, 0, 16, NULL, NULL, NULL, 152, 10,
                                        NULL, NULL) != MOE_LORA_ERR_INVALID_ARG) return 10;
    if (moe_lora_fused_shrink_expand(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 16, 2, 8, 256, 512, 132,
                                     2, 2, 16, 152, 10, 1, MOE_LORA_PATH_AUTO, NULL, NULL)
        != MOE_LORA_ERR_UNSUPPORTED) return 11;
    if (moe_lora_fused_shrink_expand_ex(NULL, 0, a, b, 0, NULL, 512, 0, NULL, NULL, NULL, NULL, NULL, NULL, 16, 2,
                                        8, 256, 512, 8, 2, 2, 16, 152, 10, 1, MOE_LORA_PATH_AUTO, NULL, NULL)
        != MOE_LORA_ERR_INVALID_ARG) return 12;
    if (moe_lora_fused_shrink_expand_naive(NULL, 0, a, b, 1, NULL, 512, 0, NULL, NULL, NULL, NULL, NULL, 16, 2, 8,
                                           260, 512, 8, 2, 2, 1, MOE_LORA_PATH_AUTO, NULL, NULL)
        != MOE_LORA_ERR_MISALIGNED) return 13;
    if (moe_lora_align_workspace_bytes(4096, 8, 256, 1, 64, MOE_LORA_ALIGN_GLOBAL) == 0) return 14;
  }
  printf("ok\n");
  return 0;
}
""")
    exe = tmp_path / "consumer"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                           "-I", os.path.join(root, "include"), str(src), "-L", lib_dir, "-lmoe_lora",
                           "-Wl,-rpath," + lib_dir, "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)

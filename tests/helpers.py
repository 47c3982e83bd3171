"""Shared test helpers: move seeded inputs to the GPU, run the library's two
stages through the binding, and compare against the CPU oracle."""
import os

import numpy as np
import torch

import oracle
from lora_moe_gb300 import binding as B
from lora_moe_gb300 import inputs as gen

POISON = 0x7FFFFFFF       # undefined align output entries keep this
TOL_ABS, TOL_REL = 1e-2, 1e-2


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def host_bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_align(inp_or_parts, E, L, bs, variant=B.ALIGN_AUTO, adapter_enabled=None, poison=True):
    """Run moe_lora_align; returns numpy (sorted, experts, ntpp, err) and device buffers."""
    topk_ids, mapping, lora_ids = inp_or_parts
    M, topk = topk_ids.shape
    buf = B.AlignBuffers(M, topk, E, L, len(lora_ids), bs, variant=variant)
    if poison:
        buf.sorted_token_ids.fill_(POISON)
        buf.expert_ids.fill_(POISON)
        buf.num_tokens_post_padded.fill_(POISON)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    en = dev_i32(adapter_enabled) if adapter_enabled is not None else None
    B.moe_lora_align(dev_i32(topk_ids), dev_i32(mapping), dev_i32(lora_ids), E, L, bs,
                     buf.sorted_token_ids, buf.expert_ids, buf.num_tokens_post_padded,
                     adapter_enabled=en, workspace=buf.workspace, variant=variant, err_flag=err)
    torch.cuda.synchronize()
    return (buf.sorted_token_ids.cpu().numpy(), buf.expert_ids.cpu().numpy(),
            buf.num_tokens_post_padded.cpu().numpy(), int(err.item()), buf)


def assert_align_equal(topk_ids, mapping, lora_ids, E, L, bs, variant=B.ALIGN_AUTO, adapter_enabled=None):
    """GPU align must equal the oracle bit for bit on the defined entries and
    leave every other entry untouched."""
    s, e, n, err, _ = gpu_align((topk_ids, mapping, lora_ids), E, L, bs, variant, adapter_enabled)
    ost, os_, oe, on = oracle.align(topk_ids, mapping, lora_ids, E, L, bs,
                                    adapter_enabled=adapter_enabled,
                                    max_num_tokens_padded=s.shape[1], max_num_m_blocks=e.shape[1],
                                    fill=POISON)
    assert np.array_equal(n, on), (n, on)
    assert np.array_equal(s, os_)
    assert np.array_equal(e, oe)
    want_err = 0
    if ost & oracle.STATUS_BAD_EXPERT_ID:
        want_err |= B.DEVERR_EXPERT_ID
    if ost & oracle.STATUS_BAD_LORA_ID:
        want_err |= B.DEVERR_LORA_ID
    assert err == want_err, (err, ost)
    return s, e, n


class DeviceInputs:
    def __init__(self, inp: gen.Inputs, variant=B.ALIGN_AUTO):
        w = inp.w
        self.w = w
        self.topk_ids = dev_i32(inp.topk_ids)
        self.mapping = dev_i32(inp.token_lora_mapping)
        self.lora_ids = dev_i32(inp.lora_ids)
        self.x = dev_bf16(inp.x)
        self.a = dev_bf16(inp.lora_a)
        self.b = dev_bf16(inp.lora_b)
        self.y_in = dev_bf16(inp.y_in)
        self.buf = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size,
                                  variant=variant)


def gpu_step(d: DeviceInputs, add_inputs=True, path=B.PATH_AUTO, variant=B.ALIGN_AUTO, adapter_enabled=None,
             poison_align=True):
    """Align then fused on the device; returns (y, err)."""
    w = d.w
    if poison_align:
        d.buf.sorted_token_ids.fill_(POISON)
        d.buf.expert_ids.fill_(POISON)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    en = dev_i32(adapter_enabled) if adapter_enabled is not None else None
    B.moe_lora_align(d.topk_ids, d.mapping, d.lora_ids, w.E, w.max_loras, w.block_size,
                     d.buf.sorted_token_ids, d.buf.expert_ids, d.buf.num_tokens_post_padded,
                     adapter_enabled=en, workspace=d.buf.workspace, variant=variant, err_flag=err)
    y = d.y_in.clone()
    B.moe_lora_fused_shrink_expand(d.x, d.a, d.b, y, d.buf.sorted_token_ids, d.buf.expert_ids,
                                   d.buf.num_tokens_post_padded, d.lora_ids, w.topk, w.block_size,
                                   add_inputs=add_inputs, adapter_enabled=en, path=path, err_flag=err)
    torch.cuda.synchronize()
    return y, int(err.item())


def covered(inp: gen.Inputs, adapter_enabled=None):
    w = inp.w
    cov = np.zeros((w.M, w.topk), bool)
    act = set(int(v) for v in inp.lora_ids)
    for m in range(w.M):
        l = int(inp.token_lora_mapping[m])
        if l in act and (adapter_enabled is None or adapter_enabled[l]):
            cov[m] = (inp.topk_ids[m] >= 0) & (inp.topk_ids[m] < w.E)
    return cov


def check_close(got_bits, ref, what=""):
    """|gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise; NaN / Inf fail."""
    got = gen.bf16_bits_to_f32(got_bits).astype(np.float64)
    assert np.isfinite(got).all(), what + ": non-finite output"
    err = np.abs(got - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d elements out of tolerance, first at %s: got %r ref %r"
                             % (what, int(bad.sum()), tuple(i), got[tuple(i)], ref[tuple(i)]))
    return float(err.max()) if err.size else 0.0


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def as_ex(inp: gen.Inputs) -> gen.ExInputs:
    """The plain call's inputs as general-call inputs (one slice, no options)."""
    return gen.ExInputs(inp, inp.x, [inp.lora_a], [inp.lora_b], None, inp.y_in, False, 0)


def compare_every_pair(ex: gen.ExInputs, outs, add_inputs=True, adapter_enabled=None, chunk=256):
    """Compare GPU outputs with the oracle on every element.

    outs: {name: uint16 [M*topk, ldy] host copy of the GPU output}.  Covered
    pairs' slice columns must satisfy |gpu - ref| <= 1e-2 + 1e-2 |ref| against
    the oracle's general definition; every other element (uncovered pairs, the
    columns no slice writes) must equal y_in bit for bit.  The oracle runs on
    chunks of `chunk` covered pairs, one chunk per host thread at a time; each
    chunk's rows are compared with every output as soon as they are ready.
    Returns {name: largest error}."""
    from concurrent.futures import ThreadPoolExecutor
    inp, w = ex.base, ex.base.w
    P = w.M * w.topk
    yin = ex.y_in.reshape(P, -1)
    S = len(ex.lora_a)
    lo, hi = ex.y_offset, ex.y_offset + S * w.N
    cov = covered(inp, adapter_enabled).reshape(-1)
    unc = np.flatnonzero(~cov)
    for name, got in outs.items():
        assert got.shape == yin.shape, name
        assert np.array_equal(got[unc], yin[unc]), "%s: uncovered pairs were modified" % name
        assert np.array_equal(got[:, :lo], yin[:, :lo]) and np.array_equal(got[:, hi:], yin[:, hi:]), \
            "%s: columns outside the slices were modified" % name
    cov_idx = np.flatnonzero(cov).astype(np.int32)
    chunks = [cov_idx[i:i + chunk] for i in range(0, len(cov_idx), chunk)]

    def work(sel):
        ref = oracle.fused_ex(ex.x, ex.lora_a, ex.lora_b, ex.y_in, inp.topk_ids, inp.token_lora_mapping,
                              inp.lora_ids, add_inputs=add_inputs, adapter_enabled=adapter_enabled,
                              topk_weights=ex.topk_weights, x_per_pair=ex.x_per_pair, y_offset=ex.y_offset,
                              pairs=sel)
        return {name: check_close(got[sel][:, lo:hi], ref[:, lo:hi],
                                  "%s %s pairs %d..%d" % (w.name, name, int(sel[0]), int(sel[-1])))
                for name, got in outs.items()}

    worst = {name: 0.0 for name in outs}
    with ThreadPoolExecutor(max_workers=max(1, host_threads())) as pool:
        for res in pool.map(work, chunks):
            for name, e in res.items():
                worst[name] = max(worst[name], e)
    return worst

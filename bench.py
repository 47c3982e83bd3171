"""Benchmark of the multi-LoRA MoE adapter path on one GB300 (per rank).

One step = one pass of the whole path over one batch: moe_lora_align followed
by moe_lora_fused_shrink_expand (add_inputs=1).  The metric is microseconds
per step (lower is better).  The headline workload is the largest
configuration of the specification, large_e_nact8 (M=4096, K=7168, N=4096,
E=256, topk=8, max_loras=8 all active, r=128, block_size=64, Zipf(1.2)
routing); inputs are synthetic and seeded.  The same run measures every other
configuration (tiny, decode Qwen3, decode gpt-oss, prefill Mixtral, large E
with 1 and 4 active adapters) and reports each under "configs": fused and
align microseconds (both align variants forced as well), the step, GB/s,
TFLOP/s and the fractions of the measured HBM and bf16 peaks.

Timing: inputs are resident in HBM; NB rotating copies of every input whose
total footprint exceeds 3x L2 are cycled so that no step finds its operands in
L2; W untimed warm-up steps; then timed regions of exactly K steps each,
replayed from CUDA graphs, each bracketed by a barrier and a device
synchronisation and timed with CUDA events on the launching stream (max over
ranks).  Regions are repeated (at least 5, and until they add up to 0.5 s of
device time) and the median is reported.  Kernel-level durations (align
alone, fused alone) are taken the same way for the roofline entry.

Launch under torchrun for N > 1: every rank runs its own replica (the path has
no exchange step); rank 0 prints the JSON line.

Options of the general fused call (moe_lora_fused_shrink_expand_ex), off by
default: --slices S (separate adapters per slice, e.g. 2 for w13's gate and
up), --per-pair-x (one input row per pair, the w2 stage), --routed-weight
(delta scaled by the router weight).  With any of them the step runs the
general call instead of the plain one.  --align-variant 1|2 forces the
shared-memory or the global-memory align (default: the library's choice).

--impl reference times the CPU oracle (test infrastructure) on the host cores
instead, on a bounded sample of pairs per step, scaled to microseconds per
full step.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lora_moe_gb300 import inputs as gen  # noqa: E402

DEFAULT_WORKLOAD = "large_e_nact8"
METRIC = "fused MoE-LoRA us/call (align + fused shrink/expand step)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernel-seconds", type=float, default=0.3,
                    help="device time spent on each kernel-level timing")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run W + this many eager steps (for ncu); prints no JSON line")
    ap.add_argument("--path", type=int, default=0, help="fused path: 0 auto, 1 CUDA cores, 2 tcgen05, 3 CUDA-core cluster, 4 CUDA-core streaming")
    ap.add_argument("--align-variant", type=int, default=0, choices=[0, 1, 2, 3],
                    help="align variant: 0 auto, 1 shared memory (one CTA per slot), 2 global memory (three "
                         "launches), 3 cluster (one launch, a thread-block cluster per slot)")
    ap.add_argument("--sets", type=int, default=0, help="rotating input sets (0: enough to exceed 3x L2)")
    ap.add_argument("--slices", type=int, default=1, help="adapter slices per layer (general call)")
    ap.add_argument("--per-pair-x", action="store_true", help="one input row per pair (general call)")
    ap.add_argument("--routed-weight", action="store_true", help="scale by the router weight (general call)")
    ap.add_argument("--naive", action="store_true",
                    help="naive block assignment: the step is the fused call alone, one work item per pair")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="also measure every configuration of the specification (per-config entries)")
    ap.add_argument("--min-regions", type=int, default=5, help="fewest timed K-step regions (median reported)")
    ap.add_argument("--min-timed-seconds", type=float, default=0.5,
                    help="timed regions are repeated until they add up to this much device time")
    ap.add_argument("--max-regions", type=int, default=200)
    return ap.parse_args()


def uses_ex(args):
    return args.slices != 1 or args.per_pair_x or args.routed_weight or args.naive


def make_step_inputs(w, args):
    """(routing inputs, general-call inputs or None)."""
    if not uses_ex(args):
        return gen.make_inputs(w), None
    ex = gen.make_ex_inputs(w, num_slices=args.slices, x_per_pair=args.per_pair_x,
                            routed_weights=args.routed_weight)
    return ex.base, ex


# --------------------------------------------------------------------------- roofline bookkeeping

def algorithmic_counts(inp: gen.Inputs, slices=1, per_pair_x=False, routed_weight=False, naive=False):
    """What the method must move / compute for one step, from the actual inputs.

    bytes = x rows of covered tokens (or covered pairs, with one input row per
    pair) once + A and B of every touched (lora, expert) segment once per slice
    + y read and write of covered pairs' slice columns + router weights of
    covered pairs + align metadata; flops = 2 r (K + N) per covered pair and
    slice."""
    w = inp.w
    act = set(int(v) for v in inp.lora_ids)
    m_cov = np.array([int(l) in act for l in inp.token_lora_mapping])
    pairs = [(int(inp.token_lora_mapping[m]), int(inp.topk_ids[m, k]))
             for m in range(w.M) if m_cov[m] for k in range(w.topk)]
    P = len(pairs)
    segs = {}
    for le in pairs:
        segs[le] = segs.get(le, 0) + 1
    S = len(segs)
    padded = sum(-(-c // w.block_size) * w.block_size for c in segs.values())
    blocks = padded // w.block_size
    r = w.rank
    x_rows = P if per_pair_x else int(m_cov.sum())
    # routing metadata the fused stage reads: the align outputs, or (naive
    # block assignment) topk_ids and token_lora_mapping
    meta = 4 * (w.M * w.topk + w.M) if naive else 4 * (padded + blocks + w.num_active_loras)
    fused_bytes = (2 * w.K * x_rows + slices * S * 2 * r * (w.K + w.N) + slices * P * w.N * 2 * 2
                   + (4 * P if routed_weight else 0) + meta)
    align_bytes = 4 * w.M * w.topk + 4 * w.M + 4 * (padded + blocks + w.num_active_loras)
    return dict(pairs=P, segments=S, padded_rows=padded, blocks=blocks, fused_bytes=fused_bytes,
                align_bytes=align_bytes, flops=2 * r * (w.K + w.N) * P * slices)


# DRAM bytes per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture of the plain call, by workload
# and kernel; profiles/ holds each capture's summary and command.  An entry
# must go when its kernel changes.
NCU_TRAFFIC = {
    ("decode_qwen3_w13", "fused_cuda_core_kernel"): 5578496,      # fused_cuda_core_decode_qwen3_w13.md
    ("decode_gptoss_w2", "fused_tcgen05_kernel"): 170909184,      # fused_tcgen05_decode_gptoss_w2.md
    ("decode_gptoss_w2", "fused_cluster_stream_kernel"): 155413504,  # fused_cluster_stream_decode_gptoss_w2.md
    ("large_e_l1", "fused_tcgen05_kernel"): 1080333056,           # fused_tcgen05_large_e_l1.md
    # the same active work as large_e_l1 (the inactive slots are never read)
    ("large_e_nact1", "fused_tcgen05_kernel"): 1080333056,        # fused_tcgen05_large_e_l1.md
    ("large_e_nact4", "fused_tcgen05_kernel"): 3439547904,        # fused_tcgen05_large_e_nact4_traffic.md
    ("large_e_nact8", "fused_tcgen05_kernel"): 6153373440,        # fused_tcgen05_large_e_nact8_traffic.md
    ("prefill_mixtral_w13_m2048", "fused_tcgen05_kernel"): 468284416,  # fused_tcgen05_prefill_mixtral_w13_m2048.md
    ("prefill_mixtral_w13", "fused_tcgen05_kernel"): 2211975168,  # fused_tcgen05_prefill_mixtral_w13_traffic.md
}


def _peaks_file():
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
        return json.load(fh)


def measured_peaks():
    """HBM copy bandwidth (GB/s): the measured figure, else the fallback."""
    try:
        return float(_peaks_file()["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor throughput (TFLOP/s) for a kernel timed alone: the
    measured burst figure, else the fallback."""
    try:
        return float(_peaks_file()["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        samples = []
        for _, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                samples.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                    reasons=dict(hw_slowdown=parts[5], hw_thermal_slowdown=parts[6],
                                                 sw_thermal_slowdown=parts[7], sw_power_cap=parts[8])))
            except ValueError:
                continue
        if not samples:
            return None
        reasons = sorted({k for s in samples for k, v in s["reasons"].items() if v.lower() == "active"})
        return {"sm_mhz": float(np.median([s["sm"] for s in samples])),
                "sm_max_mhz": max(s["sm_max"] for s in samples),
                "reasons": reasons, "samples": len(samples)}


# --------------------------------------------------------------------------- distributed plumbing

def dist_setup(use_cuda):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if use_cuda else "gloo")
        pg = dist
    return world, rank, local, pg


def barrier(pg, use_cuda):
    if pg is not None:
        if use_cuda:
            import torch
            pg.barrier(device_ids=[torch.cuda.current_device()])
        else:
            pg.barrier()


def max_over_ranks(pg, value, use_cuda):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_us_per_step(pg, ms_local, steps, world, use_cuda):
    """Whole-job microseconds per step: the slowest rank's time for its
    `steps` steps, over all ranks' steps (each rank runs its own replica)."""
    ms = max_over_ranks(pg, ms_local, use_cuda)
    return ms * 1e3 / (steps * world), ms


# --------------------------------------------------------------------------- CPU oracle timing

def time_oracle(inp: gen.Inputs, budget_s: float, pairs_per_call: int, calls: int = None, ex=None,
                with_align=True):
    """Time the oracle's align (whole batch) and fused stage (a rotating subset
    of covered pairs, every column; the general definition when `ex` holds the
    general call's inputs) and scale to microseconds per full step.

    Returns (us_per_step, description, calls_made)."""
    import oracle
    w = inp.w
    cov_idx = _covered_pairs(inp)
    cols = np.arange(w.N, dtype=np.int32)
    n = max(1, min(pairs_per_call, len(cov_idx)))
    t_align = t_fused = 0.0
    done_pairs = 0
    made = 0
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        if with_align:
            oracle.align(inp.topk_ids, inp.token_lora_mapping, inp.lora_ids, w.E, w.max_loras, w.block_size)
        t1 = time.perf_counter()
        sel = cov_idx[(made * n + np.arange(n)) % max(1, len(cov_idx))] if len(cov_idx) else cov_idx
        if len(sel):
            _oracle_pairs(inp, ex, sel, cols)
        t2 = time.perf_counter()
        t_align += t1 - t0
        t_fused += t2 - t1
        done_pairs += len(sel)
        made += 1
        if calls is not None:
            if made >= calls:
                break
        elif time.perf_counter() - t_start >= budget_s:
            break
    per_pair = t_fused / max(1, done_pairs)
    us = (t_align / made + per_pair * len(cov_idx)) * 1e6
    desc = ("%soracle fused over %d of %d covered pairs per call (all %d columns), %d calls, scaled to one "
            "full step" % ("oracle align over the whole batch + " if with_align else "", n, len(cov_idx), w.N, made))
    return us, desc, made


def _covered_pairs(inp: gen.Inputs):
    w = inp.w
    act = set(int(v) for v in inp.lora_ids)
    cov = np.array([int(inp.token_lora_mapping[f // w.topk]) in act for f in range(w.M * w.topk)])
    return np.flatnonzero(cov).astype(np.int32)


def _oracle_pairs(inp: gen.Inputs, ex, sel, cols):
    """One oracle call of the fused stage at the flat pairs `sel` (every column)."""
    import oracle
    if ex is not None:
        return oracle.fused_ex(ex.x, ex.lora_a, ex.lora_b, ex.y_in, inp.topk_ids, inp.token_lora_mapping,
                               inp.lora_ids, topk_weights=ex.topk_weights, x_per_pair=ex.x_per_pair,
                               y_offset=ex.y_offset, pairs=sel)
    return oracle.fused_sampled(inp.x, inp.lora_a, inp.lora_b, inp.y_in, inp.topk_ids, inp.token_lora_mapping,
                                inp.lora_ids, sel, cols)


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle_threads(inp: gen.Inputs, budget_s: float, pairs_per_thread: int, threads: int, ex=None,
                        with_align=True):
    """The same oracle, its fused stage spread over `threads` host threads.

    Every call's pairs are cut into `threads` contiguous chunks, one oracle
    call per chunk on its own thread; the oracle is a C library entered through
    ctypes, which drops the GIL for the call, and each pair's output depends on
    that pair alone, so the chunks run in parallel and need no merging beyond
    concatenation.  The align (one sequential pass over the batch) stays on the
    calling thread.  The first call's output is checked equal, element for
    element, to one single-threaded oracle call on the same pairs.

    Returns (us_per_step, description, threads)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    w = inp.w
    cov_idx = _covered_pairs(inp)
    cols = np.arange(w.N, dtype=np.int32)
    threads = max(1, min(threads, len(cov_idx))) if len(cov_idx) else 1
    n = max(1, min(pairs_per_thread * threads, len(cov_idx)))
    t_align = t_fused = 0.0
    done_pairs = made = 0
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t_start = time.perf_counter()
        while True:
            t0 = time.perf_counter()
            if with_align:
                oracle.align(inp.topk_ids, inp.token_lora_mapping, inp.lora_ids, w.E, w.max_loras, w.block_size)
            t1 = time.perf_counter()
            sel = cov_idx[(made * n + np.arange(n)) % max(1, len(cov_idx))] if len(cov_idx) else cov_idx
            if len(sel):
                chunks = [c for c in np.array_split(sel, threads) if len(c)]
                outs = list(pool.map(lambda c: _oracle_pairs(inp, ex, c, cols), chunks))
            t2 = time.perf_counter()
            if made == 0 and len(sel):
                one = _oracle_pairs(inp, ex, sel, cols)
                if not np.array_equal(np.concatenate(outs, axis=0), one, equal_nan=True):
                    raise RuntimeError("threaded oracle run differs from the single-threaded one")
            t_align += t1 - t0
            t_fused += t2 - t1
            done_pairs += len(sel)
            made += 1
            if time.perf_counter() - t_start >= budget_s:
                break
    per_pair = t_fused / max(1, done_pairs)
    us = (t_align / made + per_pair * len(cov_idx)) * 1e6
    desc = ("%soracle fused over %d of %d covered pairs per call split over %d threads (all %d columns), "
            "%d calls, scaled to one full step; first call checked equal to a single-threaded run"
            % ("single-threaded oracle align over the whole batch + " if with_align else "", n, len(cov_idx),
               threads, w.N, made))
    return us, desc, threads


# --------------------------------------------------------------------------- GPU side

# The workloads of the per-config entries, in the order the specification
# lists them (tiny, decode Qwen3, decode gpt-oss, prefill Mixtral, large E
# with 1 / 4 / 8 active adapters).
CONFIG_WORKLOADS = ["tiny", "decode_qwen3_w13", "decode_gptoss_w2", "prefill_mixtral_w13",
                    "large_e_nact1", "large_e_nact4", "large_e_nact8"]


class Rig:
    """NB rotating device copies of one workload's inputs (enough that their
    total footprint exceeds 3x L2), their align buffers, and the two calls of
    a step on them."""

    def __init__(self, w, args, dev, stream, err, inp=None, ex=None):
        import torch
        from lora_moe_gb300 import binding as B
        self.B, self.w, self.args, self.dev, self.stream, self.err = B, w, args, dev, stream, err
        if inp is None:
            inp, ex = make_step_inputs(w, args)
        self.inp, self.ex = inp, ex
        src = ex if ex is not None else inp
        self.src = src
        a_list = src.lora_a if ex is not None else [inp.lora_a]
        b_list = src.lora_b if ex is not None else [inp.lora_b]

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.per_set = (src.x.nbytes + sum(a.nbytes for a in a_list) + sum(b.nbytes for b in b_list) +
                        2 * src.y_in.nbytes + inp.topk_ids.nbytes + inp.token_lora_mapping.nbytes)
        self.NB = args.sets if args.sets > 0 else int(max(2, min(64, -(-3 * self.l2 // self.per_set))))
        base = dict(topk_ids=i32(inp.topk_ids), mapping=i32(inp.token_lora_mapping), lora_ids=i32(inp.lora_ids),
                    x=bf16(src.x), y=bf16(src.y_in))
        self.adapter_keys = []
        for i, (a, b) in enumerate(zip(a_list, b_list)):
            base["a%d" % i] = bf16(a)
            base["b%d" % i] = bf16(b)
            self.adapter_keys += ["a%d" % i, "b%d" % i]
        if ex is not None and ex.topk_weights is not None:
            base["w"] = torch.from_numpy(ex.topk_weights).to(dev)
        self.sets = []
        for i in range(self.NB):
            s = {k: v.clone() for k, v in base.items()}
            s["buf"] = self.new_buffers()
            self.sets.append(s)
        del base
        self.align_launches = 0 if args.naive else self.launches_of(args.align_variant)

    def new_buffers(self):
        w = self.w
        # a workspace large enough for either variant, so that any variant can be forced
        return self.B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size,
                                   device=self.dev, variant=self.B.ALIGN_GLOBAL)

    def launches_of(self, variant):
        w = self.w
        ws = self.B.align_workspace_bytes(w.M, w.topk, w.E, w.num_active_loras, w.block_size, variant)
        return 3 if ws else 1

    def auto_variant_name(self):
        w = self.w
        v = self.B.align_resolve_variant(w.M, w.topk, w.E, self.B.ALIGN_AUTO)
        return {self.B.ALIGN_SMEM: "smem", self.B.ALIGN_GLOBAL: "global", self.B.ALIGN_CLUSTER: "cluster"}[v]

    def align(self, s, variant=None):
        w, b = self.w, s["buf"]
        self.B.moe_lora_align(s["topk_ids"], s["mapping"], s["lora_ids"], w.E, w.max_loras, w.block_size,
                              b.sorted_token_ids, b.expert_ids, b.num_tokens_post_padded, workspace=b.workspace,
                              variant=self.args.align_variant if variant is None else variant, err_flag=self.err,
                              stream=self.stream)

    def fused(self, s):
        w, b, args, ex, B = self.w, s["buf"], self.args, self.ex, self.B
        S = args.slices
        if args.naive:
            B.moe_lora_fused_shrink_expand_naive(
                s["x"], [s["a%d" % i] for i in range(S)], [s["b%d" % i] for i in range(S)],
                s["y"], s["topk_ids"], s["mapping"], s["lora_ids"], w.max_loras, add_inputs=True,
                topk_weights=s.get("w"), x_per_pair=ex.x_per_pair, y_offset=ex.y_offset, path=args.path,
                err_flag=self.err, stream=self.stream)
        elif ex is None:
            B.moe_lora_fused_shrink_expand(s["x"], s["a0"], s["b0"], s["y"], b.sorted_token_ids, b.expert_ids,
                                           b.num_tokens_post_padded, s["lora_ids"], w.topk, w.block_size,
                                           add_inputs=True, path=args.path, err_flag=self.err, stream=self.stream)
        else:
            B.moe_lora_fused_shrink_expand_ex(
                s["x"], [s["a%d" % i] for i in range(S)], [s["b%d" % i] for i in range(S)],
                s["y"], b.sorted_token_ids, b.expert_ids, b.num_tokens_post_padded, s["lora_ids"], w.topk,
                w.block_size, add_inputs=True, topk_weights=s.get("w"), x_per_pair=ex.x_per_pair,
                y_offset=ex.y_offset, path=args.path, err_flag=self.err, stream=self.stream)

    def step(self, i):
        s = self.sets[i % self.NB]
        if not self.args.naive:
            self.align(s)
        self.fused(s)

    def capture(self, fn, n):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    fn(i)
        return g

    def graph_time_us(self, fn, seconds):
        """Microseconds per call of fn, replayed from a graph of NB calls (one
        per input set) for about `seconds` of device time."""
        import torch
        g = self.capture(lambda i: fn(self.sets[i % self.NB]), self.NB)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        st = self.stream
        with torch.cuda.stream(st):
            g.replay()
            st.synchronize()
            a.record(st)
            g.replay()
            b.record(st)
            st.synchronize()
            one = max(1e-6, a.elapsed_time(b))
            reps = max(1, int(seconds * 1e3 / one))
            a.record(st)
            for _ in range(reps):
                g.replay()
            b.record(st)
            st.synchronize()
        del g
        return a.elapsed_time(b) * 1e3 / (reps * self.NB)

    def check_err(self):
        v = int(self.err.item())
        assert v == 0, "device error flag %d" % v

    def release(self):
        import torch
        self.sets = []
        torch.cuda.empty_cache()


def kernel_name_of(B, w, args):
    kernel = B.fused_resolve_path(w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras, w.block_size,
                                  args.slices, args.path)
    name = {B.PATH_TCGEN05: "fused_tcgen05_kernel", B.PATH_CUDA_CORE_CLUSTER: "fused_cuda_core_kernel",
            B.PATH_CUDA_CORE_STREAM: "fused_cluster_stream_kernel"}[kernel]
    if args.naive:
        naive_path = B.fused_naive_resolve_path(w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras, args.slices,
                                                args.path)
        name = ("fused_cluster_stream_kernel" if naive_path == B.PATH_CUDA_CORE_STREAM else "fused_cuda_core_kernel") \
            + " (naive block assignment)"
    return name


def config_entry(rig, counts, peak, tc_peak, seconds):
    """Per-config numbers, each kernel alone and the align + fused step, all
    from CUDA graphs over the rotating input sets."""
    B, w = rig.B, rig.w
    for i in range(max(3, rig.NB)):
        rig.step(i)
    rig.stream.synchronize()
    rig.check_err()
    fused_us = rig.graph_time_us(rig.fused, seconds)
    align = {}
    if not rig.args.naive:
        align["align_us"] = rig.graph_time_us(rig.align, seconds)
        align["align_us_smem"] = rig.graph_time_us(lambda s: rig.align(s, B.ALIGN_SMEM), seconds)
        align["align_us_global"] = rig.graph_time_us(lambda s: rig.align(s, B.ALIGN_GLOBAL), seconds)
        align["align_us_cluster"] = rig.graph_time_us(lambda s: rig.align(s, B.ALIGN_CLUSTER), seconds)
        align["align_variant_auto"] = rig.auto_variant_name()
    step_us = rig.graph_time_us(lambda s: (rig.align(s) if not rig.args.naive else None, rig.fused(s)), seconds)
    # Decode batches: the same batch through the naive entry point (no align,
    # one work item per pair), the model's other way to run a small batch.
    if not rig.args.naive and not uses_ex(rig.args) and w.M * w.topk <= 4096:
        def naive(s):
            B.moe_lora_fused_shrink_expand_naive(s["x"], s["a0"], s["b0"], s["y"], s["topk_ids"], s["mapping"],
                                                 s["lora_ids"], w.max_loras, add_inputs=True, err_flag=rig.err,
                                                 stream=rig.stream)
        align["naive_step_us"] = rig.graph_time_us(naive, seconds)
        align["naive_kernel"] = "fused_cluster_stream_kernel" if B.fused_naive_resolve_path(
            w.M, w.topk, w.E, w.K, w.N, w.rank, w.num_active_loras) == B.PATH_CUDA_CORE_STREAM \
            else "fused_cuda_core_kernel"
    rig.check_err()
    gbs = counts["fused_bytes"] / (fused_us * 1e-6) / 1e9
    tflops = counts["flops"] / (fused_us * 1e-6) / 1e12
    kname = kernel_name_of(B, w, rig.args)
    return dict({"kernel": kname, "step_us": step_us, "fused_us": fused_us,
                 "fused_gbs": gbs, "fused_tflops": tflops, "frac_hbm": gbs / peak,
                 "frac_bf16_tensor": tflops / tc_peak,
                 "fused_bytes": counts["fused_bytes"], "flops": counts["flops"], "pairs": counts["pairs"],
                 "blocks": counts["blocks"], "traffic_ncu": NCU_TRAFFIC.get((w.name, kname))}, **align)


def run_ours(args, world, rank, local, pg):
    import torch
    from lora_moe_gb300 import binding as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = gen.WORKLOADS[args.workload]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    rig = Rig(w, args, dev, stream, err)
    inp, ex = rig.inp, rig.ex
    counts = algorithmic_counts(inp, args.slices, args.per_pair_x, args.routed_weight, args.naive)
    NB = rig.NB

    if args.profile_steps:
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.profile_steps):
                rig.step(i)
        stream.synchronize()
        rig.check_err()
        return None

    # warm-up (also primes every set's align output for the fused-only timing)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, NB)):
            rig.step(i)
    stream.synchronize()
    rig.check_err()

    g_round = rig.capture(rig.step, NB)
    rem = args.steps % NB
    g_rem = rig.capture(rig.step, rem) if rem else None
    stream.synchronize()

    # ---------------- timed regions: each exactly K steps; the median is reported
    def timed_region():
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(pg, True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps // NB):
                g_round.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        barrier(pg, True)
        return max_over_ranks(pg, e0.elapsed_time(e1), True)

    sampler = ClockSampler(local)
    sampler.start()
    regions = [timed_region()]
    want = max(args.min_regions, int(np.ceil(args.min_timed_seconds * 1e3 / max(1e-6, regions[0]))))
    while len(regions) < min(want, args.max_regions):
        regions.append(timed_region())
    clocks = sampler.stop()
    rig.check_err()
    ms = float(np.median(regions))

    # ---------------- kernel-level timing (each kernel alone, same rotation)
    fused_us = rig.graph_time_us(rig.fused, args.kernel_seconds)
    align_us = None if args.naive else rig.graph_time_us(rig.align, args.kernel_seconds)
    align_launches = rig.align_launches

    # ---------------- end to end through the public API with host buffers
    # Each step's inputs (routing, x, y_in, router weights) sit in one pinned
    # host buffer, laid out like one device buffer whose slices the calls
    # take: one host-to-device copy per step, the two calls, and y read back.
    e2e = None
    if not args.no_e2e:
        src = rig.src
        parts = [("topk_ids", inp.topk_ids), ("mapping", inp.token_lora_mapping), ("lora_ids", inp.lora_ids),
                 ("x", src.x), ("y", src.y_in)]
        if ex is not None and ex.topk_weights is not None:
            parts.append(("w", ex.topk_weights))
        layout, total = {}, 0
        for name, arr in parts:
            layout[name] = (total, arr)
            total += (arr.nbytes + 255) // 256 * 256
        host_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
        for name, (off, arr) in layout.items():
            host_pack[off:off + arr.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
        tdt = {"topk_ids": torch.int32, "mapping": torch.int32, "lora_ids": torch.int32, "x": torch.bfloat16,
               "y": torch.bfloat16, "w": torch.float32}
        # three device buffers: in the pipelined mode step i + 1's inputs go
        # up while step i computes and step i - 1's y comes back (with two, a
        # buffer's upload would wait for its previous read-back, and the
        # copies and calls would chain into one cycle per two steps)
        NBUF = 3
        packs = []
        for k in range(NBUF):
            dev_pack = torch.empty(total, dtype=torch.uint8, device=dev)
            v = {"pack": dev_pack}
            for name, (off, arr) in layout.items():
                v[name] = dev_pack[off:off + arr.nbytes].view(tdt[name]).view(arr.shape)
            for name in rig.adapter_keys:
                v[name] = rig.sets[0][name]
            v["buf"] = B.AlignBuffers(w.M, w.topk, w.E, w.max_loras, w.num_active_loras, w.block_size,
                                      device=dev, variant=args.align_variant)
            packs.append(v)
        out_host = torch.empty(src.y_in.shape, dtype=torch.int16).pin_memory()
        h2d = total
        d2h = out_host.numel() * out_host.element_size()
        n_e2e = max(4, min(args.steps, 2000))

        def e2e_step(i):
            v = packs[i % 2]
            with torch.cuda.stream(stream):
                v["pack"].copy_(host_pack, non_blocking=True)
            if not args.naive:
                rig.align(v)
            rig.fused(v)
            with torch.cuda.stream(stream):
                out_host.copy_(v["y"].view(torch.int16), non_blocking=True)

        for i in range(3):
            e2e_step(i)
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        barrier(pg, True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n_e2e):
            e2e_step(i)
        b.record(stream)
        stream.synchronize()
        eager_ms = max_over_ranks(pg, a.elapsed_time(b), True)
        # The same steps captured in a CUDA graph (the way serving engines run
        # decode steps): every replayed step still copies its inputs from
        # pinned host memory, runs the calls and reads y back to the host.
        g_e2e = rig.capture(e2e_step, 2)
        reps = max(2, n_e2e // 2)
        with torch.cuda.stream(stream):
            g_e2e.replay()
        stream.synchronize()
        barrier(pg, True)
        torch.cuda.synchronize()
        a.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g_e2e.replay()
        b.record(stream)
        stream.synchronize()
        graph_ms = max_over_ranks(pg, a.elapsed_time(b), True)
        rig.check_err()
        del g_e2e
        # Pipelined: the same copies and calls with the copies on their own
        # streams, so that step i + 1's inputs go up and step i - 1's y comes
        # back while step i computes (three packed buffers and three pinned
        # outputs rotate; a buffer is refilled only after its y has been read
        # back).
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)
        out_hosts = [out_host] + [torch.empty(src.y_in.shape, dtype=torch.int16).pin_memory()
                                  for _ in range(NBUF - 1)]
        ev_in = [torch.cuda.Event() for _ in range(NBUF)]
        ev_cmp = [torch.cuda.Event() for _ in range(NBUF)]
        ev_free = [torch.cuda.Event() for _ in range(NBUF)]

        def piped_step(i):
            k = i % NBUF
            v = packs[k]
            if i >= NBUF:
                s_in.wait_event(ev_free[k])
            with torch.cuda.stream(s_in):
                v["pack"].copy_(host_pack, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if not args.naive:
                rig.align(v)
            rig.fused(v)
            ev_cmp[k].record(stream)
            s_out.wait_event(ev_cmp[k])
            with torch.cuda.stream(s_out):
                out_hosts[k].copy_(v["y"].view(torch.int16), non_blocking=True)
                ev_free[k].record(s_out)

        def piped_run(n):
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            for i in range(n):
                piped_step(i)
            stream.wait_stream(s_out)
            stream.wait_stream(s_in)

        piped_run(4)
        torch.cuda.synchronize()
        barrier(pg, True)
        torch.cuda.synchronize()
        a.record(stream)
        piped_run(n_e2e)
        b.record(stream)
        torch.cuda.synchronize()
        piped_ms = max_over_ranks(pg, a.elapsed_time(b), True)
        rig.check_err()
        graph_us = graph_ms * 1e3 / (reps * 2 * world)
        piped_us = piped_ms * 1e3 / (n_e2e * world)
        modes = {"graph": ("CUDA graph of each step's host-to-device copy of its packed inputs, the calls and the "
                           "read-back of y, one after another", graph_us, reps * 2),
                 "pipelined": ("each step's host-to-device copy of its packed inputs, the calls and the read-back "
                               "of y, issued from the host with the copies on their own streams so that copies "
                               "of neighbouring steps overlap a step's calls", piped_us, n_e2e)}
        best = min(modes, key=lambda m: modes[m][1])
        e2e = {"value": modes[best][1], "unit": "us/call", "steps": modes[best][2],
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "mode": modes[best][0],
               "graph_value": graph_us, "pipelined_value": piped_us,
               "eager_value": eager_ms * 1e3 / (n_e2e * world)}
        del packs

    peak, peak_kind = measured_peaks()
    tc_peak, tc_kind = measured_tensor_peak()
    achieved = counts["fused_bytes"] / (fused_us * 1e-6) / 1e9
    kernel_name = kernel_name_of(B, w, args)
    res = dict(ms=ms, regions=regions, clocks=clocks, fused_us=fused_us, align_us=align_us, counts=counts, NB=NB,
               l2=rig.l2, footprint=NB * rig.per_set, kernel_name=kernel_name, align_launches=align_launches,
               e2e=e2e, achieved=achieved, peak=peak, peak_kind=peak_kind, tc_peak=tc_peak, tc_kind=tc_kind,
               inp=inp, ex=ex)
    del g_round, g_rem

    # ---------------- the other configurations, measured in the same run
    configs = {}
    if args.configs == "all" and not uses_ex(args) and args.path == 0 and args.align_variant == 0:
        configs[w.name] = config_entry(rig, counts, peak, tc_peak, args.kernel_seconds)
        rig.release()
        del rig
        for name in CONFIG_WORKLOADS:
            if name == w.name:
                continue
            wc = gen.WORKLOADS[name]
            r2 = Rig(wc, args, dev, stream, err)
            c2 = algorithmic_counts(r2.inp)
            configs[name] = config_entry(r2, c2, peak, tc_peak, args.kernel_seconds)
            r2.release()
            del r2
    res["configs"] = configs
    return res


def ex_config(args):
    """Config keys of the options off the default: the general call's (none
    for the plain call) and a forced align variant."""
    d = {}
    if uses_ex(args):
        d = {"num_slices": args.slices, "x_per_pair": bool(args.per_pair_x),
             "routed_weight": bool(args.routed_weight)}
        if args.naive:
            d["block_assignment"] = "naive (no align)"
    if args.align_variant:
        d["align_variant"] = {1: "smem (forced)", 2: "global (forced)", 3: "cluster (forced)"}[args.align_variant]
    return d


def main():
    args = parse()
    if args.steps < 1 or args.warmup < 3:
        raise SystemExit("need --steps >= 1 and --warmup >= 3")
    w = gen.WORKLOADS[args.workload]

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        inp, ex = make_step_inputs(w, args)
        # size the per-step sample so that W + K steps take a couple of minutes at most
        wa = not args.naive
        probe_us, _, _ = time_oracle(inp, 0.5, 4, ex=ex, with_align=wa)
        per_pair_budget = 120.0 / (args.steps + args.warmup)
        pairs_per_call = max(1, int(per_pair_budget / max(1e-9, probe_us * 1e-6 / max(1, algorithmic_counts(inp)["pairs"]))))
        time_oracle(inp, 0, pairs_per_call, calls=args.warmup, ex=ex, with_align=wa)
        t0 = time.perf_counter()
        us, desc, made = time_oracle(inp, 0, pairs_per_call, calls=args.steps, ex=ex, with_align=wa)
        wall = time.perf_counter() - t0
        line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/call", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
                "config": dict({"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "E": w.E, "topk": w.topk,
                                "max_loras": w.max_loras, "num_active_loras": w.num_active_loras, "rank": w.rank,
                                "block_size": w.block_size}, **ex_config(args)),
                "cpu_baseline": {"value": us, "unit": "us/call", "cores": 1, "kind": "oracle", "sample": desc},
                "e2e": {"value": us, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": wall}
        print(json.dumps(line))
        return

    import torch
    world, rank, local, pg = dist_setup(True)
    res = run_ours(args, world, rank, local, pg)
    if res is None:
        print("profile run done: %d warm-up + %d steps of %s" % (args.warmup, args.profile_steps, w.name))
        return
    counts = res["counts"]
    us_per_step = res["ms"] * 1e3 / (args.steps * world)
    cpu = cpu_threads = None
    if rank == 0 and not args.no_cpu_baseline:
        us, desc, made = time_oracle(res["inp"], 12.0, 8, ex=res["ex"], with_align=not args.naive)
        cpu = {"value": us, "unit": "us/call", "cores": 1, "kind": "oracle", "sample": desc}
        try:
            us_t, desc_t, nt = time_oracle_threads(res["inp"], 4.0, 8, host_threads(), ex=res["ex"],
                                                   with_align=not args.naive)
            cpu_threads = {"value": us_t, "unit": "us/call", "cores": nt, "kind": "oracle", "sample": desc_t}
        except Exception as exc:   # a secondary baseline: reported, never fatal to the line
            cpu_threads = {"value": None, "error": "%s: %s" % (type(exc).__name__, exc)}
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return
    regions = res["regions"]
    launches_per_step = res["align_launches"] + 1
    tflops = counts["flops"] / (res["fused_us"] * 1e-6) / 1e12
    line = {
        "metric": METRIC, "value": us_per_step, "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms"] / args.steps, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
        "data": "synthetic (seeded numpy PCG64; random-init adapters, NaN-poisoned inactive slots)",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "E": w.E, "topk": w.topk,
                   "max_loras": w.max_loras, "num_active_loras": w.num_active_loras, "rank": w.rank,
                   "block_size": w.block_size, "add_inputs": 1, "parallelism": "replicas" if world > 1 else "single",
                   "l2_policy": "%d rotating input sets, %.0f MB in total, L2 %.0f MB" % (
                       res["NB"], res["footprint"] / 1e6, res["l2"] / 1e6),
                   "timing": ("median of %d timed regions of exactly %d align+fused steps each (CUDA graphs, CUDA "
                              "events on the launching stream, barrier and device synchronisation around each "
                              "region, max over ranks)" % (len(regions), args.steps)),
                   **ex_config(args)},
        "timed_regions": {"count": len(regions), "ms_min": min(regions), "ms_median": float(np.median(regions)),
                          "ms_max": max(regions)},
        "kernels": {"align_us": res["align_us"], "fused_us": res["fused_us"],
                    "align_launches_per_call": res["align_launches"],
                    "fused_gbs": res["achieved"], "fused_tflops": tflops,
                    "fused_frac_bf16_tensor": tflops / res["tc_peak"],
                    "align_gbs": (counts["align_bytes"] / (res["align_us"] * 1e-6) / 1e9
                                  if res["align_us"] else None)},
        "algorithmic": counts,
        "roofline": {"bound": "hbm", "kernel": res["kernel_name"], "achieved": res["achieved"], "peak": res["peak"],
                     "unit": "GB/s",
                     "frac": res["achieved"] / res["peak"], "peak_kind": res["peak_kind"] + " (hbm_gbs)",
                     "traffic": None if uses_ex(args) else NCU_TRAFFIC.get((w.name, res["kernel_name"])),
                     "traffic_unit": "bytes per launch (ncu)"},
        "configs": res["configs"],
        "configs_note": ("each configuration alone: fused_us / align_us (library's variant) / align_us_smem / "
                         "align_us_global per call and step_us per align+fused step, from CUDA graphs over "
                         "rotating input sets larger than 3x L2; frac_hbm = fused algorithmic bytes / fused_us / "
                         "measured HBM copy bandwidth (%.1f GB/s); frac_bf16_tensor = flops / fused_us / "
                         "measured bf16 burst (%.1f TFLOP/s, %s)" % (res["peak"], res["tc_peak"], res["tc_kind"])),
        "cpu_baseline": cpu,
        "cpu_baseline_threads": cpu_threads,
        "e2e": res["e2e"],
        "gpu_launches": args.steps * launches_per_step,
        "gpu_launches_note": "per timed region (%d launches per step)" % launches_per_step,
        "clocks": res["clocks"],
    }
    print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()

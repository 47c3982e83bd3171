"""The host-side oracle timings that bench.py reports beside the GPU numbers:
the single-threaded one and the one with each call's covered pairs spread over
host threads, whose first call must agree element for element with one
single-threaded call on the same pairs."""
import numpy as np
import pytest

import bench
from lora_moe_gb300 import inputs as gen


@pytest.fixture(scope="module")
def tiny():
    return gen.make_inputs(gen.WORKLOADS["tiny"])


def test_threaded_timing_runs_and_checks_itself(tiny):
    us, desc, nt = bench.time_oracle_threads(tiny, 0.2, 2, 3)
    assert us > 0 and nt == 3
    assert "split over 3 threads" in desc and "checked equal" in desc


def test_threaded_timing_general_call():
    w = gen.WORKLOADS["tiny"]
    ex = gen.make_ex_inputs(w, num_slices=2, x_per_pair=True, routed_weights=True)
    us, desc, nt = bench.time_oracle_threads(ex.base, 0.2, 2, 4, ex=ex)
    assert us > 0 and nt == 4


def test_thread_count_capped_by_covered_pairs(tiny):
    n_cov = len(bench._covered_pairs(tiny))
    _, _, nt = bench.time_oracle_threads(tiny, 0.0, 1, n_cov + 50)
    assert nt == n_cov


def test_covered_pairs_follow_the_mapping(tiny):
    w = tiny.w
    act = set(int(v) for v in tiny.lora_ids)
    want = [f for f in range(w.M * w.topk) if int(tiny.token_lora_mapping[f // w.topk]) in act]
    assert bench._covered_pairs(tiny).tolist() == want


def test_threaded_timing_catches_a_chunk_that_differs(tiny, monkeypatch):
    """A planted error in the oracle output of a short (chunked) call must stop
    the run rather than be timed."""
    real = bench._oracle_pairs
    full = len(bench._covered_pairs(tiny))

    def planted(inp, ex, sel, cols):
        out = real(inp, ex, sel, cols)
        if len(sel) < full:
            out = out.copy()
            out[0, 0] += 1.0
        return out

    monkeypatch.setattr(bench, "_oracle_pairs", planted)
    with pytest.raises(RuntimeError, match="differs"):
        bench.time_oracle_threads(tiny, 0.0, 1, 2)


def test_single_threaded_timing_counts_calls(tiny):
    us, desc, made = bench.time_oracle(tiny, 0, 4, calls=3)
    assert us > 0 and made == 3 and "3 calls" in desc


def test_oracle_pairs_match_full_definition(tiny):
    """The sampled call the timings use returns the full definition's rows."""
    import oracle
    w = tiny.w
    sel = bench._covered_pairs(tiny)[:5]
    got = bench._oracle_pairs(tiny, None, sel, np.arange(w.N, dtype=np.int32))
    ref = oracle.fused(tiny.x, tiny.lora_a, tiny.lora_b, tiny.y_in, tiny.topk_ids, tiny.token_lora_mapping,
                       tiny.lora_ids).reshape(w.M * w.topk, w.N)
    assert np.array_equal(got, ref[sel])


def test_json_line_carries_the_contract_keys(monkeypatch, capsys, tiny):
    """main() around a stand-in for the device run: one JSON line with every
    key the benchmark contract names, both host baselines included."""
    import json
    import sys
    counts = bench.algorithmic_counts(tiny)

    def fake_run(args, world, rank, local, pg):
        return dict(ms=2.0, clocks={"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": []}, fused_us=1.5,
                    align_us=0.5, counts=counts, NB=8, l2=126 << 20, footprint=400 << 20,
                    kernel_name="fused_cuda_core_kernel", align_launches=1,
                    e2e={"value": 3.0, "unit": "us/call", "h2d_bytes_per_step": 10, "d2h_bytes_per_step": 20},
                    achieved=100.0, peak=6794.8, peak_kind="measured", tc_peak=1895.3, tc_kind="measured",
                    regions=[2.2, 2.0, 1.9, 2.0, 2.1], inp=tiny, ex=None,
                    configs={"tiny": {"fused_us": 1.5, "align_us": 0.5, "step_us": 2.0}})

    monkeypatch.setattr(bench, "run_ours", fake_run)
    monkeypatch.setattr(bench, "time_oracle", lambda inp, b, n, ex=None, with_align=True: (5.0, "s1", 1))
    monkeypatch.setattr(bench, "time_oracle_threads",
                        lambda inp, b, n, t, ex=None, with_align=True: (2.0, "s2", 4))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "tiny", "--steps", "4", "--warmup", "3"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline",
              "cpu_baseline_threads", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3 and d["higher_is_better"] is False
    assert d["value"] == pytest.approx(2.0 * 1e3 / 4)
    assert d["config"]["workload"] == "tiny" and d["vs_baseline"] is None
    assert set(d["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert d["roofline"]["frac"] == pytest.approx(100.0 / 6794.8)
    assert d["cpu_baseline"] == {"value": 5.0, "unit": "us/call", "cores": 1, "kind": "oracle", "sample": "s1"}
    assert d["cpu_baseline_threads"]["cores"] == 4 and d["cpu_baseline_threads"]["value"] == 2.0
    assert d["gpu_launches"] == 4 * 2
    assert d["timed_regions"]["count"] == 5 and d["timed_regions"]["ms_median"] == 2.0
    assert d["configs"]["tiny"]["fused_us"] == 1.5


def test_default_workload_and_config_list():
    """The headline is the largest configuration; the per-config entries cover
    every configuration of the specification."""
    import sys
    assert bench.DEFAULT_WORKLOAD == "large_e_nact8"
    assert bench.CONFIG_WORKLOADS == ["tiny", "decode_qwen3_w13", "decode_gptoss_w2", "prefill_mixtral_w13",
                                      "large_e_nact1", "large_e_nact4", "large_e_nact8"]
    for name in bench.CONFIG_WORKLOADS:
        assert name in gen.WORKLOADS
    old = sys.argv
    try:
        sys.argv = ["bench.py"]
        a = bench.parse()
    finally:
        sys.argv = old
    assert a.workload == "large_e_nact8" and a.configs == "all" and a.min_regions >= 5
    # with no flags the run finishes in about a minute: 200 steps of the
    # 1.2 ms headline step per timed region, at least 3 warm-up steps
    assert a.gpus == 1 and 3 <= a.warmup <= 100 and 1 <= a.steps <= 1000


@pytest.mark.parametrize("v,name", [(0, None), (1, "smem (forced)"), (2, "global (forced)"), (3, "cluster (forced)")])
def test_forced_align_variant_is_named_in_the_config(monkeypatch, v, name):
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--align-variant", str(v)])
    cfg = bench.ex_config(bench.parse())
    assert cfg.get("align_variant") == name


def test_a_failing_threaded_baseline_does_not_lose_the_line(monkeypatch, capsys, tiny):
    import json
    import sys
    counts = bench.algorithmic_counts(tiny)

    def fake_run(args, world, rank, local, pg):
        return dict(ms=2.0, clocks={}, fused_us=1.5, align_us=0.5, counts=counts, NB=8, l2=1, footprint=1,
                    kernel_name="fused_cuda_core_kernel", align_launches=1, e2e=None, achieved=1.0, peak=2.0,
                    peak_kind="measured", tc_peak=3.0, tc_kind="measured", regions=[2.0] * 5, inp=tiny, ex=None,
                    configs={})

    def boom(*a, **k):
        raise RuntimeError("threaded oracle run differs from the single-threaded one")

    monkeypatch.setattr(bench, "run_ours", fake_run)
    monkeypatch.setattr(bench, "time_oracle", lambda inp, b, n, ex=None, with_align=True: (5.0, "s1", 1))
    monkeypatch.setattr(bench, "time_oracle_threads", boom)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "tiny", "--steps", "4", "--warmup", "3"])
    bench.main()
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert d["cpu_baseline"]["value"] == 5.0
    assert d["cpu_baseline_threads"]["value"] is None and "differs" in d["cpu_baseline_threads"]["error"]

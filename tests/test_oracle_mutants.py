"""Strength of the oracle's pins: plant plausible mistakes in a copy of the
oracle's C source, build it, and check that the pin suite rejects every one.

The mistakes are planted in a temporary copy on the CPU; the committed oracle
is never modified.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from oracle import oracle as oracle_impl

import test_oracle_pins as pins
import test_oracle_pins_ex as pins_ex

SRC = os.path.join(os.path.dirname(oracle_impl.__file__), "moe_lora_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("sentinel off by one", "const int sentinel = num_pairs;", "const int sentinel = num_pairs - 1;"),
    ("no block padding",
     "const int padded = (count[e] + block_size - 1) / block_size * block_size;",
     "const int padded = count[e];"),
    ("padding rounds down",
     "const int padded = (count[e] + block_size - 1) / block_size * block_size;",
     "const int padded = count[e] / block_size * block_size;"),
    ("scatter in descending order",
     "        for (int f = 0; f < num_pairs; ++f) {\n            const int m = f / topk;\n            if (token_lora_mapping[m] != l)\n                continue;\n            const int e = topk_ids[f];\n            if (e < 0 || e >= E)\n                continue;",
     "        for (int f = num_pairs - 1; f >= 0; --f) {\n            const int m = f / topk;\n            if (token_lora_mapping[m] != l)\n                continue;\n            const int e = topk_ids[f];\n            if (e < 0 || e >= E)\n                continue;"),
    ("token index from remainder", "static int pair_is_covered(int f, const int32_t *topk_ids, const int32_t *token_lora_mapping,\n                           const int32_t *lora_ids, const int32_t *adapter_enabled,\n                           int topk, int num_experts, int max_loras, int num_active_loras,\n                           int *l_out, int *e_out)\n{\n    const int m = f / topk;",
     "static int pair_is_covered(int f, const int32_t *topk_ids, const int32_t *token_lora_mapping,\n                           const int32_t *lora_ids, const int32_t *adapter_enabled,\n                           int topk, int num_experts, int max_loras, int num_active_loras,\n                           int *l_out, int *e_out)\n{\n    const int m = f % topk;"),
    ("A operand transposed", "s += bf16_value(x_row[kk]) * bf16_value(a_row[kk]);",
     "s += bf16_value(x_row[kk]) * bf16_value(a_le[(int64_t)kk * rank + j]);"),
    ("B operand transposed", "s += bf16_value(b_row[j]) * t[j];",
     "s += bf16_value(b_le[(int64_t)j * rank + n % rank]) * t[j];"),
    ("expand sign flipped", "s += bf16_value(b_row[j]) * t[j];", "s -= bf16_value(b_row[j]) * t[j];"),
    ("add_inputs ignored", "out[n] = (add_inputs ? bf16_value(yin[n]) : 0.0) + delta;",
     "out[n] = bf16_value(yin[n]) + delta;"),
    ("last rank column dropped", "for (int j = 0; j < rank; ++j)\n        s += bf16_value(b_row[j]) * t[j];",
     "for (int j = 0; j + 1 < rank; ++j)\n        s += bf16_value(b_row[j]) * t[j];"),
    ("adapter_enabled ignored", "    if (adapter_enabled && !adapter_enabled[l])\n        return 0;\n", ""),
    ("wrong expert stride", "lora_a + ((int64_t)l * num_experts + e) * rank * K;",
     "lora_a + ((int64_t)e * num_experts + l) * rank * K;"),
    # the general definition (router weights, rows per pair, slices, offset)
    ("router weight also scales y_in", "o[c] = (add_inputs ? bf16_value(yin[c]) : 0.0) + w * delta;",
     "o[c] = w * ((add_inputs ? bf16_value(yin[c]) : 0.0) + delta);"),
    ("router weight indexed by token", "(double)topk_weights[f]", "(double)topk_weights[m * topk]"),
    ("router weight ignored", "(double)topk_weights[f]", "1.0"),
    ("rows per pair ignored", "(x_per_pair ? f : m)", "(m)"),
    ("slice column stride dropped", "const int c = y_offset + s * N + n;", "const int c = y_offset + n;"),
    ("column offset ignored", "const int c = y_offset + s * N + n;", "const int c = s * N + n;"),
    ("first slice's A reused", "lora_a[s] + ", "lora_a[0] + "),
    ("first slice's B reused", "lora_b[s] + ", "lora_b[0] + "),
    ("unwritten columns cleared when overwriting", "            o[c] = bf16_value(yin[c]);",
     "            o[c] = add_inputs ? bf16_value(yin[c]) : 0.0;"),
]

PIN_TESTS = [
    pins.test_align_worked_example,
    pins.test_align_exhaustive_tiny_with_repeats,
    lambda: [pins.test_align_random_against_brute(s) for s in range(12)],
    pins.test_align_invariants_on_workloads,
    pins.test_align_single_lora_is_plain_moe_align,
    pins.test_fused_worked_example,
    pins.test_fused_matches_grouped_matmul,
    pins.test_fused_integer_case_exact,
    pins.test_fused_zero_b_gives_zero_delta,
    pins.test_fused_one_hot_adapters_copy_x,
    pins.test_fused_dense_special_case,
    pins.test_fused_uncovered_pairs_untouched_and_poison_unread,
    pins_ex.test_fused_ex_worked_example,
    pins_ex.test_fused_ex_per_pair_rows_as_tokens,
    pins_ex.test_fused_ex_slices_are_independent_column_blocks,
    pins_ex.test_fused_ex_router_weight_scales_the_delta_only,
    pins_ex.test_fused_ex_integer_case_exact,
]


def _build_mutant(src_text, tmpdir):
    c = os.path.join(tmpdir, "mutant.c")
    so = os.path.join(tmpdir, "libmutant.so")
    with open(c, "w") as fh:
        fh.write(src_text)
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                           "-w", "-o", so, c])
    return so


def _caught(so_path):
    lib = ctypes.CDLL(so_path)
    real = oracle_impl._load()
    for name in ("oracle_moe_lora_align", "oracle_moe_lora_fused", "oracle_moe_lora_fused_sampled",
                 "oracle_moe_lora_fused_ex"):
        fn = getattr(lib, name)
        ref = getattr(real, name)
        fn.argtypes, fn.restype = ref.argtypes, ref.restype
    saved = oracle_impl._lib
    oracle_impl._lib = lib
    try:
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                return True
        return False
    finally:
        oracle_impl._lib = saved


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    mutated = src.replace(old, new, 1)
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        assert _caught(_build_mutant(mutated, tmp)), "pins did not catch: " + name
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_unmutated_copy_passes():
    tmp = tempfile.mkdtemp(prefix="oracle_copy_")
    try:
        assert not _caught(_build_mutant(open(SRC).read(), tmp))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)

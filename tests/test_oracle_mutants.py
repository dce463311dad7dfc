"""Plausible mistakes planted in copies of the oracle (on the CPU) must each be
caught by at least one pin.  This shows the pins constrain every part of the
oracle: ordering, offsets, filtering, the row copy, the reduction and the
rounding.  Each mutant runs in a child process, because some planted mistakes
index out of bounds; a crash of the child also counts as caught."""
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")
TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

MUTANTS = {
    "unstable_order": ("for (int64_t r = 0; r < R; ++r) {\n        if (key[r] < 0) {",
                       "for (int64_t r = R - 1; r >= 0; --r) {\n        if (key[r] < 0) {"),
    "inclusive_offsets": ("cursor[e] = offsets[e];", "cursor[e] = offsets[e + 1] - (count[e] > 0);"),
    "row_from_p_not_r": ("(char *)permuted_hidden + p * row_bytes,\n                   (const char *)hidden + t * row_bytes",
                         "(char *)permuted_hidden + p * row_bytes,\n                   (const char *)hidden + (p / K) * row_bytes"),
    "map_minus_one_flagged": ("if (e == -1)\n        return -1;", ""),
    "tail_not_filled": ("permuted_idx[p] = -1;\n\n    free", "(void)p;\n\n    free"),
    "id_range_off_by_one": ("g >= (int64_t)E", "g > (int64_t)E"),
    "drop_last_k": ("for (int32_t k = 0; k < K; ++k) {\n                int32_t p = inv",
                    "for (int32_t k = 0; k < K - 1; ++k) {\n                int32_t p = inv"),
    "weight_transposed": ("float prod = w[t * K + k] * x;", "float prod = w[k * T + t] * x;"),
    "truncate_not_round": ("kept += 1u;", "kept += 0u;"),
    "ties_away_from_zero": ("(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    "subtract_term": ("acc = acc + prod;", "acc = acc - prod;"),
    "scale_row_wrong_token": ("permuted_scales + p * scale_cols, scales + t * scale_cols",
                              "permuted_scales + p * scale_cols, scales + (t / 2) * scale_cols"),
    "batched_row_wrong_token": ("(char *)batched_hidden + slot * row_bytes,\n                   (const char *)hidden + t * row_bytes",
                                "(char *)batched_hidden + slot * row_bytes,\n                   (const char *)hidden + (t ^ 1) * row_bytes"),
    "e4m3_ties_away": ("if (frac > 0.5 || (frac == 0.5 && ((long long)fl & 1)))",
                       "if (frac >= 0.5)"),
    "e4m3_truncate": ("double m8 = orc_round_half_even(t * 8.0);", "double m8 = (double)(long long)(t * 8.0);"),
    "e4m3_no_saturation": ("        return (uint8_t)(sign | 0x7e); /* saturate (also +-inf) */",
                           "        return (uint8_t)(sign | 0x7f); /* saturate (also +-inf) */"),
    "e4m3_subnormal_grid": ("double m = orc_round_half_even(a * 512.0);", "double m = orc_round_half_even(a * 256.0);"),
    "quant_wrong_max": ("float scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
                        "float scale = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    "batched_capacity_off_by_one": ("        if (j >= M) {\n            inv_permuted_idx[r] = -1;",
                                    "        if (j > M) {\n            inv_permuted_idx[r] = -1;"),
    "batched_slot_stride": ("int64_t slot = (int64_t)e * M + j;", "int64_t slot = (int64_t)e * (M - 1) + j;"),
    "batched_count_unclamped": ("expert_num_tokens[e] = (int32_t)(next[e] < M ? next[e] : M);",
                                "expert_num_tokens[e] = (int32_t)next[e];"),
    "inv_below_minus_one_not_flagged": ("if (inv[t * K + k] < -1 || inv[t * K + k] >= num_rows)",
                                        "if (inv[t * K + k] >= num_rows)"),
    "quant_zero_group_scale": ("float scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
                               "float scale = amax > 0.0f ? amax / 448.0f : 0.0f;"),
    "unpermute_k_descending": ("            for (int32_t k = 0; k < K; ++k) {\n                int32_t p = inv[t * K + k];",
                               "            for (int32_t k = K - 1; k >= 0; --k) {\n                int32_t p = inv[t * K + k];"),
    "unpermute_wide_accumulator": ("            float acc = 0.0f;", "            double acc = 0.0;"),
    "quant_code_times_reciprocal": ("orc_f32_to_e4m3_satfinite(orc_bf16_to_f32(xg[i]) / scale);",
                                    "orc_f32_to_e4m3_satfinite(orc_bf16_to_f32(xg[i]) * (1.0f / scale));"),
    "unpermute_fused_multiply_add": ("                float prod = w[t * K + k] * x;\n                acc = acc + prod;",
                                     "                acc = fmaf(w[t * K + k], x, acc);"),
}

CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
orc = oracle.OracleLib({so!r})
caught = []
for pin in pins.ALL_PINS:
    try:
        pin(orc)
    except AssertionError:
        caught.append(pin.__name__)
print("CAUGHT:" + ",".join(caught))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so"))
    code = CHILD.format(root=ROOT, tests=TESTS, so=so)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True,
                          text=True, timeout=300)
    if proc.returncode != 0:
        return  # the planted mistake crashed the child: caught
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("CAUGHT:")][-1]
    assert line != "CAUGHT:", f"no pin caught mutant {name}"

"""Planted mistakes in the oracle must turn its pins red (CPU only).

Each case copies ``oracle/tail_oracle.c`` into a temporary directory, applies
one plausible mistake as a textual edit, compiles it with gcc, points the
oracle wrappers at the mutant and runs the pins that should reject it.  A
mutant that passes them all means the pins are too weak.
"""
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_moe as moe
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tail_oracle.c")

# (name, original text, mutated text, pins that must catch it)
MUTANTS = [
    ("mean_over_H", "ss / (double)Hu", "ss / (double)H",
     [pins.test_rstd_divides_by_hidden_actual_not_H]),
    ("eps_dropped", "ss / (double)Hu + (double)eps", "ss / (double)Hu",
     [pins.test_rstd_eps_dominates_tiny_rows]),
    ("eps_outside_sqrt", "1.0 / sqrt(ss / (double)Hu + (double)eps)",
     "1.0 / sqrt(ss / (double)Hu) + (double)eps",
     [pins.test_logits_scale_relation_exact]),
    ("gamma_dropped", "* (double)gamma[h]", "",
     [pins.test_logits_one_hot_columns_exact]),
    ("rstd_dropped", "j->rstd[b] * acc", "acc",
     [pins.test_logits_one_hot_columns_exact]),
    ("w_transposed", "j->w + (int64_t)h * j->V + j->v0", "j->w + (int64_t)h + j->v0",
     [lambda: pins.test_logits_match_numpy_matmul("f32")]),
    ("pads_counted_when_ignored", "return zero_pad ? 1 : (h < Hu);", "return 1;",
     [pins.test_rstd_ignores_lanes_beyond_hidden_actual_when_not_zero_padded]),
    ("tie_index_desc", "return (a->i > b->i) - (a->i < b->i);",
     "return (a->i < b->i) - (a->i > b->i);",
     [pins.test_topk_matches_lexsort_brute_force]),
    ("draw_non_strict", "target < C", "target <= C",
     [lambda: _golden("equal_3col")]),
    ("top_p_strict", "if (cum >= top_p) {", "if (cum > top_p) {",
     [lambda: _golden("equal_p05")]),
    ("no_temperature", "exp((vals[i] - vals[0]) / temp)", "exp(vals[i] - vals[0])",
     [lambda: _golden("temp2_u076")]),
    ("three_col_default_draw", "ncols == 4 ? (double)p4[3] : 0.5", "ncols == 4 ? (double)p4[3] : 0.0",
     [lambda: _golden("equal_3col")]),
    ("top_k_off_by_one", "? (long)trunc(top_k) : (long)n;", "? (long)trunc(top_k) + 1 : (long)n;",
     [lambda: _golden("unif8_k4_u09")]),
    ("bf16_widen_wrong_shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15",
     [pins.test_widen_bf16_exhaustive]),
    ("f16_subnormal_scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)",
     [pins.test_widen_f16_exhaustive_against_numpy]),
    # the producer step (MoE combine + residual add)
    ("shared_slots_folded_into_the_routed_chain",
     "if (s < n_routed)\n                    r = fmaf(ws, y, r);\n                else\n                    sh = fmaf(ws, y, sh);",
     "r = fmaf(ws, y, r);",
     [lambda: _moe_golden("shared_apart"), lambda: _moe_golden("nemotron_8")]),
    ("shared_weight_ignored", "sh = fmaf(ws, y, sh);", "sh = sh + y;",
     [lambda: _moe_golden("shared_weighted")]),
    ("shared_sum_rounded_apart", "const float acc = r + sh;",
     "const float acc = r + bits_to_float(((uint32_t)oracle_f32_to_bf16_rne(sh)) << 16);",
     [lambda: _moe_golden("shared_unrounded")]),
    ("combine_not_rounded_before_add",
     "const float d = bits_to_float(((uint32_t)oracle_f32_to_bf16_rne(acc)) << 16);", "const float d = acc;",
     [lambda: _moe_golden("round_first")]),
    ("combine_slots_reversed", "for (int s = 0; s < S; ++s) {", "for (int s = S - 1; s >= 0; --s) {",
     [lambda: _moe_golden("slot_order")]),
    ("combine_slot_index_transposed", "((int64_t)b * S + s) * H + j", "((int64_t)s * B + b) * H + j",
     [lambda: moe.test_moe_combine_exact_sums_match_numpy("f32")]),
    ("bf16_truncates", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;", "",
     [moe.test_bf16_rounding_is_nearest_ties_to_even]),
    ("bf16_ties_away", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)",
     [moe.test_bf16_rounding_is_nearest_ties_to_even]),
]


def _moe_golden(name):
    for case in moe._golden_cases():
        if case[0] == name:
            return moe.test_moe_combine_hand_worked(case)
    raise KeyError(name)


def _golden(name):
    for case in pins._golden_cases():
        if case[0] == name:
            return pins.test_sampler_hand_worked(case)
    raise KeyError(name)


@pytest.mark.parametrize("mut", MUTANTS, ids=lambda m: m[0])
def test_mutant_is_rejected(mut, tmp_path):
    name, old, new, checks = mut
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so_path),
                           str(c_path), "-lpthread", "-lm"])
    oracle.use_library(str(so_path))
    try:
        caught = 0
        for chk in checks:
            try:
                chk()
            except AssertionError:
                caught += 1
        assert caught > 0, f"mutant {name} passed every pin meant to catch it"
    finally:
        oracle.use_library(None)

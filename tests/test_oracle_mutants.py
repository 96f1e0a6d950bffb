"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source, builds
that copy, and requires at least one pin to fail on it.  The mistakes cover the
pages' "common mistakes" (problem page "SiTU-GLU", section "Common mistakes to
avoid") and the usual slips of a hand-written FFN: a wrong sign, a dropped term,
a transposed operand, a swapped split, an unstable or misplaced index.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle as oracle_mod

PINS_SCRIPT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_pins.py")

MUTANTS = {
    "sigmoid_on_up_branch": ("return oracle_softcap(u, linear_beta);",
                             "return oracle_softcap(u, linear_beta) * oracle_sigmoid(u);"),
    "hard_clamp": ("return beta * tanh(x / beta);",
                   "return x > beta ? beta : (x < -beta ? -beta : x);"),
    "shared_cap": ("return oracle_gate_branch(g, beta) * oracle_up_branch(u, linear_beta);",
                   "return oracle_gate_branch(g, beta) * oracle_up_branch(u, beta);"),
    "swapped_caps": ("return oracle_gate_branch(g, beta) * oracle_up_branch(u, linear_beta);",
                     "return oracle_gate_branch(g, linear_beta) * oracle_up_branch(u, beta);"),
    "tanh_before_divide": ("return beta * tanh(x / beta);", "return beta * tanh(x) / beta;"),
    "cap_not_multiplied_back": ("return beta * tanh(x / beta);", "return tanh(x / beta);"),
    "multiply_before_nonlinearity": (
        "return oracle_gate_branch(g, beta) * oracle_up_branch(u, linear_beta);",
        "return oracle_up_branch(oracle_gate_branch(g * u, beta), linear_beta);"),
    "sigmoid_of_capped_gate": ("return oracle_softcap(g, beta) * oracle_sigmoid(g);",
                               "return oracle_softcap(g, beta) * oracle_sigmoid(oracle_softcap(g, beta));"),
    "sigmoid_sign": ("if (g >= 0.0) return 1.0 / (1.0 + exp(-g));",
                     "if (g >= 0.0) return 1.0 / (1.0 + exp(g));"),
    "sigmoid_negative_branch": ("return e / (1.0 + e);", "return 1.0 / (1.0 + e);"),
    "act_split_swapped": ("double g = oracle_load(gate_up, in_dt, r * 2 * I + j);\n      double u = oracle_load(gate_up, in_dt, r * 2 * I + I + j);",
                          "double u = oracle_load(gate_up, in_dt, r * 2 * I + j);\n      double g = oracle_load(gate_up, in_dt, r * 2 * I + I + j);"),
    "ffn_split_swapped": ("oracle_situ_pair(gu[j], gu[I + j], beta, linear_beta)",
                          "oracle_situ_pair(gu[I + j], gu[j], beta, linear_beta)"),
    "gate_up_transposed": ("oracle_load(w_gate_up, w_dt, n * M + k)",
                           "oracle_load(w_gate_up, w_dt, k * (2 * I) + n)"),
    "down_transposed": ("oracle_load(w_down, w_dt, m * I + j)", "oracle_load(w_down, w_dt, j * M + m)"),
    "dropped_first_term": ("for (int64_t k = 0; k < M; ++k) s +=", "for (int64_t k = 1; k < M; ++k) s +="),
    "dropped_last_down_term": ("for (int64_t j = 0; j < I; ++j) s +=", "for (int64_t j = 0; j + 1 < I; ++j) s +="),
    "unstable_index": ("for (int64_t i = 0; i < n; ++i) token_index[cursor[expert_ids[i]]++] = (int32_t)i;",
                       "for (int64_t i = n - 1; i >= 0; --i) token_index[cursor[expert_ids[i]]++] = (int32_t)i;"),
    "offsets_off_by_one": ("offsets[e + 1] += 1;", "offsets[e] += 1;"),
    "gather_sorted_position": ("int64_t t = flat / k_eff;", "int64_t t = r / k_eff;"),
    "scatter_sorted_position": ("y + flat * M);", "y + r * M);"),
    "bf16_decode_shift": ("((uint32_t)v) << 16", "((uint32_t)v) << 15"),
    "grad_missing_sigmoid_term": ("da = sg / (c * c) + beta * tanh(g / beta) * sg * sgm;",
                                  "da = sg / (c * c);"),
    "grad_sign_flip": ("da = sg / (c * c) + beta * tanh(g / beta) * sg * sgm;",
                       "da = sg / (c * c) - beta * tanh(g / beta) * sg * sgm;"),
    "grad_up_cap_swapped": ("const double c = cosh(u / linear_beta);",
                            "const double c = cosh(u / beta);"),
    "grad_products_swapped": ("*dh_dg = oracle_up_branch(u, linear_beta) * da;",
                              "*dh_dg = oracle_gate_branch(g, beta) * da;"),
    "bwd_dh_transposed": ("oracle_load(w_down, w_dt, m * I + j);\n      double pg",
                          "oracle_load(w_down, w_dt, j * M + m);\n      double pg"),
    "bwd_dw_down_wrong_operand": ("s += oracle_load(dy, dy_dt, r * M + m) * h[r * I + j];",
                                  "s += oracle_load(x, x_dt, r * M + m) * h[r * I + j];"),
    "grouped_bwd_wrong_expert_slab": (
        "const char* wd = (const char*)w_down + (size_t)e * (size_t)(M * I) * esz;",
        "const char* wd = (const char*)w_down;"),
    "grouped_bwd_dx_overwrites_slot": ("dx[t * M + k] += acc;", "dx[t * M + k] = acc;"),
    "grouped_bwd_dw_token_row": ("dwg_e[n * M + k] += dgu[n] * oracle_load(x, x_dt, t * M + k);",
                                "dwg_e[n * M + k] += dgu[n] * oracle_load(x, x_dt, k);"),
    "mx_scale_emax_7": ("int x = (e - 1) - 8;", "int x = (e - 1) - 7;"),
    "mx_scale_ceil": ("int x = (e - 1) - 8;", "int x = e - 8;"),
    "e4m3_truncates": ("const double r = nearbyint(a / ldexp(1.0, fl - 3)) * ldexp(1.0, fl - 3);",
                       "const double r = floor(a / ldexp(1.0, fl - 3)) * ldexp(1.0, fl - 3);"),
    "e4m3_no_clamp": ("if (r >= 448.0) return s | 0x7Eu; /* clamped", "if (r >= 1e300) return s | 0x7Eu; /* clamped"),
    "e4m3_subnormal_quantum": ("if (fl < -6) fl = -6;", "if (fl < -7) fl = -7;"),
    "e4m3_bias_8": ("return sign * ldexp(8.0 + m, e - 10);", "return sign * ldexp(8.0 + m, e - 11);"),
    "mx_block_scale_of_wrong_block": ("scales[r * (K / 32) + k / 32]", "scales[r * (K / 32) + k / 64]"),
    "bf16_round_truncates": ("r = nearbyint(a / q) * q;", "r = floor(a / q) * q;"),
    "e2m1_scale_emax_3": ("const uint32_t c = oracle_mx_scale_code_emax(amax, 2);",
                          "const uint32_t c = oracle_mx_scale_code_emax(amax, 3);"),
    "e2m1_nibbles_swapped": ("codes[(r * K + 32 * b + i) / 2] = (uint8_t)(lo | (hi << 4));",
                             "codes[(r * K + 32 * b + i) / 2] = (uint8_t)(hi | (lo << 4));"),
    "e2m1_truncates": ("const double r = nearbyint(a / q) * q;\n  if (r == 0.0) return s;\n  if (r >= 6.0)",
                       "const double r = floor(a / q) * q;\n  if (r == 0.0) return s;\n  if (r >= 6.0)"),
    "e2m1_decode_bias": ("return sign * ldexp(2.0 + m, e - 2);", "return sign * ldexp(2.0 + m, e - 1);"),
    "combine_wrong_weight": ("oracle_load(w, w_dt, t * k_eff + k) * y[(t * k_eff + k) * M + m]",
                             "oracle_load(w, w_dt, t * k_eff) * y[(t * k_eff + k) * M + m]"),
    "combine_dropped_slot": ("for (int32_t k = 0; k < k_eff; ++k)\n        s +=",
                             "for (int32_t k = 1; k < k_eff; ++k)\n        s +="),
}


def _run_pins(lib_path):
    """Run all pins on the build at lib_path in a child process.  Returns the list
    of failing pins, or ["<crashed: rc>"] if the child died before reporting."""
    proc = subprocess.run([sys.executable, PINS_SCRIPT, lib_path], capture_output=True,
                          text=True, timeout=300)
    for line in proc.stdout.splitlines():
        if line.startswith("PINS_FAILED "):
            return json.loads(line[len("PINS_FAILED "):])
    return [f"<crashed: rc={proc.returncode}>"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle_mod._SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    mutated = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib_path = oracle_mod.build(str(path), str(tmp_path / f"libmutant_{name}.so"))
    failed = _run_pins(lib_path)
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_unmutated_copy_passes(tmp_path):
    """Control: a verbatim copy built the same way passes every pin."""
    src = open(oracle_mod._SRC).read()
    path = tmp_path / "copy.c"
    path.write_text(src)
    lib_path = oracle_mod.build(str(path), str(tmp_path / "libcopy.so"))
    assert _run_pins(lib_path) == []

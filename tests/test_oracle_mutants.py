"""Plant a plausible mistake in a copy of the oracle, build it, and check that
the pins of ``test_oracle.py`` catch it.  All of this runs on the CPU."""
import os

import pytest

import oracle
import test_oracle as pins
import test_oracle_fp8 as pins8
import test_oracle_smooth as pins_sm
from w8a8_quantised_moe_gb300 import workloads as wl

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")

# (name, text in oracle.c, replacement, pins that must catch it)
MUTANTS = [
    ("round_half_away", "rintf(x[k] / s)", "roundf(x[k] / s)",
     [pins.test_quant_golden_4x4]),
    ("scale_over_128", "float s = amax / 127.0f;", "float s = amax / 128.0f;",
     [pins.test_quant_golden_4x4]),
    ("gemm_transposed_b", "(int64_t)b[n * K + kk]", "(int64_t)b[kk * N + n]",
     [lambda: pins.test_gemm_matches_numpy_int64(33, 64, 256)]),
    ("router_drops_bias", "if (bias) acc += (double)bias[e];", "",
     [lambda: [pins.test_router_golden(c) for c in pins._router_cases()]]),
    ("router_tie_to_higher", "logit[e] > logit[best]", "logit[e] >= logit[best]",
     [lambda: [pins.test_router_golden(c) for c in pins._router_cases()]]),
    ("silu_sign", "float d = 1.0f + expf(-g);", "float d = 1.0f + expf(g);",
     [pins.test_epilogue_gate_up_closed_form]),
    ("bf16_round_half_up", "u += 0x7fffu + lsb;", "u += 0x8000u;",
     [pins.test_bf16_rounding_matches_torch, pins.test_combine_golden]),
    ("slots_descending_tokens", "int32_t s = next[e]++;",
     "int32_t s = offsets[e + 1] - 1 - (next[e]++ - offsets[e]);",
     [lambda: pins.test_permute_matches_stable_argsort(37, 8, 2)]),
    ("combine_weights_reversed", "float term = topk_w[t * k + j] * o[(int64_t)slot_of[t * k + j] * H + c];",
     "float term = topk_w[t * k + (k - 1 - j)] * o[(int64_t)slot_of[t * k + j] * H + c];",
     [pins.test_combine_golden]),
    ("dequant_drops_weight_scale", "    v = v * s_act;\n    v = v * s_w;\n", "    v = v * s_act;\n",
     [pins.test_linear_golden_2x4]),
    ("moe_wrong_expert_w2", "oracle_gemm_s8(q_h + s0 * I, w2_q + e * H * I", "oracle_gemm_s8(q_h + s0 * I, w2_q",
     [lambda: pins.test_sparse_equals_brute_force_dense(wl.CONFIGS["tiny"])]),
    ("moe_wrong_slot_scale", "s_slot[s] = s_x[t];", "s_slot[s] = s_x[s % T];",
     [lambda: pins.test_sparse_equals_brute_force_dense(wl.CONFIGS["tiny"])]),
    # the FP8 (E4M3) layer
    ("fp8_scale_over_447", "float s = amax / 448.0f;", "float s = amax / 447.0f;",
     [pins8.test_quantize_rows_fp8_invariants]),
    ("fp8_ties_to_odd", "else c = (lo % 2 == 0) ? lo : hi;", "else c = (lo % 2 == 1) ? lo : hi;",
     [pins8.test_e4m3_golden_table, pins8.test_e4m3_encode_against_torch]),
    ("fp8_no_saturation", "if (a >= 448.0f) return (uint8_t)(sign | 0x7E);",
     "if (a >= 464.0f) return (uint8_t)(sign | 0x7F);", [pins8.test_e4m3_golden_table]),
    ("fp8_gemm_binary32_running_sum", "double sum = 0.0;", "float sum = 0.0f;",
     [pins8.test_gemm_fp8_cancellation, pins8.test_gemm_fp8_exact_against_integer_arithmetic]),
    ("fp8_subnormal_exponent", "if (e == 0) v = ldexpf((float)m, -9);", "if (e == 0) v = ldexpf((float)m, -10);",
     [pins8.test_e4m3_decode_every_code_against_torch]),
    ("fp8_moe_wrong_w13_expert", "oracle_gemm_fp8(q_slot + s0 * H, w13_q + e * 2 * I * H",
     "oracle_gemm_fp8(q_slot + s0 * H, w13_q",
     [lambda: pins8.test_moe_forward_fp8_equals_dense_brute_force(16, 256, 128, 8, 2)]),
    # SmoothQuant-folded activations
    ("smooth_multiplies_activation", "float r = 1.0f / sm[h];", "float r = sm[h];",
     [pins_sm.test_power_of_two_factors_leave_the_layer_unchanged, pins_sm.test_smoothing_worked_by_hand]),
    ("smooth_expert0_for_every_slot", "smooth + e * H, H, tmp,", "smooth, H, tmp,",
     [lambda: pins_sm.test_sparse_smoothed_layer_equals_dense_brute_force(16, 128, 64, 6, 2)]),
    ("smooth_fold_divides_weights", "row[k] = w[r * K + k] * s[k];", "row[k] = w[r * K + k] / s[k];",
     [pins_sm.test_quantize_rows_smoothed_unit_and_power_of_two_factors]),
    ("smooth_alpha_swapped", "pow(a, alpha) / pow(b, 1.0 - alpha)", "pow(a, 1.0 - alpha) / pow(b, alpha)",
     [pins_sm.test_smooth_factors_worked_by_hand]),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, source, name, old, new, checks):
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib = oracle.compile_source(str(src), str(tmp_path / f"lib{name}.so"))
    caught = []
    with oracle.using_library(lib):
        for check in checks:
            try:
                check()
            except (AssertionError, oracle.OracleError):
                caught.append(check)
    assert caught, f"no pin caught the planted mistake '{name}'"

"""Plant a plausible mistake in a copy of the oracle, build it, and check that
the pins of ``test_oracle.py`` catch it.  All of this runs on the CPU."""
import os

import pytest

import oracle
import test_oracle as pins
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
    ("dequant_drops_weight_scale", "    v = v * s_w;\n", "",
     [pins.test_linear_golden_2x4]),
    ("moe_wrong_expert_w2", "w2_q + e * H * I, n, H, I, acc2 + s0 * H", "w2_q, n, H, I, acc2 + s0 * H",
     [lambda: pins.test_sparse_equals_brute_force_dense(wl.CONFIGS["tiny"])]),
    ("moe_wrong_slot_scale", "s_slot[s] = s_x[t];", "s_slot[s] = s_x[s % T];",
     [lambda: pins.test_sparse_equals_brute_force_dense(wl.CONFIGS["tiny"])]),
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

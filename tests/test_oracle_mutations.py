"""The pins must catch a wrong oracle.

Each case plants one plausible slip in a temporary copy of the oracle's C
source (a dropped term, a swapped operand, a wrong index, an unstable sort, a
lost weight, an off-by-one exponent, a missing residual or shared expert, a
wrong FP8 activation scale, group, rounding or a skipped quantisation),
builds it with gcc, swaps it in and checks that at least one pin of
test_oracle_pins.py fails.  The committed oracle is never modified."""

import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTATIONS = {
    "silu dropped": ("return a / (1.0 + exp(-a));", "return a;"),
    "gate and up swapped": ("h[f] = oracle_silu(g[f]) * u[f];", "h[f] = oracle_silu(u[f]) * g[f];"),
    "scale block index transposed": ("m->s[(r / 128) * (m->cols / 128) + c / 128]",
                                     "m->s[(c / 128) * (m->rows / 128) + r / 128]"),
    "input index reversed": ("a += wq(&ex->gate, f, c) * x[c];", "a += wq(&ex->gate, f, c) * x[d - 1 - c];"),
    "router weight dropped": ("acc[c] += wt * o[c];", "acc[c] += o[c];"),
    "e4m3 bias off by one": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "rmsnorm eps dropped": ("sqrtf(variance + (float)eps)", "sqrtf(variance)"),
    "rmsnorm cast to bf16 dropped": ("float normed = bf16_round((float)oracle_bf16_value(h_bf16[c]) * inv);",
                                     "float normed = (float)oracle_bf16_value(h_bf16[c]) * inv;"),
    "sort ties reversed": ("    for (int64_t p = 0; p < R; ++p) {\n        int32_t e = ids[p];",
                           "    for (int64_t p = R - 1; p >= 0; --p) {\n        int32_t e = ids[p];"),
    "residual dropped": ("acc[c] += oracle_bf16_value(jb->resid[t * d + c]);", "(void)0;"),
    "shared expert dropped": ("            for (int64_t c = 0; c < d; ++c)\n                acc[c] += o[c];\n        }",
                              "        }"),
    "fp8 scale for a 240 maximum": ("float s = amax / 448.0f;", "float s = amax / 240.0f;"),
    "fp8 amax over the rest of the row": ("        for (int64_t i = 0; i < 128; ++i) {\n            float m",
                                          "        for (int64_t i = 0; i < n - g * 128; ++i) {\n            float m"),
    "fp8 ties to the odd code": ("(dist == best_dist && (c & 1) == 0)", "(dist == best_dist && (c & 1) == 1)"),
    "fp8 h not quantised": ("    if (fp8_act) {\n        oracle_fp8_dynamic(dff, h, g, NULL, NULL);\n        h = g;\n    }",
                            ""),
    "fp8 token row not quantised": ("        if (jb->fp8_act)\n            oracle_fp8_dynamic(d, xin, xin, NULL, NULL);",
                                    ""),
}

# the pins, with one parameter set each where they are parametrised
PINS = [
    (pins.test_e4m3_all_codes_match_torch, {}),
    (pins.test_e4m3_named_points, {}),
    (pins.test_dequant_matches_library_and_scale_layout, {}),
    (pins.test_silu_special_values_and_library, {}),
    (pins.test_expert_matches_fp64_matmul_with_library_silu, {}),
    (pins.test_expert_closed_form_with_permutation_weights, {}),
    (pins.test_rmsnorm_constant_rows_closed_form, {}),
    (pins.test_rmsnorm_invariants, {}),
    (pins.test_permute_matches_bincount_and_stable_argsort, dict(n=37, k=8, E=384, seed=2)),
    (pins.test_permute_ties_are_by_flat_index_and_skewed_counts, {}),
    (pins.test_oracle_matches_fp64_restatement_tiny, {}),
    (pins.test_single_expert_unit_weight_reduces_to_expert, {}),
    (pins.test_routed_sum_is_linear_in_router_weights_and_uses_each_slot, {}),
    (pins.test_layer_forward_matches_fp64_restatement, {}),
    (pins.test_layer_forward_zero_router_weights_no_shared_is_identity, {}),
    (pins.test_e4m3_encode_matches_torch_cast_and_saturates, {}),
    (pins.test_fp8_dynamic_group_invariants, {}),
    (pins.test_fp8_dynamic_groups_are_independent_and_scale_equivariant, {}),
    (pins.test_expert_fp8_act_matches_torch_restatement, {}),
    (pins.test_moe_infer_fp8_act_matches_torch_restatement_tiny, {}),
    (pins.test_layer_forward_fp8_act_quantises_the_normalised_row_and_shared_expert, {}),
]


def _build_mutant(old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    path_c = os.path.join(tmp, "mutant.c")
    path_so = os.path.join(tmp, "mutant.so")
    open(path_c, "w").write(src.replace(old, new, 1))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", path_c, "-o", path_so, "-lm"])
    return oracle._configure(ctypes.CDLL(path_so))


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_a_planted_mistake_fails_a_pin(name):
    old, new = MUTATIONS[name]
    with tempfile.TemporaryDirectory() as tmp:
        mutant = _build_mutant(old, new, tmp)
        saved = oracle.lib()
        oracle._lib = mutant
        caught = []
        try:
            for fn, kw in PINS:
                try:
                    fn(**kw)
                except AssertionError:
                    caught.append(fn.__name__)
        finally:
            oracle._lib = saved
    assert caught, f"no pin caught: {name}"

"""The oracle's pins are strong enough to catch plausible mistakes.

Each case below plants one plausible mistake in a private copy of the oracle's
C source (a dropped scale, an off-by-one mask, a transposed index, a wrong
rounding ...), compiles it into a temporary directory, swaps it in, and runs the
pin tests of ``test_oracle_pins.py``.  At least one pin must fail for every
mutant.  Everything runs on the CPU; the real oracle is restored afterwards.
"""
from __future__ import annotations

import subprocess

import pytest

import oracle
from oracle import build as oracle_build

from . import test_oracle_pins as pins

# (name, original text, planted mistake, which occurrence: 1 = first only, 0 = all)
MUTANTS = [
    ("decode_drops_scale", "s[p] = dot * inv_sqrt_d;", "s[p] = dot;", 1),
    ("decode_scale_by_d", "const double inv_sqrt_d = 1.0 / sqrt((double)D);",
     "const double inv_sqrt_d = 1.0 / (double)D;", 1),
    ("live_length_off_by_one", ": (int64_t)cp) + 1;", ": (int64_t)cp);", 1),
    ("decode_k_transposed", "const uint16_t *k = K + ((b * S + p) * H + h) * D;",
     "const uint16_t *k = K + ((b * H + h) * S + p) * D;", 1),
    ("decode_v_transposed", "const uint16_t *v = V + ((b * S + p) * H + h) * D;",
     "const uint16_t *v = V + ((b * H + h) * S + p) * D;", 1),
    ("decode_q_head_zero", "const uint16_t *q = Q + (b * H + h) * D;",
     "const uint16_t *q = Q + (b * H) * D;", 1),
    ("decode_no_normalisation", "const double w = s[p] / den;", "const double w = s[p];", 1),
    ("decode_no_max", "if (s[p] > M) M = s[p];", "", 1),
    ("decode_exp_sign", "s[p] = exp(s[p] - M);", "s[p] = exp(M - s[p]);", 1),
    ("f16_subnormal_exponent", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)", 1),
    ("f16_normal_bias", "ldexp((double)(1024 + frac), e - 25)",
     "ldexp((double)(1024 + frac), e - 24)", 1),
    ("f16_round_truncates", "double q = rint(a * ldexp(1.0, 10 - E));",
     "double q = floor(a * ldexp(1.0, 10 - E));", 1),
    ("qk_mask_ge", "if ((uint64_t)p > (uint64_t)current_pos[b]) {",
     "if ((uint64_t)p >= (uint64_t)current_pos[b]) {", 1),
    ("qk_pages_mask_ge", "if ((uint64_t)p > (uint64_t)current_pos[b]) score = -INFINITY;",
     "if ((uint64_t)p >= (uint64_t)current_pos[b]) score = -INFINITY;", 1),
    ("qk_pages_no_scale", "score = score * scale;", "", 1),
    ("pv_no_normalisation", "const double wp = w[p] / den;", "const double wp = w[p];", 1),
    ("pv_no_max", "if (s > M) M = s;", "", 1),
    ("paged_row_offset", "const uint16_t *k = K_pages + ((pg * page_size + p % page_size) * H + h) * D;",
     "const uint16_t *k = K_pages + ((pg * page_size + p / page_size) * H + h) * D;", 1),
    ("paged_v_page_of_k", "const uint16_t *v = V_pages + ((pg * page_size + p % page_size) * H + h) * D;",
     "const uint16_t *v = V_pages + ((pg + p % page_size) * H + h) * D;", 1),
    ("softmax_no_normalisation", "for (int64_t c = 0; c < cols; ++c) o[c] = has_nan ? NAN : o[c] / den;",
     "for (int64_t c = 0; c < cols; ++c) o[c] = has_nan ? NAN : o[c];", 1),
    ("rope_sin_sign", "o[i0] = u * cos(a) - w * sin(a);", "o[i0] = u * cos(a) + w * sin(a);", 1),
    ("rope_theta_exponent", "const double theta = pow(base, -2.0 * (double)i / (double)rope_dims);",
     "const double theta = pow(base, -1.0 * (double)i / (double)rope_dims);", 1),
    ("pv_v_transposed", "const uint16_t *v = V + ((b * S + p) * H + h) * D;\n"
     "                const double wp",
     "const uint16_t *v = V + ((b * H + h) * S + p) * D;\n                const double wp", 1),
]


def _pin_checks():
    cases = {c["name"]: c for c in pins._page_cases()["cases"]}
    return [
        ("f16_decode", pins.test_f16_decode_every_bit_pattern),
        ("f32_to_f16", pins.test_f32_to_f16_round_to_nearest_even),
        ("sdpa_48_35_8", lambda: pins.test_decode_matches_torch_sdpa_every_current_pos(48, 35, 8)),
        ("sdpa_8_7_3", lambda: pins.test_decode_matches_torch_sdpa_every_current_pos(8, 7, 3)),
        ("sdpa_large", pins.test_decode_matches_sdpa_large_scores),
        ("pv_softmax", pins.test_pv_matches_torch_softmax),
        ("single_live", pins.test_single_live_position_returns_v0_exactly),
        ("zero_query", pins.test_zero_query_gives_mean_of_live_v),
        ("two_live", pins.test_two_live_positions_sigmoid_exact_scores),
        ("mask_nan", lambda: pins.test_masked_positions_have_zero_weight("nan")),
        ("page_mask", lambda: pins.test_page_qk_inputs_exact_scores(cases["causal_mask"])),
        ("page_single_channel", pins.test_page_qk_single_channel_is_one_rounded_product),
        ("pv_closed", pins.test_pv_closed_forms),
        ("qk_square", pins.test_qk_f64_square_head_dims_exact),
        ("paged_identity", pins.test_paged_identity_table_equals_dense),
        ("softmax_torch", pins.test_softmax_matches_torch_fp64),
        ("rope_complex", lambda: pins.test_rope_equals_complex_rotation(False, 64)),
        ("paged_random", lambda: pins.test_paged_random_and_shared_tables_equal_dense_gather(5)),
    ]


@pytest.mark.parametrize("name,orig,mutated,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, mutated, count):
    src = open(oracle_build.SRC).read()
    assert orig in src, f"mutation target for {name} not found in the oracle source"
    mutant_src = src.replace(orig, mutated, count) if count else src.replace(orig, mutated)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(mutant_src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-shared",
                    "-fPIC", str(c_path), "-o", str(so_path), "-lm"], check=True)
    saved = oracle._LIB
    failed = []
    try:
        oracle._LIB = oracle._load(str(so_path))
        for label, check in _pin_checks():
            try:
                check()
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(label)
    finally:
        oracle._LIB = saved
    assert failed, f"no pin caught the planted mistake {name}"

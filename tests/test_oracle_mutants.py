"""The oracle's pins must catch plausible mistakes.

Each case compiles a copy of oracle.c with one planted mistake (a dropped term,
a wrong sign, a transposed index, a row/column mix-up, a wrong rounding rule)
into a temporary library, points the oracle wrapper at it, and checks that at
least one pin test fails.  Everything runs on the CPU.
"""
import os
import subprocess

import pytest

import oracle as O

import test_oracle as T
import test_oracle_pairs as TP

SRC = os.path.join(os.path.dirname(O.__file__), "oracle.c")

MUTANTS = {
    "drop_beta_term": ("v += p->beta * c;", "v += 0.0 * c;"),
    "c_relu_dropped": ("if (p->c_act == OR_ACT_RELU) c = (c > 0.0) ? c : 0.0;", ""),
    "negated_alpha": ("double v = p->alpha * acc;", "double v = -p->alpha * acc;"),
    "transposed_A_index": ("? i + k * lda : i * lda + k", "? k + i * lda : i * lda + k"),
    "transposed_B_index": ("? k + j * ldb : k * ldb + j", "? k + j * ldb : j * ldb + k"),
    "bias_indexed_by_row": ("if (p->bias_mode == OR_BIAS_COL) v += load_float(p->bias_dtype, p->bias, j);",
                            "if (p->bias_mode == OR_BIAS_COL) v += load_float(p->bias_dtype, p->bias, i);"),
    "relu_dropped": ("if (p->act == OR_ACT_RELU) v = (v > 0.0) ? v : 0.0;\n    return v;", "return v;"),
    "ties_round_up": ("(fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0", "fl + 1.0"),
    "int_beta_sign": ("v += beta * c;", "v -= beta * c;"),
    "k_loop_short_f16": ("for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) acc += f16_table",
                         "for (int64_t k = 1; k < p->K; ++k, ia += da, ib += db) acc += f16_table"),
    "k_loop_short_int": ("for (int64_t k = 0; k < p->K; ++k, ia += da, ib += db) acc += (int64_t)",
                         "for (int64_t k = 1; k < p->K; ++k, ia += da, ib += db) acc += (int64_t)"),
    "b_step_wrong": ("b_offset(p->layout_b, 1, j, p->ldb) - b0 : 0;\n    double acc",
                     "b_offset(p->layout_b, 1, j, p->ldb) - b0 + 1 : 0;\n    double acc"),
    "bf16_table_is_f16": ("acc += bf16_table[A[ia]] * bf16_table[B[ib]]",
                          "acc += f16_table[A[ia]] * bf16_table[B[ib]]"),
    # int8 requantising output
    "requant_in_fp64": ("const float prod = (float)v32 * (float)p->out_scale;    /* both roundings to nearest even, in fp32 */\n    float r = nearbyintf(prod);",
                        "const double prod = (double)v32 * p->out_scale;\n    float r = (float)nearbyint(prod);"),
    "requant_no_saturation": ("if (r > 127.0f) r = 127.0f;", ""),
    "requant_round_half_away": ("float r = nearbyintf(prod);                             /* ties", "float r = roundf(prod);                             /* ties"),
    "requant_scale_ignored": ("(float)v32 * (float)p->out_scale;", "(float)v32 * 1.0f;"),
    # transforms of A and B after load
    "transform_A_dropped": ("acc += transform_operand(p->ab_dtype, load_float(p->ab_dtype, p->A, ia), p->a_act, p->a_scale) *",
                            "acc += load_float(p->ab_dtype, p->A, ia) *"),
    "transform_B_takes_A_parameters": ("load_float(p->ab_dtype, p->B, ib), p->b_act, p->b_scale);",
                                       "load_float(p->ab_dtype, p->B, ib), p->a_act, p->a_scale);"),
    "transform_relu_before_scale": ("    double v = (double)((float)scale * (float)x);\n    if (act == OR_ACT_RELU) v = (v > 0.0) ? v : 0.0;",
                                    "    double v = (act == OR_ACT_RELU && x < 0.0) ? 0.0 : x;\n    v = (double)((float)scale * (float)v);"),
    "transform_scale_in_fp64": ("double v = (double)((float)scale * (float)x);", "double v = scale * x;"),
    "transform_not_rounded_to_f16": ("if (dtype == OR_F16) return oracle_f16_to_double(oracle_f16_from_double(v));",
                                     "if (dtype == OR_F16) return v;"),
    "transform_int8_relu_dropped": ("const int64_t b = (p->b_act == OR_ACT_RELU && B[ib] < 0) ? 0 : B[ib];",
                                    "const int64_t b = B[ib];"),
    # complex / dual-number GEMM
    "pair_unit_square_sign": ("re += a * c + u2 * (b * d);", "re += a * c - u2 * (b * d);"),
    "pair_dual_as_complex": ("unit == OR_UNIT_IMAGINARY ? -1.0 : 0.0;", "unit == OR_UNIT_IMAGINARY ? -1.0 : -1.0;"),
    "pair_cross_term_sign": ("im += a * d + b * c;", "im += a * d - b * c;"),
    "pair_imag_of_A_read_as_real": ("b = load_float(p->ab_dtype, p->A, 2 * ea + 1);",
                                    "b = load_float(p->ab_dtype, p->A, 2 * ea);"),
    "pair_conjugated_B": ("d = load_float(p->ab_dtype, p->B, 2 * eb + 1);",
                          "d = -load_float(p->ab_dtype, p->B, 2 * eb + 1);"),
    "pair_c_unit_part_ignored": ("p->C, 2 * (i * p->ldc + j) + part);", "p->C, 2 * (i * p->ldc + j));"),
    "pair_relu_dropped": ("if (p->act == OR_ACT_RELU) v = (v > 0.0) ? v : 0.0;\n        store_float",
                          "store_float"),
    "pair_bias_not_paired": ("v += load_float(p->bias_dtype, p->bias, 2 * j + part);",
                             "v += load_float(p->bias_dtype, p->bias, j + part);"),
}

PINS = [
    lambda: [T.test_hand_worked_examples(c, lay) for c in T._golden_cases() for lay in T.LAYOUTS],
    lambda: [T.test_small_integers_match_numpy_int_matmul(lay, ab, epi)
             for lay in T.LAYOUTS for ab in ["f16", "s8"]
             for epi in ["plain", "alpha_beta", "bias_col_relu", "bias_row_relu",
                         "relu_on_c_and_d"]],
    lambda: [T.test_identity_A_gives_op_B(lay, "f32") for lay in T.LAYOUTS],
    lambda: [T.test_f16_rounding_cases(x, b) for x, b in T.F16_CASES],
    lambda: [T.test_bf16_rounding_cases(x, b) for x, b in T.BF16_CASES],
    lambda: T.test_random_float_within_fp64_rounding_of_exact_sum(),
    lambda: T.test_requant_ties_round_to_even_and_saturate(),
    lambda: T.test_requant_product_is_taken_in_fp32(),
    lambda: T.test_requant_matches_numpy_closed_form(),
    lambda: [T.test_transform_relu_matches_numpy_on_small_integers(lay, ab, acts) for lay in T.LAYOUTS
             for ab in ["f16", "s8"] for acts in [("relu", "none"), ("none", "relu")]],
    lambda: [T.test_transform_takes_the_scale_in_fp32_then_rounds_to_the_operand_type(ab)
             for ab in ["f16", "bf16"]],
    lambda: [TP.test_hand_worked_pairs(c, lay) for c in TP._golden() for lay in TP.LAYOUTS],
    lambda: [TP.test_block_matrix_representation(u, lay) for u in ("complex", "dual")
             for lay in TP.LAYOUTS],
    lambda: [TP.test_complex_small_integers_match_numpy(lay, "f16") for lay in TP.LAYOUTS],
]


def _pins_fail() -> bool:
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mutated),
                    "-o", str(lib), "-lm"], check=True)
    saved = O._lib
    try:
        O._lib = None
        O._load_from(str(lib))
        assert _pins_fail(), f"no pin caught the planted mistake '{name}'"
    finally:
        O._lib = saved


def test_unmutated_oracle_passes_the_same_pins():
    assert not _pins_fail()

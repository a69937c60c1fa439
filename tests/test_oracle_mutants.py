"""The oracle's pins have teeth: plausible slips planted in the oracle fail them.

Each mutant is the oracle's own C source with one textual change, compiled
on the CPU into a temporary library and swapped in for the real one while a
fixed set of pin tests runs.  A mutant must make at least one pin fail.
"""

import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ref_gemm.c")

MUTANTS = {
    "float_accumulator": ("double sum = 0.0;", "float sum = 0.0f;"),
    "float_product": ("sum += (double)A[i * K + k] * (double)B[k * N + j];",
                      "sum += (double)(A[i * K + k] * B[k * N + j]);"),
    "drops_last_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    "skips_first_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    "a_reversed_in_k": ("(double)A[i * K + k]", "(double)A[i * K + (K - 1 - k)]"),
    "b_reversed_in_k": ("(double)B[k * N + j]", "(double)B[(K - 1 - k) * N + j]"),
    "truncating_conversion": ("return (float)sum;",
                              "float f = (float)sum; if ((double)f > sum && sum > 0) "
                              "f = __builtin_nextafterf(f, 0.0f); return f;"),
    "absolute_value_result": ("return (float)sum;", "return (float)(sum < 0 ? -sum : sum);"),
    # the general form's own loop and its alpha/beta step
    "ex_alpha_product_rounded_to_float": ("double r = alpha * sum;",
                                          "double r = (double)(float)(alpha * sum);"),
    "ex_beta_product_in_float": ("r += beta * (double)C[i * ldc + j];",
                                 "r += (double)((float)beta * C[i * ldc + j]);"),
    "ex_beta_applied_when_zero": ("if (beta != 0.0) r += beta", "r += beta"),
    "ex_float_accumulator": ("            double sum = 0.0;\n            for (int64_t k = 0; k < K; ++k) {",
                             "            float sum = 0.0f;\n            for (int64_t k = 0; k < K; ++k) {"),
    "ex_transa_indices_swapped": ("transa ? (double)A[k * lda + i] : (double)A[i * lda + k]",
                                  "transa ? (double)A[i * lda + k] : (double)A[k * lda + i]"),
    "ex_transb_indices_swapped": ("transb ? (double)B[j * ldb + k] : (double)B[k * ldb + j]",
                                  "transb ? (double)B[k * ldb + j] : (double)B[j * ldb + k]"),
    "ex_leading_dimension_ignored": ("(double)A[i * lda + k]", "(double)A[i * K + k]"),
    "ex_alpha_dropped": ("double r = alpha * sum;", "double r = sum;"),
}

PINS = [
    pins.test_one_by_one_is_rounded_product,
    lambda: pins.test_quantised_inputs_match_exact_integer_product((37, 29, 53)),
    lambda: pins.test_all_ones_gives_k((5, 7, 1000)),
    pins.test_identity_and_permutation_are_exact,
    lambda: pins.test_bruteforce_tiny_dyadic(7, 13, 17),
    pins.test_general_floats_agree_with_correctly_rounded_sum,
    pins.test_double_accumulation_survives_cancellation,
    lambda: pins.test_final_conversion_rounds_to_nearest_even([1.0, 2.0 ** -24, 2.0 ** -40]),
    pins.test_transpose_invariant_bitwise,
    pins.test_general_form_reduces_to_plain_product,
    pins.test_transposed_storage_gives_same_bits,
    pins.test_leading_dimensions_pick_the_right_submatrix,
    pins.test_alpha_beta_exact_on_dyadic_values,
    pins.test_alpha_beta_rounded_once_near_cancellation,
    pins.test_alpha_beta_general_values_within_one_ulp_of_exact,
    pins.test_beta_zero_never_reads_c,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} no longer in the oracle"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", str(mutated), "-o", str(lib)], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle._bind(str(lib)))
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"mutant {name} passed every pin"

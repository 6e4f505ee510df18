"""Run the oracle's pins against a deliberately broken build of the oracle.

Usage: python -m tests._mutant_runner <path-to-mutant.so>
Exit status 0 means every pin passed (the mutant survived); anything else
(an assertion, a crash) means the pins caught the planted mistake.
"""
import sys

import numpy as np

import oracle
from tests import _bits
from tests import test_oracle_gemm as g
from tests import test_oracle_exact as x
from tests import test_oracle_split as s
from tests import test_oracle_tc as tc


def run_pins():
    # split pins on a reduced stratified sample
    a = _bits.f32_patterns_stratified((0x00, 0x7F), 12)
    s._check_bf16x9(a)
    s._check_tf32(_bits.f32_patterns_stratified((0, 1023, 0x155), 13)[::7])
    s.test_bf16x9_split_golden()
    s.test_tf32x3_split_golden()
    # GEMM pins
    for tA, tB in g.TRANS:
        g.test_f64_gemm_against_exact_rationals(tA, tB)
        g.test_tf32x3_gemm_against_exact_rationals(tA, tB)
        g.test_one_hot_rows_select_exactly(tA, tB)
        for v in (oracle.BF16X9_FIVE_BANDS, oracle.BF16X9_ONE_ACCUMULATOR):
            g.test_bf16x9_gemm_against_exact_rationals(v, tA, tB)
    g.test_f64_gemm_small_integers_exact_golden()
    g.test_sgemm_f32_within_summation_bound()
    g.test_sgemm_f32_is_one_fused_chain_in_k_order()
    g.test_bf16x9_bands_hold_the_nine_products()
    g.test_tf32x3_terms_are_the_three_products()
    g.test_tf32x3_drops_lo_times_lo_closed_form()
    g.test_bf16x6_keeps_bands_0_to_2_closed_form()
    g.test_tf32x1_single_product_is_hi_times_hi()
    g.test_tf32x1_closed_form_and_bound()
    for tA, tB in g.TRANS:
        g.test_bf16x6_against_exact_rationals(tA, tB)
    g.test_alpha_beta_bias_placement()
    g.test_beta_zero_never_reads_c()
    g.test_k_zero_gives_beta_c_plus_bias()
    for seed in (0, 1, 2):
        g.test_bf16x9_meets_or_beats_native_fp32(seed)
    # tensor-core model pins
    tc.test_exact_sums_are_exact()
    tc.test_alignment_uses_the_unnormalised_product_exponent()
    tc.test_terms_are_truncated_toward_zero()
    tc.test_block_sum_rounds_toward_zero()
    tc.test_wide_alignment_to_nearest_is_the_correctly_rounded_sum()
    tc.test_two_alignment_bits_lose_only_below_the_window()
    for mode in ("bf16x9", "bf16x6", "tf32x3", "tf32x1"):
        tc.test_bf16_exact_inputs_reduce_to_one_block_chain(mode)
    for mode in ("bf16x9", "tf32x3"):
        tc.test_model_within_the_stated_error_bound(mode)
    tc.test_split_pieces_are_reduced_owner_first()
    tc.test_issue_order_is_smallest_band_first()
    tc.test_each_32_deep_stage_starts_from_zero_and_is_promoted_to_nearest()
    # exact-accumulation reference pins
    for tA, tB in x.TRANS:
        x.test_bf16x9_exact_sum_is_the_correctly_rounded_dot_product(tA, tB)
        x.test_tf32x3_exact_sum_closed_form(tA, tB)
    x.test_bf16x6_and_tf32x1_exact_sum_closed_forms()
    x.test_exact_cancellation_of_huge_terms()
    x.test_rounding_is_nearest_even_once()
    x.test_subnormal_and_overflowing_results()
    x.test_epilogue_and_row_sampling()
    x.test_sequential_fp32_accumulation_stays_near_the_exact_sum()


if __name__ == "__main__":
    with oracle.use_library(sys.argv[1]):
        run_pins()
    np.seterr(all="ignore")
    sys.exit(0)

"""Pins of the oracle's tensor-core accumulation model (no GPU).

The model ([TC models] "Methodology", "Results": blocks of 16 BF16 products
or 8 TF32 products, 2 extra alignment bits, truncation) is pinned here by
cases worked out by hand, each chosen so that one plausible mistake changes
the answer:
  - alignment on the exponent of the unnormalised product (e(a) + e(b)),
    not on the product's own exponent;
  - each term truncated toward zero below 2^(e_max - 25);
  - the block's sum rounded toward zero;
and by its limits: with many alignment bits and rounding to nearest a block
FMA is the correctly rounded exact sum, and the full model stays within the
BF16x9 error bound of the float64 GEMM.  (The GPU tests check it bit for bit
against the hardware.)
"""
import math

import numpy as np
import pytest

import oracle


def bfma(c, a, b, **kw):
    return oracle.tc_block_fma(c, np.array(a, np.float32), np.array(b, np.float32), **kw)


def test_exact_sums_are_exact():
    assert bfma(0.0, [1.0, 1.0, 1.0], [0.5, 0.25, 0.125]) == 0.875
    assert bfma(2.0, [3.0, -1.0], [4.0, 2.0]) == 12.0


def test_alignment_uses_the_unnormalised_product_exponent():
    # 1.5 * 1.5 = 2.25 has exponent 1, but e(1.5) + e(1.5) = 0 sets e_max = 0:
    # bits are kept down to 2^-25, so 2^-12 * 2^-13 = 2^-25 survives the
    # cancellation of the two large products.  (Aligning on the product's own
    # exponent would keep only down to 2^-24 and return 0.)
    assert bfma(0.0, [1.5, -1.5, 2.0 ** -12], [1.5, 1.5, 2.0 ** -13]) == 2.0 ** -25
    # the FP32 accumulator input is aligned on its own exponent
    assert bfma(2.0 ** -25, [1.5, -1.5], [1.5, 1.5]) == 2.0 ** -25


def test_terms_are_truncated_toward_zero():
    # -2^-26 lies below the last kept bit 2^-25: it is dropped (toward zero),
    # not floored to -2^-25
    assert bfma(0.0, [1.5, -1.5, -(2.0 ** -12)], [1.5, 1.5, 2.0 ** -14]) == 0.0
    assert bfma(0.0, [1.5, -1.5, -(2.0 ** -12)], [1.5, 1.5, 2.0 ** -13]) == -(2.0 ** -25)


def test_block_sum_rounds_toward_zero():
    # 1 + 3 * 2^-25: kept exactly (e_max = 0), then rounded to FP32 -- toward
    # zero gives 1, to nearest 1 + 2^-23
    a, b = [1.5 * 2.0 ** -12], [2.0 ** -12]
    assert bfma(1.0, a, b) == 1.0
    assert bfma(1.0, a, b, round_mode=oracle.TC_NEAREST) == 1.0 + 2.0 ** -23
    assert bfma(-1.0, [-x for x in a], b) == -1.0


def test_wide_alignment_to_nearest_is_the_correctly_rounded_sum():
    # terms within 2^20 of one another: 20 alignment bits keep every bit
    rng = np.random.default_rng(3)
    for _ in range(300):
        a = (rng.choice([-1, 1], 16) * rng.uniform(0.5, 2, 16) * 2.0 ** rng.integers(-3, 4, 16)).astype(np.float32)
        b = (rng.choice([-1, 1], 16) * rng.uniform(0.5, 2, 16)).astype(np.float32)
        a = (a.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)   # BF16 values
        b = (b.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        c = np.float32(rng.uniform(-4, 4))
        exact = math.fsum([float(c)] + [float(x) * float(y) for x, y in zip(a, b)])
        got = bfma(c, a, b, neab=20, round_mode=oracle.TC_NEAREST)
        assert got == float(np.float32(exact))


def test_two_alignment_bits_lose_only_below_the_window():
    # with every term inside the 25-bit window (no cancellation below it) the
    # block is exact before the final rounding toward zero
    rng = np.random.default_rng(4)
    for _ in range(200):
        a = (rng.uniform(1, 2, 16).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        b = (rng.uniform(1, 2, 16).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        exact = math.fsum(float(x) * float(y) for x, y in zip(a, b))
        got = bfma(0.0, a, b)
        f = float(np.float32(exact))
        want = f if abs(f) <= abs(exact) else float(np.nextafter(np.float32(f), np.float32(0)))
        assert got == want


@pytest.mark.parametrize("mode", ["bf16x9", "bf16x6", "tf32x3", "tf32x1"])
def test_bf16_exact_inputs_reduce_to_one_block_chain(mode):
    """With operands that need one component, only the hi*hi product is
    nonzero: the model of one 32-deep stage is the chain of block FMAs over
    the k-values, which this test spells out through the block FMA itself."""
    rng = np.random.default_rng(5)
    mask = 0xFFFF0000 if mode.startswith("bf16") else 0xFFFFE000
    A = (rng.standard_normal((4, 32)).astype(np.float32).view(np.uint32) & np.uint32(mask)).view(np.float32)
    B = (rng.standard_normal((32, 5)).astype(np.float32).view(np.uint32) & np.uint32(mask)).view(np.float32)
    C = oracle.gemm_tc(oracle.Problem(A, B), mode=mode)
    blk = oracle.TC_BLOCK[mode]
    for m in range(4):
        for n in range(5):
            t = 0.0
            for k0 in range(0, 32, blk):
                t = bfma(t, A[m, k0:k0 + blk], B[k0:k0 + blk, n])
            assert C[m, n] == np.float32(t)


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_model_within_the_stated_error_bound(mode):
    rng = np.random.default_rng(6)
    for (M, N, K) in [(5, 7, 64), (3, 4, 300), (2, 3, 1)]:
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        p = oracle.Problem(A, B)
        C = oracle.gemm_tc(p, mode=mode)
        err = oracle.normwise_error(C, oracle.gemm_f64(p), oracle.absdenom_f64(p))
        assert err <= oracle.normwise_bound(mode, K)


def test_split_pieces_are_reduced_owner_first():
    """pieces = S splits the k-stages; element (m, n) of a tile is owned by
    piece (4 e + c) mod S with e = 4 (n mod 256) // 128 + (m mod 128) // 32 and
    c = (n mod 128) // 32.  Spelled out here for column blocks that give
    different owners, against the one-piece model of each k-range."""
    rng = np.random.default_rng(8)
    K = 96                                   # three 32-deep stages
    A = rng.standard_normal((40, K)).astype(np.float32)
    B = rng.standard_normal((K, 160)).astype(np.float32)
    got = oracle.gemm_tc(oracle.Problem(A, B), pieces=3)
    parts = [oracle.gemm_tc(oracle.Problem(A[:, 32 * q:32 * q + 32], B[32 * q:32 * q + 32])) for q in range(3)]
    for m in (0, 33, 39):
        for n in (0, 40, 70, 100, 130, 159):
            e = 4 * ((n % 256) // 128) + (m % 128) // 32
            owner = (4 * e + (n % 128) // 32) % 3
            acc = parts[owner][m, n]
            for q in range(3):
                if q != owner:
                    acc = np.float32(acc + parts[q][m, n])
            assert got[m, n] == acc


def test_issue_order_is_smallest_band_first():
    """The products of a stage go into the accumulator smallest band first,
    the order this library reads into [Blog] Fig. 1's band accumulation
    (bands 4, 3, 2, 1, 0).  Worked by hand for a = b = 1 + 2^-8 + 2^-16,
    whose components in natural magnitude are 1, 2^-8 and 2^-16 (K = 1, so
    each product is one block FMA with the accumulator):
      smallest first, the accumulator holds 2^-32, then 2^-24 + 2^-32,
      2^-23 + 2^-32, then the band-2 products make 3 2^-16 + 2^-23 + 2^-32;
      adding 2^-8 (alignment exponent -8, FP32 result rounded toward zero)
      drops 2^-32; the second 2^-8 and finally 1 keep everything else:
      1 + 2^-7 + 3 2^-16 + 2^-23 (the correctly rounded a*b);
      largest first, the two band-3 products of 2^-24 arrive at an
      accumulator near 1 whose FP32 rounding toward zero drops each of them:
      1 + 2^-7 + 3 2^-16."""
    a = np.float32(1.0 + 2.0 ** -8 + 2.0 ** -16)
    C = oracle.gemm_tc(oracle.Problem(np.array([[a]]), np.array([[a]])), mode="bf16x9")
    assert C[0, 0] == np.float32(1.0 + 2.0 ** -7 + 3 * 2.0 ** -16 + 2.0 ** -23)
    assert C[0, 0] != np.float32(1.0 + 2.0 ** -7 + 3 * 2.0 ** -16)


def test_each_32_deep_stage_starts_from_zero_and_is_promoted_to_nearest():
    """Stages of 32 k-values, each summed from zero and added into the FP32
    result with rounding to nearest.  Worked by hand for K = 64, operands
    exact in BF16 (one component each): a_0 b_0 = 1 and three products
    2^-12 2^-13 = 2^-25 at k = 32, 33, 34 (all other products zero).  Stage
    one gives 1; stage two sums its three products exactly to 3 2^-25, and
    1 + 3 2^-25 rounded to nearest is 1 + 2^-23.  (One 64-deep stage would
    add the 2^-25 products to an accumulator holding 1: kept within the
    2-bit alignment window, 1 + 3 2^-25, then rounded toward zero to 1.)"""
    A = np.zeros((1, 64), np.float32)
    B = np.zeros((64, 1), np.float32)
    A[0, 0] = B[0, 0] = 1.0
    A[0, 32:35] = 2.0 ** -12
    B[32:35, 0] = 2.0 ** -13
    C = oracle.gemm_tc(oracle.Problem(A, B), mode="bf16x9")
    assert C[0, 0] == np.float32(1.0 + 2.0 ** -23)

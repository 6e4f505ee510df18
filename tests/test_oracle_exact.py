"""Pins of the oracle's exact-accumulation reference, gemm_exact (no GPU).

gemm_exact sums the method's selected component products over k with no
rounding and rounds the sum once to FP32 ("Unlocking Tensor Core performance
for machine-learning interatomic potentials", "How Tensor Core FP32 bridges
the hardware gap": Fig. 1 for BF16x9's nine products, Eq. 1 for TF32x3's
three).  Each pin below comes from outside the function:
  - closed forms of the products' sum in exact rational arithmetic: BF16x9's
    split is exact, so its nine products add up to a*b and the reference is
    the correctly rounded dot product; TF32x3's three products are
    (hi + lo)(hi' + lo') - lo lo'; BF16x6 drops bands 3-4; one-pass TF32
    keeps hi hi -- each from the pinned splits;
  - hand-made sums whose rounding is fixed by IEEE round-to-nearest-even:
    exact cancellation of huge terms, ties, a tie broken by a far-away bit,
    subnormal results and overflow;
  - the FP32 epilogue on exact inputs, and row sampling.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _bits

TRANS = [(False, False), (True, False), (False, True), (True, True)]


def f32_nearest(q: Fraction) -> np.float32:
    """The FP32 number nearest the rational q, ties to even (gradual
    underflow; beyond the largest finite value it rounds to infinity)."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    e = max(e, -126)                       # below 2^-126 the spacing stays 2^-149
    ulp = Fraction(2) ** (e - 23)
    n = q / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * ulp
    if v >= Fraction(2) ** 128 - Fraction(2) ** 103:   # halfway to the next binade and above: infinity
        return np.float32(sign * np.inf)
    return np.float32(sign * float(v))


def _layout(A_op, B_op, tA, tB):
    A = np.ascontiguousarray(A_op.T) if tA else A_op
    B = np.ascontiguousarray(B_op.T) if tB else B_op
    return A, B


def _fr(x):
    return Fraction(float(x))


@pytest.mark.parametrize("tA,tB", TRANS)
def test_bf16x9_exact_sum_is_the_correctly_rounded_dot_product(tA, tB):
    """The BF16x9 split reconstructs every finite FP32 value exactly, so the
    nine scaled products of a pair add up to a*b: with exact accumulation the
    emulated result is the correctly rounded exact dot product."""
    rng = np.random.default_rng(31)
    for (M, N, K) in [(3, 4, 1), (4, 5, 9), (2, 3, 40)]:
        A_op = _bits.random_bits_matrix(rng, (M, K), -40, 40)
        B_op = _bits.random_bits_matrix(rng, (K, N), -40, 40)
        A, B = _layout(A_op, B_op, tA, tB)
        C = oracle.gemm_exact(oracle.Problem(A, B, transA=tA, transB=tB), "bf16x9")
        ex = _bits.exact_gemm(A_op, B_op)
        for m in range(M):
            for n in range(N):
                assert C[m, n] == f32_nearest(ex[m][n]), (m, n)


@pytest.mark.parametrize("tA,tB", TRANS)
def test_tf32x3_exact_sum_closed_form(tA, tB):
    """hi hi' + hi lo' + lo hi' = (hi + lo)(hi' + lo') - lo lo' (Eq. 1 with
    the residual product dropped), from the pinned TF32x3 split."""
    rng = np.random.default_rng(32)
    for (M, N, K) in [(3, 2, 1), (2, 4, 17)]:
        A_op = _bits.random_bits_matrix(rng, (M, K), -30, 30)
        B_op = _bits.random_bits_matrix(rng, (K, N), -30, 30)
        A, B = _layout(A_op, B_op, tA, tB)
        C = oracle.gemm_exact(oracle.Problem(A, B, transA=tA, transB=tB), "tf32x3")
        ah, al = (x.reshape(M, K) for x in oracle.split_tf32x3(A_op))
        bh, bl = (x.reshape(K, N) for x in oracle.split_tf32x3(B_op))
        for m in range(M):
            for n in range(N):
                s = sum(((_fr(ah[m, k]) + _fr(al[m, k])) * (_fr(bh[k, n]) + _fr(bl[k, n]))
                         - _fr(al[m, k]) * _fr(bl[k, n]) for k in range(K)), Fraction(0))
                assert C[m, n] == f32_nearest(s), (m, n)


def test_bf16x6_and_tf32x1_exact_sum_closed_forms():
    """BF16x6 = a b minus the band-3 and band-4 products (s1 t2 + s2 t1 +
    s2 t2 in natural magnitude); one-pass TF32 = hi hi'."""
    rng = np.random.default_rng(33)
    M, N, K = 3, 4, 11
    A = _bits.random_bits_matrix(rng, (M, K), -20, 20)
    B = _bits.random_bits_matrix(rng, (K, N), -20, 20)
    p = oracle.Problem(A, B)
    C6 = oracle.gemm_exact(p, "bf16x6")
    C1 = oracle.gemm_exact(p, "tf32x1")
    sa = [x.reshape(M, K) for x in oracle.split_bf16x9_f32(A)]
    sb = [x.reshape(K, N) for x in oracle.split_bf16x9_f32(B)]
    ah, _ = (x.reshape(M, K) for x in oracle.split_tf32x3(A))
    bh, _ = (x.reshape(K, N) for x in oracle.split_tf32x3(B))
    for m in range(M):
        for n in range(N):
            s6 = Fraction(0)
            s1 = Fraction(0)
            for k in range(K):
                a = [_fr(sa[i][m, k]) / 256 ** i for i in range(3)]
                b = [_fr(sb[j][k, n]) / 256 ** j for j in range(3)]
                s6 += _fr(A[m, k]) * _fr(B[k, n]) - (a[1] * b[2] + a[2] * b[1] + a[2] * b[2])
                s1 += _fr(ah[m, k]) * _fr(bh[k, n])
            assert C6[m, n] == f32_nearest(s6)
            assert C1[m, n] == f32_nearest(s1)


def _dot(a, b, mode="bf16x9"):
    A = np.array([a], np.float32)
    B = np.array(b, np.float32).reshape(-1, 1)
    return float(oracle.gemm_exact(oracle.Problem(A, B), mode)[0, 0])


def test_exact_cancellation_of_huge_terms():
    # 2^100 + 2^-100 - 2^100: a sequential FP32 sum loses the middle term
    assert _dot([2.0 ** 50, 2.0 ** -50, -(2.0 ** 50)], [2.0 ** 50, 2.0 ** -50, 2.0 ** 50]) == 2.0 ** -100
    # the far ends of the FP32 range in one sum: FLT_MAX^2 - FLT_MAX^2 + tiny
    fm = float(np.finfo(np.float32).max)
    assert _dot([fm, -fm, 2.0 ** -149], [fm, fm, 2.0 ** 0]) == 2.0 ** -149


def test_rounding_is_nearest_even_once():
    # 1 + 2^-24 is halfway between 1 and 1 + 2^-23: ties to even give 1
    assert _dot([1.0, 2.0 ** -12], [1.0, 2.0 ** -12]) == 1.0
    # 1 + 3 2^-24: halfway between 1 + 2^-23 and 1 + 2^-22, even is 1 + 2^-22
    assert _dot([1.0, 2.0 ** -12, 2.0 ** -12], [1.0, 2.0 ** -12, 2.0 ** -11]) == 1.0 + 2.0 ** -22
    # a bit far below the tie breaks it upward: 1 + 2^-24 + 2^-80
    assert _dot([1.0, 2.0 ** -12, 2.0 ** -40], [1.0, 2.0 ** -12, 2.0 ** -40]) == 1.0 + 2.0 ** -23
    # and downward when negative: 1 + 2^-24 - 2^-80 rounds to 1
    assert _dot([1.0, 2.0 ** -12, -(2.0 ** -40)], [1.0, 2.0 ** -12, 2.0 ** -40]) == 1.0
    # negative results round symmetrically
    assert _dot([-1.0, -(2.0 ** -12), -(2.0 ** -40)], [1.0, 2.0 ** -12, 2.0 ** -40]) == -(1.0 + 2.0 ** -23)


def test_subnormal_and_overflowing_results():
    # 2^-75 * 2^-75 = 2^-150: halfway between 0 and the smallest subnormal -> 0 (even);
    # a second such product makes 2^-149 exactly
    assert _dot([2.0 ** -75], [2.0 ** -75]) == 0.0
    assert _dot([2.0 ** -75, 2.0 ** -75], [2.0 ** -75, 2.0 ** -75]) == 2.0 ** -149
    # 3 2^-151 = 0.75 of the smallest subnormal -> rounds up to it
    assert _dot([2.0 ** -75, 2.0 ** -76], [2.0 ** -75, 2.0 ** -75]) == 2.0 ** -149
    # sums beyond FLT_MAX round to infinity
    fm = float(np.finfo(np.float32).max)
    assert _dot([fm, fm], [1.0, 1.0]) == np.inf
    assert _dot([fm, fm], [-1.0, -1.0]) == -np.inf


def test_epilogue_and_row_sampling():
    rng = np.random.default_rng(34)
    A = rng.integers(-8, 9, (6, 5)).astype(np.float32)
    B = rng.integers(-8, 9, (5, 7)).astype(np.float32)
    Cold = rng.integers(-8, 9, (6, 7)).astype(np.float32)
    bias = rng.integers(-8, 9, 7).astype(np.float32)
    p = oracle.Problem(A, B, alpha=2.0, beta=-1.0, C_old=Cold, bias=bias)
    want = 2.0 * (A.astype(np.float64) @ B) - Cold + bias        # small integers: exact
    for mode in ("bf16x9", "tf32x3", "bf16x6", "tf32x1"):
        C = oracle.gemm_exact(p, mode)
        assert np.array_equal(C, want.astype(np.float32))
        rows = np.array([5, 0, 3])
        assert np.array_equal(oracle.gemm_exact(p, mode, rows), C[rows])
    # beta = 0 never reads C_old
    Cnan = np.full((6, 7), np.nan, np.float32)
    C0 = oracle.gemm_exact(oracle.Problem(A, B, beta=0.0, C_old=Cnan), "bf16x9")
    assert np.array_equal(C0, (A.astype(np.float64) @ B).astype(np.float32))


def test_sequential_fp32_accumulation_stays_near_the_exact_sum():
    """The oracle's own FP32 accumulations of the same products differ from
    the exact-accumulation reference only by accumulation error: within the
    classical bound of a sequential sum, gamma_n sum |terms| (n terms per
    output: 9K for BF16x9's per-band sums and their recombination, 3K for
    TF32x3), checked on random data."""
    rng = np.random.default_rng(35)
    M, N, K = 4, 5, 300
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    p = oracle.Problem(A, B)
    D = oracle.absdenom_f64(p)
    for mode, nterms in (("bf16x9", 9 * K + 5), ("tf32x3", 3 * K)):
        Cx = oracle.gemm_exact(p, mode).astype(np.float64)
        Ce = oracle.gemm_emulated(p, mode).astype(np.float64)
        u = 2.0 ** -24
        gamma = nterms * u / (1 - nterms * u)
        # |C_emu - C_exact| <= gamma |products| + the two final roundings
        assert np.all(np.abs(Ce - Cx) <= gamma * D * 1.01 + 2 * u * np.abs(Cx))

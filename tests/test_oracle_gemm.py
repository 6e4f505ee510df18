"""Pins for the oracle's GEMMs (no GPU).

Each pin comes from outside the oracle: exact rational arithmetic on tiny
problems (brute force), closed forms (one-hot and identity operands, integer
data), the classical error bounds of floating-point summation, and the blog's
accuracy statement that BF16x9 meets or beats native FP32 against an FP64
reference ("Unlocking Tensor Core performance for machine-learning
interatomic potentials", "Limitations and decision criteria").  The method
itself: "How Tensor Core FP32 bridges the hardware gap", Fig. 1 (BF16x9: nine
products on five anti-diagonal bands), Fig. 2 and Eq. 1 (TF32x3: hi*hi +
hi*lo + lo*hi, lo*lo dropped).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _bits

U = 2.0 ** -24
TRANS = [(False, False), (True, False), (False, True), (True, True)]


def _layout(A_op, B_op, tA, tB):
    """Store op(A), op(B) in the transposed-or-not layout the call names."""
    A = np.ascontiguousarray(A_op.T) if tA else A_op
    B = np.ascontiguousarray(B_op.T) if tB else B_op
    return A, B


def _rel_err_vs_exact(C, exact, absden):
    worst = 0.0
    for m in range(len(exact)):
        for n in range(len(exact[0])):
            d = absden[m][n]
            e = abs(Fraction(float(C[m][n])) - exact[m][n])
            if d == 0:
                assert e == 0
                continue
            worst = max(worst, float(e / d))
    return worst


# ------------------------------------------------------------- float64 ------
@pytest.mark.parametrize("tA,tB", TRANS)
def test_f64_gemm_against_exact_rationals(tA, tB):
    rng = np.random.default_rng(11)
    for (M, N, K) in [(3, 4, 1), (5, 3, 7), (4, 6, 33)]:
        A_op = _bits.random_bits_matrix(rng, (M, K), -40, 40)
        B_op = _bits.random_bits_matrix(rng, (K, N), -40, 40)
        A, B = _layout(A_op, B_op, tA, tB)
        C64 = oracle.gemm_f64(oracle.Problem(A, B, transA=tA, transB=tB))
        ex = _bits.exact_gemm(A_op, B_op)
        den = _bits.exact_absgemm(A_op, B_op)
        # sequential binary64 summation: |error| <= (K-1) 2^-53 sum|a b| (+ higher order)
        assert _rel_err_vs_exact(C64, ex, den) <= max(K - 1, 1) * 2.0 ** -53 * 1.0001
        # the normwise denominator is the exact |A||B| up to binary64 rounding
        D = oracle.absdenom_f64(oracle.Problem(A, B, transA=tA, transB=tB))
        for m in range(M):
            for n in range(N):
                assert abs(Fraction(float(D[m, n])) - den[m][n]) <= den[m][n] * K * 2.0 ** -52


def test_f64_gemm_small_integers_exact_golden():
    """Golden integer example (tests/golden/gemm_integer_example.txt)."""
    A, B, bias, Cold, want = _integer_golden()
    p = oracle.Problem(A, B, alpha=2.0, beta=-1.0, C_old=Cold, bias=bias)
    assert np.array_equal(oracle.gemm_f64(p), want.astype(np.float64))
    for C in (oracle.sgemm_f32(p), oracle.gemm_bf16x9(p), oracle.gemm_tf32x3(p),
              oracle.gemm_bf16x9(p, variant=oracle.BF16X9_ONE_ACCUMULATOR)):
        assert np.array_equal(C, want)


# ---------------------------------------------------------- FP32 SGEMM ------
def test_sgemm_f32_within_summation_bound():
    rng = np.random.default_rng(12)
    for K in (1, 2, 17, 64):
        A = _bits.random_bits_matrix(rng, (4, K), -10, 10)
        B = _bits.random_bits_matrix(rng, (K, 5), -10, 10)
        C = oracle.sgemm_f32(oracle.Problem(A, B))
        gamma = K * U / (1 - K * U)
        err = _rel_err_vs_exact(C, _bits.exact_gemm(A, B), _bits.exact_absgemm(A, B))
        assert err <= gamma
        if K == 1:  # one product, rounded once
            assert np.array_equal(C, (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32))


def test_sgemm_f32_is_one_fused_chain_in_k_order():
    """Native FP32 is defined as acc = fmaf(a_k, b_k, acc) for k = 0, 1, ...
    from +0.  Row 0: 2^24 + 1 rounds back to 2^24 (tie to even) before
    -2^24 arrives, so the ascending chain gives 0 (descending would give 1).
    Row 1: (1 + 2^-12)^2 - (1 + 2^-11) = 2^-24 survives only when the
    multiply is fused into the add."""
    A = np.array([[2.0 ** 24, 1.0, -2.0 ** 24], [-(1 + 2.0 ** -11), 1 + 2.0 ** -12, 0.0]], np.float32)
    B = np.array([[1.0, 1.0], [1.0, 1 + 2.0 ** -12], [1.0, 0.0]], np.float32)
    C = oracle.sgemm_f32(oracle.Problem(A, B))
    assert C[0, 0] == 0.0
    assert C[1, 1] == 2.0 ** -24
    # epilogue: fmaf(alpha, acc, beta * C_old) + bias, one rounding for alpha acc + beta C_old
    acc = np.float32(1 + 2.0 ** -12)
    Cold = np.array([[-(1 + 2.0 ** -11)]], np.float32)
    p = oracle.Problem(np.array([[acc]], np.float32), np.array([[1.0]], np.float32), alpha=float(acc), beta=1.0,
                       C_old=Cold, bias=np.array([0.5], np.float32))
    assert oracle.sgemm_f32(p)[0, 0] == np.float32(2.0 ** -24 + 0.5)


# -------------------------------------------------------------- BF16x9 ------
def _band_exact(a, b):
    """Exact band sums from the (separately pinned) split: T_b = sum over
    i+j=b of c_i(a) c_j(b), so that a b = sum_b 2^-8b T_b."""
    ca = oracle.split_bf16x9_f32(np.array([a], np.float32))
    cb = oracle.split_bf16x9_f32(np.array([b], np.float32))
    T = [Fraction(0)] * 5
    for i in range(3):
        for j in range(3):
            T[i + j] += Fraction(float(ca[i][0])) * Fraction(float(cb[j][0]))
    return T


def test_bf16x9_bands_hold_the_nine_products():
    """K = 1: the five band sums carry exactly the nine products, each on
    band i + j; their scaled sum is a b with no error (the split is exact)."""
    rng = np.random.default_rng(13)
    A = _bits.random_bits_matrix(rng, (6, 1), -20, 20)
    B = _bits.random_bits_matrix(rng, (1, 7), -20, 20)
    _, bands = oracle.gemm_bf16x9(oracle.Problem(A, B), with_bands=True)
    for m in range(6):
        for n in range(7):
            T = _band_exact(A[m, 0], B[0, n])
            assert sum(T[b] * Fraction(2) ** (-8 * b) for b in range(5)) == \
                Fraction(float(A[m, 0])) * Fraction(float(B[0, n]))
            Tabs = _band_exact(abs(A[m, 0]), abs(B[0, n]))
            for b in range(5):
                got = Fraction(float(bands[b, m, n]))
                # at most two FP32 roundings of the band's (up to three) products
                assert abs(got - T[b]) <= Tabs[b] * 2 * U, (m, n, b)
                if Tabs[b] == 0:
                    assert got == 0
            # each scaled band lies below the top of its band: |T_b| < 2^(Ea+Eb+2)
            ea = _bits.binade_exponent(np.array([A[m, 0]], np.float32))[0]
            eb = _bits.binade_exponent(np.array([B[0, n]], np.float32))[0]
            for b in range(5):
                assert abs(T[b]) < Fraction(2) ** int(ea + eb + 3)


@pytest.mark.parametrize("variant", [oracle.BF16X9_FIVE_BANDS, oracle.BF16X9_ONE_ACCUMULATOR])
@pytest.mark.parametrize("tA,tB", TRANS)
def test_bf16x9_gemm_against_exact_rationals(variant, tA, tB):
    rng = np.random.default_rng(14)
    for (M, N, K) in [(3, 3, 1), (4, 5, 8), (3, 4, 24)]:
        A_op = _bits.random_bits_matrix(rng, (M, K), -12, 12)
        B_op = _bits.random_bits_matrix(rng, (K, N), -12, 12)
        A, B = _layout(A_op, B_op, tA, tB)
        C = oracle.gemm_bf16x9(oracle.Problem(A, B, transA=tA, transB=tB), variant=variant)
        err = _rel_err_vs_exact(C, _bits.exact_gemm(A_op, B_op), _bits.exact_absgemm(A_op, B_op))
        # five FP32 sums of length <= 3K each, recombined with four FP32 adds:
        # well inside (K + 4) u; a dropped or misplaced product of bands 0-2
        # costs at least 2^-16 relative, far above it.
        assert err <= (K + 4) * U * 1.0001


# -------------------------------------------------------------- TF32x3 ------
def test_tf32x3_terms_are_the_three_products():
    """K = 1: the three term sums are hi*hi, hi*lo and lo*hi exactly (each a
    product of 11-bit significands); lo*lo is absent, so the result differs
    from a*b by lo_a lo_b plus the split residuals, and by nothing else."""
    rng = np.random.default_rng(15)
    A = _bits.random_bits_matrix(rng, (5, 1), -20, 20)
    B = _bits.random_bits_matrix(rng, (1, 6), -20, 20)
    C, T = oracle.gemm_tf32x3(oracle.Problem(A, B), with_terms=True)
    ha, la = oracle.split_tf32x3(A.ravel())
    hb, lb = oracle.split_tf32x3(B.ravel())
    for m in range(5):
        for n in range(6):
            ah, al, bh, bl = (Fraction(float(x)) for x in (ha[m], la[m], hb[n], lb[n]))
            assert Fraction(float(T[0, m, n])) == ah * bh
            assert Fraction(float(T[1, m, n])) == ah * bl
            assert Fraction(float(T[2, m, n])) == al * bh
            s3 = ah * bh + ah * bl + al * bh
            # C is that three-term sum, rounded twice in FP32
            assert abs(Fraction(float(C[m, n])) - s3) <= abs(s3) * 2 * U * 1.0001
            exact = Fraction(float(A[m, 0])) * Fraction(float(B[0, n]))
            ra = Fraction(float(A[m, 0])) - ah - al
            rb = Fraction(float(B[0, n])) - bh - bl
            assert exact - s3 == al * bl + (ah + al) * rb + ra * (bh + bl) + ra * rb


def test_tf32x3_drops_lo_times_lo_closed_form():
    """a = b = 1 + 2^-11 - 2^-23: hi = 1 and lo = 2^-11 (the residual
    2^-11 - 2^-23 needs 11 fraction bits and rounds up), so the three kept
    products sum to 1 + 2^-10 exactly, while lo*lo = 2^-22 would make it
    1 + 2^-10 + 2^-22, an FP32 number two ulps away."""
    a = np.array([[1 + 2.0 ** -11 - 2.0 ** -23]], np.float32)
    hi, lo = oracle.split_tf32x3(a.ravel())
    assert hi[0] == 1.0 and lo[0] == 2.0 ** -11
    C = oracle.gemm_tf32x3(oracle.Problem(a, a))
    assert C[0, 0] == np.float32(1 + 2.0 ** -10)


@pytest.mark.parametrize("tA,tB", TRANS)
def test_tf32x3_gemm_against_exact_rationals(tA, tB):
    rng = np.random.default_rng(16)
    for (M, N, K) in [(3, 3, 1), (4, 5, 8), (3, 4, 24)]:
        A_op = _bits.random_bits_matrix(rng, (M, K), -12, 12)
        B_op = _bits.random_bits_matrix(rng, (K, N), -12, 12)
        A, B = _layout(A_op, B_op, tA, tB)
        C = oracle.gemm_tf32x3(oracle.Problem(A, B, transA=tA, transB=tB))
        err = _rel_err_vs_exact(C, _bits.exact_gemm(A_op, B_op), _bits.exact_absgemm(A_op, B_op))
        # 3K FP32 additions plus the dropped lo*lo and split residuals
        # (|a - hi - lo| <= 2^-23 |a| each): (3K) u + 3 2^-22
        assert err <= 3 * K * U + 3 * 2.0 ** -22


def test_tf32x3_single_product_error_floor():
    """K = 1: the method's own error (lo*lo dropped, split residuals) reaches
    beyond 4u but stays below 2^-21 = 8u, which is why the TF32x3 normwise
    bound reads K as max(K, 2); BF16x9 at K = 1 stays near one rounding."""
    rng = np.random.default_rng(20)
    a = _bits.random_bits_matrix(rng, (4000, 1), -10, 10)
    b = _bits.random_bits_matrix(rng, (1, 50), -10, 10)
    exact = a.astype(np.float64) @ b.astype(np.float64)  # exact: 48-bit products
    rel_tf = np.abs(oracle.gemm_tf32x3(oracle.Problem(a, b)) - exact) / np.abs(exact)
    rel_bf = np.abs(oracle.gemm_bf16x9(oracle.Problem(a, b)) - exact) / np.abs(exact)
    assert rel_tf.max() > 4 * U and rel_tf.max() <= 8 * U
    assert rel_tf.max() <= oracle.normwise_bound("tf32x3", 1)
    assert rel_bf.max() <= oracle.normwise_bound("bf16x9", 1)


# ----------------------------------------------------- comparator modes ----
def test_bf16x6_keeps_bands_0_to_2_closed_form():
    """a = b = 1 + 2^-8 + 2^-16 has components (1, 1, 1), so the band sums are
    S = (1, 2, 3, 2, 1).  BF16x6 keeps bands 0-2: 1 + 2^-7 + 3 2^-16 exactly;
    BF16x9 adds 2 2^-24 + 2^-32, which rounds to one more ulp (2^-23)."""
    a = np.array([[1 + 2.0 ** -8 + 2.0 ** -16]], np.float32)
    p = oracle.Problem(a, a)
    assert oracle.gemm_bf16x6(p)[0, 0] == np.float32(1 + 2.0 ** -7 + 3 * 2.0 ** -16)
    assert oracle.gemm_bf16x9(p)[0, 0] == np.float32(1 + 2.0 ** -7 + 3 * 2.0 ** -16 + 2.0 ** -23)


@pytest.mark.parametrize("tA,tB", TRANS)
def test_bf16x6_against_exact_rationals(tA, tB):
    rng = np.random.default_rng(22)
    for (M, N, K) in [(3, 3, 1), (4, 5, 8), (3, 4, 24)]:
        A_op = _bits.random_bits_matrix(rng, (M, K), -12, 12)
        B_op = _bits.random_bits_matrix(rng, (K, N), -12, 12)
        A, B = _layout(A_op, B_op, tA, tB)
        C = oracle.gemm_bf16x6(oracle.Problem(A, B, transA=tA, transB=tB))
        err = _rel_err_vs_exact(C, _bits.exact_gemm(A_op, B_op), _bits.exact_absgemm(A_op, B_op))
        # three FP32 band sums + recombination, plus the dropped bands 3-4
        # (each |c_i c_j| 2^-8(i+j) < 4 2^-24 |a b|): (K + 2) u + 2^-20
        assert err <= (K + 2) * U + 2.0 ** -20
        assert err <= oracle.normwise_bound("bf16x6", K)


def test_tf32x1_single_product_is_hi_times_hi():
    """One-pass TF32 at K = 1 is hi(a) hi(b) exactly (11-bit significands)."""
    rng = np.random.default_rng(23)
    a = _bits.random_bits_matrix(rng, (50, 1), -20, 20)
    b = _bits.random_bits_matrix(rng, (1, 40), -20, 20)
    C = oracle.gemm_tf32x1(oracle.Problem(a, b))
    ha, _ = oracle.split_tf32x3(a.ravel())
    hb, _ = oracle.split_tf32x3(b.ravel())
    assert np.array_equal(C.astype(np.float64), np.outer(ha.astype(np.float64), hb.astype(np.float64)))


def test_tf32x1_closed_form_and_bound():
    """a = b = 1 + 2^-11 + 2^-12 rounds to hi = 1 + 2^-10, so one-pass TF32
    gives (1 + 2^-10)^2 = 1 + 2^-9 + 2^-20; random data stays inside
    2 K u + 2^-10 of the exact product sum."""
    a = np.array([[1 + 2.0 ** -11 + 2.0 ** -12]], np.float32)
    assert oracle.gemm_tf32x1(oracle.Problem(a, a))[0, 0] == np.float32(1 + 2.0 ** -9 + 2.0 ** -20)
    rng = np.random.default_rng(24)
    A = _bits.random_bits_matrix(rng, (4, 24), -12, 12)
    B = _bits.random_bits_matrix(rng, (24, 5), -12, 12)
    C = oracle.gemm_tf32x1(oracle.Problem(A, B))
    err = _rel_err_vs_exact(C, _bits.exact_gemm(A, B), _bits.exact_absgemm(A, B))
    assert 2.0 ** -16 < err <= oracle.normwise_bound("tf32x1", 24)


# ------------------------------------------- closed forms (all variants) ----
def _all_modes(p):
    return {
        "sgemm": oracle.sgemm_f32(p),
        "bf16x9": oracle.gemm_bf16x9(p),
        "bf16x9_1acc": oracle.gemm_bf16x9(p, variant=oracle.BF16X9_ONE_ACCUMULATOR),
        "tf32x3": oracle.gemm_tf32x3(p),
    }


@pytest.mark.parametrize("tA,tB", TRANS)
def test_one_hot_rows_select_exactly(tA, tB):
    """op(A) with one-hot rows picks rows of op(B): every mode must return
    them bit for bit, in every storage order (pins operand indexing)."""
    rng = np.random.default_rng(17)
    M, N, K = 6, 9, 7
    sel = rng.integers(0, K, M)
    A_op = np.zeros((M, K), np.float32)
    A_op[np.arange(M), sel] = 1.0
    B_op = rng.standard_normal((K, N)).astype(np.float32)
    A, B = _layout(A_op, B_op, tA, tB)
    for name, C in _all_modes(oracle.Problem(A, B, transA=tA, transB=tB)).items():
        want = B_op[sel]
        if name == "tf32x3":  # lo*lo dropped: hi + lo of each entry, within 2^-23
            assert np.all(np.abs(C - want) <= 2.0 ** -23 * np.abs(want))
        else:
            assert np.array_equal(C, want), name
    C64 = oracle.gemm_f64(oracle.Problem(A, B, transA=tA, transB=tB))
    assert np.array_equal(C64, B_op[sel].astype(np.float64))


def test_alpha_beta_bias_placement():
    """alpha = 2, beta = 0.5 and a bias on an identity product: every term is
    exact, so C = 2 B + 0.5 C_old + bias exactly."""
    rng = np.random.default_rng(18)
    n = 8
    Bm = (rng.integers(-64, 64, (n, n)) / 8).astype(np.float32)
    Cold = (rng.integers(-64, 64, (n, n)) / 4).astype(np.float32)
    bias = (rng.integers(-8, 8, n) / 2).astype(np.float32)
    p = oracle.Problem(np.eye(n, dtype=np.float32), Bm, alpha=2.0, beta=0.5, C_old=Cold, bias=bias)
    want = 2 * Bm.astype(np.float64) + 0.5 * Cold + bias
    for name, C in _all_modes(p).items():
        assert np.array_equal(C.astype(np.float64), want), name
    assert np.array_equal(oracle.gemm_f64(p), want)


def test_beta_zero_never_reads_c():
    A = np.ones((2, 3), np.float32)
    B = np.ones((3, 2), np.float32)
    Cold = np.full((2, 2), np.nan, np.float32)
    p = oracle.Problem(A, B, beta=0.0, C_old=Cold)
    for name, C in _all_modes(p).items():
        assert np.array_equal(C, np.full((2, 2), 3.0, np.float32)), name


def test_k_zero_gives_beta_c_plus_bias():
    A = np.zeros((3, 0), np.float32)
    B = np.zeros((0, 4), np.float32)
    Cold = np.arange(12, dtype=np.float32).reshape(3, 4)
    bias = np.array([1, -1, 2, -2], np.float32)
    p = oracle.Problem(A, B, beta=2.0, C_old=Cold, bias=bias)
    for name, C in _all_modes(p).items():
        assert np.array_equal(C, 2 * Cold + bias), name


def test_row_sample_matches_full():
    rng = np.random.default_rng(19)
    A = rng.standard_normal((40, 24)).astype(np.float32)
    B = rng.standard_normal((24, 10)).astype(np.float32)
    p = oracle.Problem(A, B, bias=rng.standard_normal(10).astype(np.float32))
    rows = np.array([0, 7, 39, 13])
    assert np.array_equal(oracle.gemm_bf16x9(p)[rows], oracle.gemm_bf16x9(p, rows=rows))
    assert np.array_equal(oracle.gemm_tf32x3(p)[rows], oracle.gemm_tf32x3(p, rows=rows))
    assert np.array_equal(oracle.gemm_f64(p)[rows], oracle.gemm_f64(p, rows=rows))


# ------------------------------------------------- the accuracy statement ----
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bf16x9_meets_or_beats_native_fp32(seed):
    """"BF16x9 reaches or exceeds native FP32 accuracy against an FP64
    reference" (Limitations and decision criteria), on the tiny workload's
    distribution; TF32x3 stays inside its looser 4 K u bound."""
    rng = np.random.default_rng(seed)
    M, N, K = 64, 64, 256
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    p = oracle.Problem(A, B)
    C64, D = oracle.gemm_f64(p), oracle.absdenom_f64(p)
    e_bf = oracle.normwise_error(oracle.gemm_bf16x9(p), C64, D)
    e_32 = oracle.normwise_error(oracle.sgemm_f32(p), C64, D)
    e_tf = oracle.normwise_error(oracle.gemm_tf32x3(p), C64, D)
    assert e_bf <= e_32
    assert e_bf <= oracle.normwise_bound("bf16x9", K)
    assert e_tf <= oracle.normwise_bound("tf32x3", K)


def _integer_golden():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "gemm_integer_example.txt")
    blocks, cur = {}, None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                blocks[cur] = []
                continue
            blocks[cur].append([float(x) for x in line.split()])
    g = {k: np.array(v, np.float32) for k, v in blocks.items()}
    return g["A"], g["B"], g["bias"].ravel(), g["C_old"], g["C"]

"""Independent checkers for the oracle's pins: bit patterns, exact rationals.

Nothing here repeats the oracle's formulas.  The checks state the defining
properties of each step (a component is a BF16 or TF32 number; the split
reconstructs the input exactly; a rounding is the nearest or the truncated
value) and verify them with numpy and with exact rational arithmetic.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def f32_patterns_stratified(upper_fracs, low_bits: int, seed: int = 0):
    """Every sign, every finite exponent, every pattern of the `low_bits`
    lowest fraction bits, combined with the given upper fraction patterns
    (placed above the low bits).  Returns float32 values (no Inf/NaN)."""
    low = np.arange(1 << low_bits, dtype=np.uint32)
    out = []
    for sign in (0, 1):
        for e in range(255):
            for up in upper_fracs:
                word = (np.uint32(sign) << np.uint32(31)) | (np.uint32(e) << np.uint32(23)) | \
                       (np.uint32(up) << np.uint32(low_bits)) | low
                out.append(word)
    return np.concatenate(out).view(np.float32)


def binade_exponent(x: np.ndarray) -> np.ndarray:
    """E(x) with 2^E <= |x| < 2^(E+1) for normal x; -126 for subnormals and 0."""
    b = x.view(np.uint32)
    e = ((b >> 23) & 0xFF).astype(np.int64)
    return np.where(e == 0, -126, e - 127)


def low_bits_zero(x: np.ndarray, nbits: int) -> bool:
    return bool(np.all((x.view(np.uint32) & np.uint32((1 << nbits) - 1)) == 0))


def fr(x) -> Fraction:
    return Fraction(float(x))


def exact_gemm(A, B, transA=False, transB=False):
    """Exact rational op(A) op(B) for tiny matrices."""
    A = np.asarray(A, np.float32)
    B = np.asarray(B, np.float32)
    Aop = A.T if transA else A
    Bop = B.T if transB else B
    M, K = Aop.shape
    N = Bop.shape[1]
    return [[sum((fr(Aop[m, k]) * fr(Bop[k, n]) for k in range(K)), Fraction(0))
             for n in range(N)] for m in range(M)]


def exact_absgemm(A, B, transA=False, transB=False):
    A = np.abs(np.asarray(A, np.float32))
    B = np.abs(np.asarray(B, np.float32))
    return exact_gemm(A, B, transA, transB)


def random_bits_matrix(rng: np.random.Generator, shape, emin=-30, emax=30):
    """Random FP32 values with random sign, exponent in [emin, emax] and a
    full random 23-bit fraction (so that every BF16x9 component is used)."""
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, n, dtype=np.uint32) << np.uint32(31)
    exp = (rng.integers(emin, emax + 1, n) + 127).astype(np.uint32) << np.uint32(23)
    frac = rng.integers(0, 1 << 23, n, dtype=np.uint32)
    return (sign | exp | frac).view(np.float32).reshape(shape)

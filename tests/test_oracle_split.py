"""Pins for the oracle's operand splits (no GPU).

BF16x9 split: "each FP32 operand is split into three scaled BF16 components"
(blog "Unlocking Tensor Core performance for machine-learning interatomic
potentials", section "How Tensor Core FP32 bridges the hardware gap", Fig. 1).
TF32x3 split: "a leading TF32 component and a smaller residual component", no
scale factor (same section, Fig. 2).

The pins are properties the pages and the number formats fix: three BF16
numbers with 8-bit significands cover the 24-bit FP32 significand, so the
split must reconstruct every finite FP32 value exactly; TF32 keeps 10
fraction bits, so hi + lo leaves a residual below 2^-23 |a| when both are the
nearest TF32 numbers.  The sweep covers every sign, every finite exponent and
every pattern of the low fraction bits; EMU_EXHAUSTIVE=1 widens it to all
2^32 bit patterns.
"""
import os

import numpy as np
import pytest

import oracle
from tests import _bits

FULL = os.environ.get("EMU_EXHAUSTIVE") == "1"


def _bf16x9_sweep():
    if FULL:
        for hi in range(1 << 8):
            words = (np.uint32(hi) << np.uint32(24)) | np.arange(1 << 24, dtype=np.uint32)
            a = words.view(np.float32)
            yield a[np.isfinite(a)]
    else:
        # every sign x exponent x low-16-bit pattern, with the upper 7 fraction
        # bits all-zero, all-one and mixed; in chunks to bound memory
        a = _bits.f32_patterns_stratified((0x00, 0x7F, 0x2A), 16)
        for s in range(0, a.size, 1 << 23):
            yield a[s:s + (1 << 23)]


def _check_bf16x9(a):
    c0, c1, c2 = oracle.split_bf16x9_f32(a)
    comps = (c0, c1, c2)
    for c in comps:
        assert np.all(np.isfinite(c)), "a finite input gave a non-finite component"
        assert _bits.low_bits_zero(c, 16), "a component is not a BF16 number"
    a64 = a.astype(np.float64)
    rec = c0.astype(np.float64) + c1.astype(np.float64) * 2.0 ** -8 + c2.astype(np.float64) * 2.0 ** -16
    bad = np.nonzero(rec != a64)[0]
    assert bad.size == 0, f"inexact reconstruction for {a[bad[:4]]}"
    # "scaled": every component carries the input's binade, |c_i| < 2^(E(a)+1)
    lim = np.exp2(_bits.binade_exponent(a) + 1.0)
    for c in comps:
        assert np.all(np.abs(c.astype(np.float64)) < lim)
    # c0 is the truncation of a: same sign, not larger, within one BF16 ulp
    ulp_bf16 = np.exp2(_bits.binade_exponent(a) - 7.0)
    d0 = np.abs(a64) - np.abs(c0.astype(np.float64))
    assert np.all(d0 >= 0) and np.all(d0 < ulp_bf16)
    nz = c0 != 0
    assert np.all(np.signbit(c0[nz]) == np.signbit(a[nz]))
    # c1 is the truncation of the scaled remainder r1 = 2^8 (a - c0)
    r1 = (a64 - c0.astype(np.float64)) * 256.0
    d1 = np.abs(r1) - np.abs(c1.astype(np.float64))
    r1_32 = r1.astype(np.float32)  # exact: r1 has at most 16 significant bits
    assert np.array_equal(r1_32.astype(np.float64), r1)
    ulp1 = np.exp2(_bits.binade_exponent(r1_32) - 7.0)
    assert np.all(d1 >= 0) and np.all((d1 < ulp1) | (r1 == 0))


def test_bf16x9_split_exact_and_bf16():
    for a in _bf16x9_sweep():
        _check_bf16x9(a)


def test_bf16x9_split_golden():
    """Hand-derived components (tests/golden/split_examples.txt)."""
    rows = _golden("bf16x9")
    a = np.array([int(r[0], 16) for r in rows], np.uint32).view(np.float32)
    want = [np.array([int(r[i], 16) for r in rows], np.uint16) for i in (1, 2, 3)]
    got = oracle.split_bf16x9(a)
    for i in range(3):
        assert np.array_equal(got[i], want[i]), (i, got[i], want[i])


def test_bf16x9_nonfinite_documented():
    """Inf and NaN are outside the split's domain: Inf - Inf is NaN, so the
    lower components of an infinite input are NaN (no IEEE Inf propagation)."""
    a = np.array([np.inf, -np.inf, np.nan], np.float32)
    c0, c1, c2 = oracle.split_bf16x9_f32(a)
    assert np.isinf(c0[0]) and np.isinf(c0[1]) and np.isnan(c0[2])
    assert np.all(np.isnan(c1)) and np.all(np.isnan(c2))


# ------------------------------------------------------------------ TF32 ----
def _tf32_sweep():
    if FULL:
        for hi in range(1 << 8):
            words = (np.uint32(hi) << np.uint32(24)) | np.arange(1 << 24, dtype=np.uint32)
            a = words.view(np.float32)
            yield a[np.isfinite(a)]
    else:
        a = _bits.f32_patterns_stratified((0, 1, 0x155, 0x2AA, 0x3FE, 1023, 512, 73), 13)
        for s in range(0, a.size, 1 << 23):
            yield a[s:s + (1 << 23)]


def _assert_nearest_tf32(x64, t, what):
    """t (float32) is a TF32 number nearest to the exact value x64, ties to even."""
    assert _bits.low_bits_zero(t, 13), f"{what}: not a TF32 number"
    tb = t.view(np.uint32)
    mag = tb & np.uint32(0x7FFFFFFF)
    sgn = tb & np.uint32(0x80000000)
    up = (sgn | (mag + np.uint32(0x2000))).view(np.float32).astype(np.float64)
    dn_mag = np.where(mag >= 0x2000, mag - np.uint32(0x2000), np.uint32(0x2000))
    dn_sgn = np.where(mag >= 0x2000, sgn, sgn ^ np.uint32(0x80000000))
    dn = (dn_sgn | dn_mag).view(np.float32).astype(np.float64)
    e = np.abs(x64 - t.astype(np.float64))
    e_up = np.abs(x64 - up)
    e_dn = np.abs(x64 - dn)
    fin = np.isfinite(up)
    assert np.all(e[fin] <= e_up[fin]), f"{what}: a larger neighbour is nearer"
    assert np.all(e <= e_dn), f"{what}: a smaller neighbour is nearer"
    tie = (e == e_up) | (e == e_dn)
    odd = ((tb >> np.uint32(13)) & np.uint32(1)) == 1
    assert not np.any(tie & odd), f"{what}: a tie was not broken to even"


def _check_tf32(a):
    hi, lo = oracle.split_tf32x3(a, oracle.TF32X3_HI_RN)
    a64 = a.astype(np.float64)
    ok = np.isfinite(hi)  # hi rounds to Inf only beyond the largest TF32 number
    assert np.all(np.abs(a[~ok]) > 3.40e38)
    a, a64, hi, lo = a[ok], a64[ok], hi[ok], lo[ok]
    _assert_nearest_tf32(a64, hi, "hi")
    resid = a64 - hi.astype(np.float64)  # exact
    _assert_nearest_tf32(resid, lo, "lo")
    big = np.abs(a64) >= 2.0 ** -100
    r2 = np.abs(resid - lo.astype(np.float64))
    assert np.all(r2[big] <= 2.0 ** -23 * np.abs(a64[big]))

    hz, lz = oracle.split_tf32x3(a, oracle.TF32X3_HI_RZ)
    assert _bits.low_bits_zero(hz, 13) and _bits.low_bits_zero(lz, 13)
    d = np.abs(a64) - np.abs(hz.astype(np.float64))
    assert np.all(d >= 0) and np.all(d < np.exp2(_bits.binade_exponent(a) - 10.0))
    _assert_nearest_tf32(a64 - hz.astype(np.float64), lz, "lo (hi truncated)")
    rz = np.abs(a64 - hz.astype(np.float64) - lz.astype(np.float64))
    assert np.all(rz[big] <= 2.0 ** -22 * np.abs(a64[big]))


def test_tf32x3_split_nearest_and_residual():
    for a in _tf32_sweep():
        _check_tf32(a)


def test_tf32x3_split_golden():
    rows = _golden("tf32x3")
    a = np.array([int(r[0], 16) for r in rows], np.uint32).view(np.float32)
    hi, lo = oracle.split_tf32x3(a)
    assert np.array_equal(hi.view(np.uint32), np.array([int(r[1], 16) for r in rows], np.uint32))
    assert np.array_equal(lo.view(np.uint32), np.array([int(r[2], 16) for r in rows], np.uint32))


def _golden(section):
    path = os.path.join(os.path.dirname(__file__), "golden", "split_examples.txt")
    rows, cur = [], None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = line[1:-1]
                continue
            if cur == section:
                rows.append(line.split())
    assert rows, section
    return rows

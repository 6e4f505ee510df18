"""CPU oracle for FP32 GEMM emulated with BF16x9 and TF32x3 (numpy + ctypes).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the library.  It shares
no code with the CUDA path.  The arithmetic lives in ``emu_oracle.c``; this
module builds it with gcc, loads it and marshals numpy arrays.

Every function follows the blog post "Unlocking Tensor Core performance for
machine-learning interatomic potentials", section "How Tensor Core FP32
bridges the hardware gap" (Fig. 1 for BF16x9, Fig. 2 and Eq. 1 for TF32x3);
the float64 GEMM and the sequential FP32 SGEMM are the plain definitions the
method is judged against ("Limitations and decision criteria").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "emu_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16X9_FIVE_BANDS = 0
BF16X9_ONE_ACCUMULATOR = 1
TF32X3_HI_RN = 0
TF32X3_HI_RZ = 1


def build(force: bool = False) -> str:
    """Compile emu_oracle.c into liboracle.so (OpenMP when gcc has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            i32 = ctypes.c_int
            f32 = ctypes.c_float
            f64 = ctypes.c_double
            L.oracle_split_bf16x9.argtypes = [P, i64, P, P, P]
            L.oracle_split_bf16x9_f32.argtypes = [P, i64, P, P, P]
            L.oracle_split_tf32x3.argtypes = [P, i64, i32, P, P]
            gemm_head = [i32, i32, i64, i64, i64]
            L.oracle_gemm_f64.argtypes = gemm_head + [f64, P, i64, P, i64, f64, P, i64, P, P, i64, P]
            L.oracle_gemm_absdenom_f64.argtypes = gemm_head + [f64, P, i64, P, i64, f64, P, i64, P, P, i64, P]
            L.oracle_sgemm_f32.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, P, i64, P]
            L.oracle_gemm_bf16x9.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, i32, P, i64, P, P]
            L.oracle_gemm_tf32x3.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, i32, P, i64, P, P]
            L.oracle_gemm_bf16x6.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, P, i64, P]
            L.oracle_gemm_tf32x1.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, P, i64, P]
            L.oracle_gemm_exact_sum.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, i32, P, i64, P]
            L.oracle_gemm_tc.argtypes = gemm_head + [f32, P, i64, P, i64, f32, P, i64, P, P, i64, P,
                                                     i32, i32, i32, i32, i32, i32]
            L.oracle_tc_block_fma.argtypes = [f32, P, P, i32, i32, i32]
            L.oracle_tc_block_fma.restype = f32
            for name in ("oracle_gemm_f64", "oracle_gemm_absdenom_f64", "oracle_sgemm_f32",
                         "oracle_gemm_bf16x9", "oracle_gemm_tf32x3", "oracle_gemm_bf16x6",
                         "oracle_gemm_tf32x1", "oracle_gemm_exact_sum", "oracle_gemm_tc",
                         "oracle_num_threads"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


class use_library:
    """Temporarily route every oracle call through another build of the C
    source (the tests use it to check that planted mistakes fail the pins)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        self._saved = _lib
        L = ctypes.CDLL(self.path)
        for name in ("oracle_split_bf16x9", "oracle_split_bf16x9_f32", "oracle_split_tf32x3",
                     "oracle_gemm_f64", "oracle_gemm_absdenom_f64", "oracle_sgemm_f32",
                     "oracle_gemm_bf16x9", "oracle_gemm_tf32x3", "oracle_gemm_bf16x6",
                     "oracle_gemm_tf32x1", "oracle_gemm_exact_sum", "oracle_gemm_tc", "oracle_tc_block_fma",
                     "oracle_num_threads"):
            f, g = getattr(L, name), getattr(self._saved, name)
            f.argtypes, f.restype = g.argtypes, g.restype
        _lib = L
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def build_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle's C source to out_path."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", src,
                    "-o", out_path, "-lm"], check=True, capture_output=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ---------------------------------------------------------------- splits ----
def split_bf16x9(a):
    """BF16x9 split (Fig. 1): three scaled BF16 components as uint16 bit patterns.

    a = c0 + 2^-8 c1 + 2^-16 c2, each component rounded toward zero to BF16.
    """
    a = _f32(a).ravel()
    s = [np.empty(a.size, np.uint16) for _ in range(3)]
    lib().oracle_split_bf16x9(_ptr(a), a.size, *(_ptr(x) for x in s))
    return tuple(s)


def split_bf16x9_f32(a):
    """Same split, each component returned as the full FP32 word."""
    a = _f32(a).ravel()
    s = [np.empty(a.size, np.float32) for _ in range(3)]
    lib().oracle_split_bf16x9_f32(_ptr(a), a.size, *(_ptr(x) for x in s))
    return tuple(s)


def split_tf32x3(a, variant: int = TF32X3_HI_RN):
    """TF32x3 split (Fig. 2): hi = nearest TF32 (or truncated), lo = nearest TF32 of a - hi."""
    a = _f32(a).ravel()
    hi = np.empty(a.size, np.float32)
    lo = np.empty(a.size, np.float32)
    lib().oracle_split_tf32x3(_ptr(a), a.size, int(variant), _ptr(hi), _ptr(lo))
    return hi, lo


# ----------------------------------------------------------------- GEMMs ----
class Problem:
    """C = alpha * op(A) op(B) + beta * C_old (+ bias), row-major operands."""

    def __init__(self, A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0,
                 C_old=None, bias=None):
        self.A = _f32(A)
        self.B = _f32(B)
        self.transA = bool(transA)
        self.transB = bool(transB)
        self.M = self.A.shape[1] if transA else self.A.shape[0]
        self.K = self.A.shape[0] if transA else self.A.shape[1]
        kb = self.B.shape[1] if transB else self.B.shape[0]
        self.N = self.B.shape[0] if transB else self.B.shape[1]
        if kb != self.K:
            raise ValueError("inner dimensions differ")
        self.alpha = float(alpha)
        self.beta = float(beta)
        self.C_old = None if C_old is None else _f32(C_old)
        if self.beta != 0.0 and (self.C_old is None or self.C_old.shape != (self.M, self.N)):
            raise ValueError("beta != 0 needs C_old of shape (M, N)")
        self.bias = None if bias is None else _f32(bias).ravel()

    def _head(self):
        lda = self.A.shape[1] if self.A.ndim == 2 else 1
        ldb = self.B.shape[1] if self.B.ndim == 2 else 1
        return (int(self.transA), int(self.transB), self.M, self.N, self.K), lda, ldb

    def _rows(self, rows):
        if rows is None:
            return None, self.M
        r = np.ascontiguousarray(rows, dtype=np.int64)
        if r.size and (r.min() < 0 or r.max() >= self.M):
            raise ValueError("row index out of range")
        return r, r.size

    def _cold(self):
        c = self.C_old if (self.beta != 0.0 and self.C_old is not None) else None
        return _ptr(c), (self.N if c is not None else 0)


def gemm_f64(p: Problem, rows=None):
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float64)
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_f64(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                               _ptr(p.bias), _ptr(r), nr, _ptr(out))
    if rc:
        raise MemoryError("oracle_gemm_f64")
    return out


def absdenom_f64(p: Problem, rows=None):
    """D = |alpha| |op(A)||op(B)| + |beta||C_old| + |bias| (normwise-error denominator)."""
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float64)
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_absdenom_f64(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp,
                                        ldc, _ptr(p.bias), _ptr(r), nr, _ptr(out))
    if rc:
        raise MemoryError("oracle_gemm_absdenom_f64")
    return out


def sgemm_f32(p: Problem, rows=None):
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    cp, ldc = p._cold()
    rc = lib().oracle_sgemm_f32(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                                _ptr(p.bias), _ptr(r), nr, _ptr(out))
    if rc:
        raise MemoryError("oracle_sgemm_f32")
    return out


def gemm_bf16x9(p: Problem, rows=None, variant: int = BF16X9_FIVE_BANDS, with_bands=False):
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    bands = np.empty((5, nr, p.N), np.float32) if with_bands else None
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_bf16x9(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                                  _ptr(p.bias), int(variant), _ptr(r), nr, _ptr(out), _ptr(bands))
    if rc:
        raise MemoryError("oracle_gemm_bf16x9")
    return (out, bands) if with_bands else out


def gemm_tf32x3(p: Problem, rows=None, variant: int = TF32X3_HI_RN, with_terms=False):
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    terms = np.empty((3, nr, p.N), np.float32) if with_terms else None
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_tf32x3(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                                  _ptr(p.bias), int(variant), _ptr(r), nr, _ptr(out), _ptr(terms))
    if rc:
        raise MemoryError("oracle_gemm_tf32x3")
    return (out, terms) if with_terms else out


def gemm_bf16x6(p: Problem, rows=None):
    """Comparator: BF16x9 without bands 3 and 4 (six products)."""
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_bf16x6(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                                  _ptr(p.bias), _ptr(r), nr, _ptr(out))
    if rc:
        raise MemoryError("oracle_gemm_bf16x6")
    return out


def gemm_tf32x1(p: Problem, rows=None):
    """Comparator: one-pass TF32 (hi(a) hi(b) only)."""
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_tf32x1(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                                  _ptr(p.bias), _ptr(r), nr, _ptr(out))
    if rc:
        raise MemoryError("oracle_gemm_tf32x1")
    return out


EXACT_KIND = {"bf16x9": 0, "bf16x6": 1, "tf32x3": 2, "tf32x1": 3}


def gemm_exact(p: Problem, mode: str, rows=None):
    """The emulated result with exact accumulation: the mode's selected
    component products (BF16x9 Fig. 1: nine scaled products; TF32x3 Eq. 1:
    hi hi + hi lo + lo hi; BF16x6: bands 0-2; one-pass TF32: hi hi), summed
    over k with no rounding, rounded once to FP32 (nearest even), then the
    FP32 epilogue.  The reference for the elementwise agreement of any FP32
    accumulation of those products."""
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_exact_sum(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                                     _ptr(p.bias), EXACT_KIND[mode], _ptr(r), nr, _ptr(out))
    if rc == -2:
        raise ValueError("gemm_exact: bad mode or K too large")
    if rc:
        raise MemoryError("oracle_gemm_exact_sum")
    return out


# Tensor-core model parameters ([TC models] "Results"): blocks of 16 products
# for BF16 inputs (one 16-deep instruction of the kernel), 8 for TF32 (one
# 8-deep instruction), 2 extra alignment bits, rounding toward zero.
TC_NEAB = 2
TC_TOWARD_ZERO, TC_NEAREST = 0, 1
TC_KIND = {"bf16x9": 0, "bf16x6": 1, "tf32x3": 2, "tf32x1": 3}
TC_BLOCK = {"bf16x9": 16, "bf16x6": 16, "tf32x3": 8, "tf32x1": 8}


def tc_block_fma(c, a, b, neab=TC_NEAB, round_mode=TC_TOWARD_ZERO):
    """One block FMA of the tensor-core model: FP32 c plus sum a_i b_i."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    assert a.shape == b.shape and a.ndim == 1
    return float(lib().oracle_tc_block_fma(float(c), _ptr(a), _ptr(b), len(a), int(neab), int(round_mode)))


def gemm_tc(p: Problem, mode="bf16x9", rows=None, *, pieces=1, stage_k=32, block=None, neab=TC_NEAB,
            round_mode=TC_TOWARD_ZERO):
    """The emulated GEMM through the tensor-core accumulation model, in the
    kernel's issue order (see oracle_gemm_tc); pieces > 1 models a split of
    every tile's k-range into that many pieces, reduced owner first."""
    block = TC_BLOCK[mode] if block is None else block
    (h, lda, ldb), (r, nr) = p._head(), p._rows(rows)
    out = np.empty((nr, p.N), np.float32)
    cp, ldc = p._cold()
    rc = lib().oracle_gemm_tc(*h, p.alpha, _ptr(p.A), lda, _ptr(p.B), ldb, p.beta, cp, ldc,
                              _ptr(p.bias), _ptr(r), nr, _ptr(out), TC_KIND[mode], int(stage_k), int(block),
                              int(neab), int(round_mode), int(pieces))
    if rc == -2:
        raise ValueError("gemm_tc: bad mode, block, stage or pieces")
    if rc:
        raise MemoryError("oracle_gemm_tc")
    return out


def gemm_emulated(p: Problem, mode: str, rows=None):
    """The oracle's emulated result for mode 'bf16x9', 'tf32x3', 'bf16x6' or 'tf32x1'."""
    if mode == "bf16x9":
        return gemm_bf16x9(p, rows)
    if mode == "tf32x3":
        return gemm_tf32x3(p, rows)
    if mode == "bf16x6":
        return gemm_bf16x6(p, rows)
    if mode == "tf32x1":
        return gemm_tf32x1(p, rows)
    raise ValueError(mode)


# --------------------------------------------------------------- metrics ----
U = 2.0 ** -24  # FP32 unit roundoff


def normwise_error(C, C64, D):
    """max_ij |C - C64| / D (Higham's componentwise-normwise form); entries
    with D == 0 must match exactly (they contribute inf otherwise)."""
    C = np.asarray(C, np.float64)
    diff = np.abs(C - C64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(D > 0, diff / np.where(D > 0, D, 1.0), np.where(diff == 0, 0.0, np.inf))
    return float(q.max()) if q.size else 0.0


def normwise_bound(mode: str, K: int) -> float:
    """2 K u for BF16x9, 4 K u for TF32x3 (u = 2^-24).

    TF32x3 reads K as max(K, 2): dropping lo*lo (Eq. 1) and the two split
    residuals leave up to 2^-21 = 8u per product, so at K = 1 no TF32x3
    result, the oracle's included, can meet 4u.
    Comparators: BF16x6 drops bands 3-4 (at most 2^-20 of each |a b|):
    2 K u + 2^-20; one-pass TF32 keeps 11 significant bits per operand (at
    most 2^-10 of each |a b|): 2 K u + 2^-10."""
    if mode == "bf16x6":
        return 2.0 * max(int(K), 1) * U + 2.0 ** -20
    if mode == "tf32x1":
        return 2.0 * max(int(K), 1) * U + 2.0 ** -10
    k = max(int(K), 1) if mode == "bf16x9" else max(int(K), 2)
    return (2.0 if mode == "bf16x9" else 4.0) * k * U


def elementwise_excess(C, C_ref, rel=1e-5):
    """Largest |C - C_ref| / (rel * max(|C_ref|, rms(C_ref))); <= 1 passes.

    The rms floor: entries near zero come from cancellation, where any two
    accumulation orders differ by far more than 1e-5 of the entry itself."""
    C = np.asarray(C, np.float64)
    E = np.asarray(C_ref, np.float64)
    if E.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(E * E)))
    scale = rel * np.maximum(np.abs(E), rms)
    diff = np.abs(C - E)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0), np.where(diff == 0, 0.0, np.inf))
    return float(q.max())

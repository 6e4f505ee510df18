"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle


def device():
    import torch
    return torch.device("cuda:0")


def to_dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(device())


def to_dev_padded(x, fill=0.0):
    """2-D device copy whose leading dimension is padded to a multiple of 4
    elements (what TMA needs); the padding holds `fill`."""
    import torch
    r, c = x.shape
    ld = (c + 3) // 4 * 4
    buf = torch.full((r, ld), fill, dtype=torch.float32, device=device())
    buf[:, :c] = torch.from_numpy(np.ascontiguousarray(x)).to(device())
    return buf[:, :c]


# C guard band: every C buffer the tests hand to the library has extra
# columns past N (and one extra row) holding this NaN pattern; a store outside
# the logical M x N view would overwrite it.
GUARD_BITS = np.uint32(0x7FC0DEAD)


def gpu_sgemm(mode, A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0, C_old=None):
    """C = alpha op(A) op(B) + beta C_old through emu_sgemm.  A and B get NaN
    padding past their logical edge; C lives in a buffer with a guard band
    (4 to 7 extra columns and one extra row) filled with GUARD_BITS, checked
    after the call."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    M = A.shape[1] if transA else A.shape[0]
    N = B.shape[0] if transB else B.shape[1]
    ldc = (N + 3) // 4 * 4 + 4
    guard = torch.from_numpy(np.full((M + 1, ldc), GUARD_BITS, np.uint32).view(np.float32)).to(device())
    C = guard[:M, :N]
    if beta != 0.0:
        C.copy_(torch.from_numpy(np.ascontiguousarray(C_old, np.float32)))
    else:
        C.fill_(float("nan"))  # beta = 0 never reads C
    # padding of A and B is NaN: a read past the logical edge would show
    emu.sgemm(to_dev_padded(A, float("nan")), to_dev_padded(B, float("nan")), mode=mode, transA=transA,
              transB=transB, alpha=alpha, beta=beta, C=C)
    st = emu.emu_stream_check()
    assert st == 0, emu.emu_status_string(st)
    full = guard.cpu().numpy().view(np.uint32)
    assert np.all(full[:M, N:] == GUARD_BITS), "a store landed in C's padding columns"
    assert np.all(full[M, :] == GUARD_BITS), "a store landed past C's last row"
    return full[:M, :N].view(np.float32).copy()


# Metrics of every comparison in this process, written as JSON lines to the
# file named by EMU_PARITY_REPORT (if set) by the session hook in conftest.py.
REPORT = []

# The oracle's sequential FP32 accumulation is itself a reference for the 1e-5
# elementwise bar only where it lies within this fraction of the bar from the
# exact-accumulation result; beyond that (long sums, TF32x3 at K = 4096) its
# own rounding error is a large part of the bar and only the exact
# reference is asserted.
SEQUENTIAL_TRUST = 0.5


def compare(mode, C, p: oracle.Problem, rows=None, elementwise=True, label=None):
    """Check a GPU result against the oracle:
      - normwise error against the float64 GEMM within 2 K u (BF16x9) or
        4 K u (TF32x3), u = 2^-24;
      - elementwise: |C - C_ref| <= 1e-5 max(|C_ref|, rms(C_ref)) against the
        exact-accumulation result (the method's products summed exactly and
        rounded once), and against the oracle's sequential FP32 emulation
        wherever that one is within SEQUENTIAL_TRUST of the bar from the
        exact result -- plain bars, no credit term;
      - finite output.
    Returns the metrics (also appended to REPORT)."""
    C = np.asarray(C)
    Cs = C if rows is None else C[rows]
    C64 = oracle.gemm_f64(p, rows)
    D = oracle.absdenom_f64(p, rows)
    nw = oracle.normwise_error(Cs, C64, D)
    bound = oracle.normwise_bound(mode, p.K)
    out = {"label": label, "mode": mode, "M": p.M, "N": p.N, "K": p.K,
           "rows": int(p.M if rows is None else len(rows)), "normwise": nw, "bound": bound}
    if elementwise:
        Cx = oracle.gemm_exact(p, mode, rows)
        Ce = oracle.gemm_emulated(p, mode, rows)
        out["excess_vs_exact"] = oracle.elementwise_excess(Cs, Cx)
        out["excess_vs_sequential"] = oracle.elementwise_excess(Cs, Ce)
        out["sequential_vs_exact"] = oracle.elementwise_excess(Ce, Cx)
        out["sequential_asserted"] = out["sequential_vs_exact"] <= SEQUENTIAL_TRUST
    REPORT.append(out)
    assert nw <= bound, f"{mode}: normwise error {nw:.3e} > {bound:.3e}"
    if elementwise:
        assert out["excess_vs_exact"] <= 1.0, (
            f"{mode}: elementwise excess {out['excess_vs_exact']:.3f} against the exact-accumulation result")
        if out["sequential_asserted"]:
            assert out["excess_vs_sequential"] <= 1.0, (
                f"{mode}: elementwise excess {out['excess_vs_sequential']:.3f} against the sequential oracle")
    assert np.all(np.isfinite(Cs)), "non-finite output on finite data"
    return out

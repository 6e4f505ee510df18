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


def gpu_sgemm(mode, A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0, C_old=None):
    import fp32_emulated_gemm_gb300 as emu
    M = A.shape[1] if transA else A.shape[0]
    N = B.shape[0] if transB else B.shape[1]
    if beta != 0.0:
        C = to_dev_padded(C_old)
    else:
        C = to_dev_padded(np.zeros((M, N), np.float32), fill=float("nan"))
        C.fill_(float("nan"))
    # padding of A and B is NaN: a read past the logical edge would show
    emu.sgemm(to_dev_padded(A, float("nan")), to_dev_padded(B, float("nan")), mode=mode, transA=transA,
              transB=transB, alpha=alpha, beta=beta, C=C)
    st = emu.emu_stream_check()
    assert st == 0, emu.emu_status_string(st)
    return C.cpu().numpy()


def compare(mode, C, p: oracle.Problem, rows=None, elementwise=True):
    """Normwise error vs the float64 oracle (bound 2Ku / 4Ku) and elementwise
    agreement with the oracle's emulated result (1e-5 relative, rms floor).
    Returns the metrics for reporting."""
    C = np.asarray(C)
    Cs = C if rows is None else C[rows]
    C64 = oracle.gemm_f64(p, rows)
    D = oracle.absdenom_f64(p, rows)
    nw = oracle.normwise_error(Cs, C64, D)
    bound = oracle.normwise_bound(mode, p.K)
    out = {"normwise": nw, "bound": bound}
    assert nw <= bound, f"{mode}: normwise error {nw:.3e} > {bound:.3e}"
    if elementwise:
        Ce = oracle.gemm_emulated(p, mode, rows)
        ex = oracle.elementwise_excess(Cs, Ce, C64=C64)
        out["elementwise_excess"] = ex
        out["elementwise_excess_plain"] = oracle.elementwise_excess(Cs, Ce)
        assert ex <= 1.0, (f"{mode}: elementwise excess {ex:.3f} (> 1 means beyond 1e-5 relative of the "
                           f"oracle and farther from float64 than the oracle)")
    assert np.all(np.isfinite(Cs)), "non-finite output on finite data"
    return out

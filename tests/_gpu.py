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


def gpu_sgemm(mode, A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0, C_old=None):
    import fp32_emulated_gemm_gb300 as emu
    M = A.shape[1] if transA else A.shape[0]
    N = B.shape[0] if transB else B.shape[1]
    if beta != 0.0:
        C = to_dev(C_old)
    else:
        import torch
        C = torch.full((M, N), float("nan"), device=device(), dtype=torch.float32)
    emu.sgemm(to_dev(A), to_dev(B), mode=mode, transA=transA, transB=transB, alpha=alpha, beta=beta, C=C)
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
        ex = oracle.elementwise_excess(Cs, Ce)
        out["elementwise_excess"] = ex
        assert ex <= 1.0, f"{mode}: elementwise excess {ex:.3f} (> 1 means beyond 1e-5 relative)"
    assert np.all(np.isfinite(Cs)), "non-finite output on finite data"
    return out

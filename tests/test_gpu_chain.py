"""Chained plans on the GPU: every CTA pair runs one equal run of k-stages,
taken tile by tile; a tile cut at a run boundary is split between the two
pairs, the low k-stages first on one pair (which publishes its running FP32
sum) and the high k-stages last on the other (which starts from that sum).
The stage sums are then added in the same order, with the same roundings, as
in an uncut tile, so a chained launch must give the bits of the unsplit plan
(EMU_SPLIT_K=1) on every element, and those of the oracle's tensor-core model
without pieces.  The tolerances against the plain oracle (_gpu.compare) hold
as for every plan.

Plans are forced with EMU_CHAIN=1 (chained wherever there are at least as
many tiles as CTA pairs, with the planner's bounds), EMU_CHAIN=2 (the same
with the even cuts c U / P, which cut tiles in more places: pieces of one
stage, runs of three or more units) and EMU_CHAIN=0 with EMU_SPLIT_K=1
(whole tiles).
"""
import numpy as np
import pytest

import oracle
from fp32_emulated_gemm_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
PAIRS = 76  # co-resident CTA pairs of this kernel on a GB300


def _same_bits(got, want, what):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    diff = got.view(np.uint32) != want.view(np.uint32)
    assert not diff.any(), f"{what}: {int(diff.sum())} of {diff.size} elements differ, " \
                           f"e.g. {got[diff][:3]} vs {want[diff][:3]}"


def _plans(M, N, K, monkeypatch, chain="1"):
    """Set the chained plan up and check it cuts tiles; return the plan."""
    import fp32_emulated_gemm_gb300 as emu
    monkeypatch.setenv("EMU_CHAIN", chain)
    plan = emu.emu_plan_query(M, N, K, PAIRS)
    assert plan["chain"] == 1 and plan["slots"] == PAIRS - 1, plan
    return plan


def _unsplit(monkeypatch):
    monkeypatch.setenv("EMU_CHAIN", "0")
    monkeypatch.setenv("EMU_SPLIT_K", "1")


CASES = {
    # ragged in every dimension: 8 x 10 tiles of 7 k-stages, runs of 7-8 stages
    "ragged": ((2000, 2500, 200), "1"),
    "ragged_even": ((2000, 2500, 200), "2"),
    # 2 k-stages per tile, runs of 2-3 (even cuts): cut tiles split 1 + 1
    "two_stages_even": ((2560, 2048, 64), "2"),
    # 300 tiles of 3 stages, runs of about 12 (even cuts): whole tiles
    # between the cut ones
    "many_units_even": ((5120, 3840, 96), "2"),
    # 300 tiles of 7 stages, runs of about 28
    "many_units": ((5120, 3840, 224), "1"),
}


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3", "bf16x6", "tf32x1"])
@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("tA,tB", [(False, False), (True, True)])
def test_chained_plan_gives_the_unsplit_bits(mode, case, tA, tB, monkeypatch):
    import fp32_emulated_gemm_gb300 as emu
    (M, N, K), chain = CASES[case]
    rng = np.random.default_rng(61)
    A = rng.standard_normal((K, M) if tA else (M, K)).astype(np.float32)
    B = rng.standard_normal((N, K) if tB else (K, N)).astype(np.float32)
    Cold = rng.standard_normal((M, N)).astype(np.float32)
    kw = dict(transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    _plans(M, N, K, monkeypatch, chain)
    C = _gpu.gpu_sgemm(mode, A, B, **kw)
    assert emu.emu_stream_check() == 0
    _unsplit(monkeypatch)
    C1 = _gpu.gpu_sgemm(mode, A, B, **kw)
    _same_bits(C, C1, "chained vs unsplit plan")
    rows = W.sample_rows(M, every=97, edge=3)
    p = oracle.Problem(A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    _same_bits(C[rows], oracle.gemm_tc(p, mode=mode, rows=rows, pieces=1), "chained vs tensor-core model")
    _gpu.compare(mode, C, p, rows, label=f"chained {case}")


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
@pytest.mark.parametrize("chain", ["1", "2"])
def test_chained_pet_small_forward_with_bias(mode, chain, monkeypatch):
    """The PET-small forward pass (96 tiles of 8 k-stages on 76 pairs) through
    emu_linear_fwd with its bias."""
    import fp32_emulated_gemm_gb300 as emu
    s = W.PET_SMALL
    X, Wt, b, _ = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    Xd, Wd, bd = _gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b)
    _plans(s.M, s.N, s.K, monkeypatch, chain)
    Y = emu.linear_fwd(Xd, Wd, bd, mode=mode).cpu().numpy()
    assert emu.emu_stream_check() == 0
    _unsplit(monkeypatch)
    Y1 = emu.linear_fwd(Xd, Wd, bd, mode=mode).cpu().numpy()
    _same_bits(Y, Y1, "chained vs unsplit plan")
    rows = W.sample_rows(s.M, every=97, edge=4)
    p = oracle.Problem(X, Wt, transB=True, bias=b)
    _same_bits(Y[rows], oracle.gemm_tc(p, mode=mode, rows=rows, pieces=1), "chained vs tensor-core model")


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_chained_input_gradient_shape(mode, monkeypatch):
    """An input-gradient product (op(B) MN-major in memory, transposed in the
    split) with 80 tiles of 32 k-stages: long runs, cut tiles of unequal
    halves."""
    import fp32_emulated_gemm_gb300 as emu
    M, Kin, Nout = 2560, 2048, 1024           # dX[M, Kin] = dY[M, Nout] W[Nout, Kin]
    rng = np.random.default_rng(62)
    dY = rng.standard_normal((M, Nout)).astype(np.float32)
    Wt = (rng.standard_normal((Nout, Kin)) / np.sqrt(Nout)).astype(np.float32)
    dYd, Wd = _gpu.to_dev(dY), _gpu.to_dev(Wt)
    _plans(M, Kin, Nout, monkeypatch)
    dX = emu.linear_bwd_input(dYd, Wd, mode=mode).cpu().numpy()
    assert emu.emu_stream_check() == 0
    _unsplit(monkeypatch)
    dX1 = emu.linear_bwd_input(dYd, Wd, mode=mode).cpu().numpy()
    _same_bits(dX, dX1, "chained vs unsplit plan")
    rows = W.sample_rows(M, every=89, edge=2)
    p = oracle.Problem(dY, Wt)
    _same_bits(dX[rows], oracle.gemm_tc(p, mode=mode, rows=rows, pieces=1), "chained vs tensor-core model")
    _gpu.compare(mode, dX, p, rows, label="chained input gradient")


@pytest.mark.parametrize("case", range(6))
def test_random_chained_shapes_give_the_unsplit_bits(case, monkeypatch):
    """Seeded random shapes with at least as many tiles as CTA pairs (so the
    plan can chain), random layouts, alpha, beta and C_old, and both bound
    choices: every element equal to the unsplit plan's, sampled rows equal to
    the tensor-core model's."""
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(3000 + case)
    mode = ["bf16x9", "tf32x3", "bf16x6", "tf32x1"][case % 4]
    while True:
        M, N = int(rng.integers(1500, 6000)), int(rng.integers(1500, 4500))
        K = int(rng.integers(33, 700))
        if -(-M // 256) * -(-N // 256) >= PAIRS:
            break
    tA, tB = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    alpha, beta = float(rng.choice([1.0, 0.5, -1.25])), float(rng.choice([0.0, 1.0, -0.75]))
    A = rng.standard_normal((K, M) if tA else (M, K)).astype(np.float32)
    B = rng.standard_normal((N, K) if tB else (K, N)).astype(np.float32)
    Cold = rng.standard_normal((M, N)).astype(np.float32)
    kw = dict(transA=tA, transB=tB, alpha=alpha, beta=beta, C_old=Cold)
    chain = "1" if case % 2 == 0 else "2"
    monkeypatch.setenv("EMU_CHAIN", chain)
    plan = emu.emu_plan_query(M, N, K, PAIRS)
    assert plan["chain"] == 1, plan
    C = _gpu.gpu_sgemm(mode, A, B, **kw)
    assert emu.emu_stream_check() == 0
    _unsplit(monkeypatch)
    _same_bits(C, _gpu.gpu_sgemm(mode, A, B, **kw), f"chained vs unsplit, {mode} M={M} N={N} K={K} tA={tA} tB={tB}")
    rows = np.unique(rng.integers(0, M, size=12)).astype(np.int64)
    p = oracle.Problem(A, B, transA=tA, transB=tB, alpha=alpha, beta=beta, C_old=Cold)
    _same_bits(C[rows], oracle.gemm_tc(p, mode=mode, rows=rows, pieces=1), "chained vs tensor-core model")

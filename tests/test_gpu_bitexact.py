"""The CUDA path against the oracle's tensor-core model, bit for bit.

The oracle models each tensor-core instruction as one block FMA ([TC models]
"Results": 16 BF16 or 8 TF32 products, 2 extra alignment bits, truncation)
and follows the kernel's order of work: 32-deep stages, a fresh accumulator
per stage fed product by product smallest first, an FP32 sum over stages,
and for split tiles the pieces' sums added owner first.  Plans are forced
with EMU_SPLIT_K so that the test, not the library, fixes the split.  Every
element must carry the same bits.

A REGRESSION LOCK, not parity evidence: the model's alignment reference and
final rounding were fitted to this kernel's output, and its stage length,
issue order and owner map are the kernel's own schedule.  It pins the
kernel's current bits (any change to its arithmetic or order shows here);
the parity claim rests on the plain oracle and tolerances (_gpu.compare).
"""
import numpy as np
import pytest

import oracle
from fp32_emulated_gemm_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
MODES = ["bf16x9", "tf32x3", "bf16x6", "tf32x1"]


def _same_bits(got, want):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    diff = got.view(np.uint32) != want.view(np.uint32)
    assert not diff.any(), f"{int(diff.sum())} of {diff.size} elements differ, e.g. {got[diff][:3]} vs {want[diff][:3]}"


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("pieces", [1, 3])
@pytest.mark.parametrize("tA,tB", [(False, False), (True, True)])
def test_sgemm_matches_tensor_core_model(mode, pieces, tA, tB, monkeypatch):
    monkeypatch.setenv("EMU_SPLIT_K", str(pieces))
    rng = np.random.default_rng(21)
    M, N, K = 300, 260, 200                       # ragged in every dimension, 7 k-stages
    A = rng.standard_normal((K, M) if tA else (M, K)).astype(np.float32)
    B = rng.standard_normal((N, K) if tB else (K, N)).astype(np.float32)
    Cold = rng.standard_normal((M, N)).astype(np.float32)
    C = _gpu.gpu_sgemm(mode, A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    p = oracle.Problem(A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    _same_bits(C, oracle.gemm_tc(p, mode=mode, pieces=pieces))


@pytest.mark.parametrize("mode", MODES)
def test_wide_magnitudes_match_tensor_core_model(mode, monkeypatch):
    """Entries 2^u, u uniform in [-20, 20], random sign: alignment and
    truncation decide many bits."""
    monkeypatch.setenv("EMU_SPLIT_K", "1")
    rng = np.random.default_rng(22)
    M, N, K = 256, 256, 160
    A = (rng.choice([-1.0, 1.0], (M, K)) * 2.0 ** rng.uniform(-20, 20, (M, K))).astype(np.float32)
    B = (rng.choice([-1.0, 1.0], (K, N)) * 2.0 ** rng.uniform(-20, 20, (K, N))).astype(np.float32)
    _same_bits(_gpu.gpu_sgemm(mode, A, B), oracle.gemm_tc(oracle.Problem(A, B), mode=mode))


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_pet_small_layer_matches_tensor_core_model(mode, monkeypatch):
    """The PET-small forward (with bias) and input gradient, one plan without
    a split, on a sample of rows that covers every tile row."""
    import fp32_emulated_gemm_gb300 as emu
    monkeypatch.setenv("EMU_SPLIT_K", "1")
    s = W.PET_SMALL
    X, Wt, b, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    rows = W.sample_rows(s.M, every=97, edge=4)
    Y = emu.linear_fwd(_gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b), mode=mode)
    dX = emu.linear_bwd_input(_gpu.to_dev(dY), _gpu.to_dev(Wt), mode=mode)
    assert emu.emu_stream_check() == 0
    _same_bits(Y.cpu().numpy()[rows], oracle.gemm_tc(oracle.Problem(X, Wt, transB=True, bias=b), mode=mode, rows=rows))
    _same_bits(dX.cpu().numpy()[rows], oracle.gemm_tc(oracle.Problem(dY, Wt), mode=mode, rows=rows))


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_multiwave_split_plan_matches_tensor_core_model(mode, monkeypatch):
    """96 units of a forced 4-way split on 76 pairs: two waves of split
    tiles, so some pairs reduce a split tile and then go on to another unit.
    Rows sampled from every tile row."""
    import fp32_emulated_gemm_gb300 as emu
    monkeypatch.setenv("EMU_SPLIT_K", "4")
    M, N, K = 1536, 1024, 512
    plan = emu.emu_plan_query(M, N, K, 76)
    assert plan["split_a"] == 4 and plan["units"] > plan["pairs"]
    rng = np.random.default_rng(24)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    rows = W.sample_rows(M, every=61, edge=2)
    C = _gpu.gpu_sgemm(mode, A, B)
    _same_bits(C[rows], oracle.gemm_tc(oracle.Problem(A, B), mode=mode, rows=rows, pieces=4))


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_hybrid_plan_matches_tensor_core_model(mode, monkeypatch):
    """The hybrid plan for the PET-small forward pass (the library chains
    this product by default; EMU_CHAIN=0 gives the plan it would take
    otherwise): whole tiles in the first wave, the tail tiles split.  Rows of
    whole tiles follow the unsplit model, rows of tail tiles the split one."""
    import fp32_emulated_gemm_gb300 as emu
    monkeypatch.setenv("EMU_CHAIN", "0")
    s = W.PET_SMALL
    plan = emu.emu_plan_query(s.M, s.N, s.K, 76)
    assert plan["split_a"] == 1 and plan["split_b"] > 1 and plan["tiles_a"] % plan["tiles_n"] == 0
    first_split_row = plan["tiles_a"] // plan["tiles_n"] * 256
    X, Wt, b, _ = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    Y = emu.linear_fwd(_gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b), mode=mode)
    assert emu.emu_stream_check() == 0
    Y = Y.cpu().numpy()
    rows = W.sample_rows(s.M, every=89, edge=3)
    p = oracle.Problem(X, Wt, transB=True, bias=b)
    whole, tail = rows[rows < first_split_row], rows[rows >= first_split_row]
    assert len(whole) and len(tail)
    _same_bits(Y[whole], oracle.gemm_tc(p, mode=mode, rows=whole, pieces=1))
    _same_bits(Y[tail], oracle.gemm_tc(p, mode=mode, rows=tail, pieces=plan["split_b"]))


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_many_piece_split_matches_tensor_core_model(mode, monkeypatch):
    """16 pieces per tile: few warps own chunks, so the owners read the other
    pieces' partials through the output staging area, several at once; the
    sum order (owner first, then increasing piece) is unchanged."""
    monkeypatch.setenv("EMU_SPLIT_K", "16")
    rng = np.random.default_rng(25)
    M, N, K = 300, 260, 2048
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    rows = W.sample_rows(M, every=37, edge=2)
    C = _gpu.gpu_sgemm(mode, A, B)
    _same_bits(C[rows], oracle.gemm_tc(oracle.Problem(A, B), mode=mode, rows=rows, pieces=16))


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_weight_gradient_plan_matches_tensor_core_model(mode):
    """The PET-small weight gradient with the library's own plan (4 tiles in
    18 pieces), bit for bit against the model on sampled rows of dW."""
    import fp32_emulated_gemm_gb300 as emu
    s = W.PET_SMALL
    plan = emu.emu_plan_query(s.N, s.K, s.M, 76)
    assert plan["split_a"] >= 12
    X, _, _, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    dW = emu.linear_bwd_weight(_gpu.to_dev(dY), _gpu.to_dev(X), mode=mode)
    assert emu.emu_stream_check() == 0
    rows = W.sample_rows(s.N, every=97, edge=2)
    want = oracle.gemm_tc(oracle.Problem(dY, X, transA=True), mode=mode, rows=rows, pieces=plan["split_a"])
    _same_bits(dW.cpu().numpy()[rows], want)


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
@pytest.mark.parametrize("pipe", ["0", "1"])
def test_one_owner_split_matches_tensor_core_model(mode, pipe, monkeypatch):
    """32 pieces: every piece owns exactly one 32-column chunk, so one warp per
    CTA reduces and borrows all of the staging area (both pipeline shapes:
    8 or 4 blocks of 4 KB)."""
    monkeypatch.setenv("EMU_SPLIT_K", "32")
    monkeypatch.setenv("EMU_PIPE", pipe)
    rng = np.random.default_rng(27)
    M, N, K = 250, 200, 4096
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    rows = W.sample_rows(M, every=41, edge=2)
    C = _gpu.gpu_sgemm(mode, A, B)
    _same_bits(C[rows], oracle.gemm_tc(oracle.Problem(A, B), mode=mode, rows=rows, pieces=32))

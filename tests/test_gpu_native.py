"""Native FP32 (EMU_MODE_FP32) and the performant strategy on the GPU.

The native path computes each output as one chain of fmaf over k in
ascending order, then the epilogue, which is the oracle's plain FP32 SGEMM
by definition, so every element must carry the same bits.  Under the
performant strategy a small product requested in an emulated mode must give
the native bits, and a large one the emulated bits of the eager strategy.
"""
import numpy as np
import pytest

import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu


def _same_bits(got, want):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    diff = got.view(np.uint32) != want.view(np.uint32)
    assert not diff.any(), f"{int(diff.sum())} of {diff.size} elements differ, e.g. {got[diff][:3]} vs {want[diff][:3]}"


@pytest.mark.parametrize("tA,tB", [(False, False), (True, False), (False, True), (True, True)])
# micro-tiles: 1 x 1 per thread for the small outputs, 2 x 2 for (1030, 645),
# 4 x 4 for (2050, 1283) (the library picks the largest that fills the SMs)
@pytest.mark.parametrize("M,N,K", [(300, 260, 200), (64, 1000, 37), (130, 70, 1), (65, 64, 16), (1, 5, 1000),
                                   (1030, 645, 45), (2050, 1283, 40)])
def test_native_fp32_matches_oracle_bitwise(tA, tB, M, N, K):
    rng = np.random.default_rng(41)
    A = rng.standard_normal((K, M) if tA else (M, K)).astype(np.float32)
    B = rng.standard_normal((N, K) if tB else (K, N)).astype(np.float32)
    Cold = rng.standard_normal((M, N)).astype(np.float32)
    C = _gpu.gpu_sgemm("fp32", A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    p = oracle.Problem(A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    _same_bits(C, oracle.sgemm_f32(p))
    # beta == 0 never reads C (the helper fills it with NaN)
    _same_bits(_gpu.gpu_sgemm("fp32", A, B, transA=tA, transB=tB),
               oracle.sgemm_f32(oracle.Problem(A, B, transA=tA, transB=tB)))


def test_native_fp32_order_and_fusion():
    """Cases whose bits depend on the order of the k-chain and on fusing the
    multiply into the add (k ascending, one rounding per step)."""
    A = np.array([[2.0 ** 24, 1.0, -2.0 ** 24], [-(1 + 2.0 ** -11), 1 + 2.0 ** -12, 0.0]], np.float32)
    B = np.array([[1.0, 1.0], [1.0, 1 + 2.0 ** -12], [1.0, 0.0]], np.float32)
    C = _gpu.gpu_sgemm("fp32", A, B)
    assert C[0, 0] == 0.0 and C[1, 1] == 2.0 ** -24
    _same_bits(C, oracle.sgemm_f32(oracle.Problem(A, B)))


def test_native_linear_layer_matches_oracle_bitwise():
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(42)
    M, N, K = 333, 100, 72
    X = rng.standard_normal((M, K)).astype(np.float32)
    Wt = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    dY = rng.standard_normal((M, N)).astype(np.float32)
    dW0 = rng.standard_normal((N, K)).astype(np.float32)
    Y = emu.linear_fwd(_gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b), mode="fp32")
    dX = emu.linear_bwd_input(_gpu.to_dev(dY), _gpu.to_dev(Wt), mode="fp32")
    dW = emu.linear_bwd_weight(_gpu.to_dev(dY), _gpu.to_dev(X), mode="fp32", out=_gpu.to_dev(dW0), beta=1.0)
    assert emu.emu_stream_check() == 0
    _same_bits(Y.cpu().numpy(), oracle.sgemm_f32(oracle.Problem(X, Wt, transB=True, bias=b)))
    _same_bits(dX.cpu().numpy(), oracle.sgemm_f32(oracle.Problem(dY, Wt)))
    _same_bits(dW.cpu().numpy(), oracle.sgemm_f32(oracle.Problem(dY, X, transA=True, beta=1.0, C_old=dW0)))


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_performant_strategy_small_native_large_emulated(mode):
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(43)
    small, large = (192, 256, 256), (2048, 1536, 512)
    out = {}
    for name, (M, N, K) in (("small", small), ("large", large)):
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        eager = _gpu.gpu_sgemm(mode, A, B)
        with emu.strategy("performant"):
            chosen = emu.emu_dispatch_query(mode, M, N, K)
            perf = _gpu.gpu_sgemm(mode, A, B)
        out[name] = chosen
        if chosen == "fp32":
            _same_bits(perf, oracle.sgemm_f32(oracle.Problem(A, B)))
        else:
            _same_bits(perf, eager)
    assert out == {"small": "fp32", "large": mode}
    assert emu.emu_get_strategy() == "eager"


def test_packed_calls_reject_native_mode():
    import torch
    import fp32_emulated_gemm_gb300 as emu
    B = torch.zeros((64, 64), device="cuda")
    with pytest.raises((emu.EmuError, KeyError, ValueError)):
        emu.pack_b(B, mode="fp32")


def test_emu_linear_module_in_native_mode():
    """EmuLinear with mode="fp32": forward and input gradient are the native
    kernel's (bit-identical to the oracle's SGEMM); prepack has no packed
    form to use and is ignored."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    torch.manual_seed(5)
    layer = emu.EmuLinear(72, 40, mode="fp32", prepack=True).cuda()
    x = torch.randn(130, 72, device="cuda", requires_grad=True)
    y = layer(x)
    g = torch.randn_like(y)
    y.backward(g)
    assert emu.emu_stream_check() == 0
    W = layer.weight.detach().cpu().numpy()
    b = layer.bias.detach().cpu().numpy()
    X = x.detach().cpu().numpy()
    _same_bits(y.detach().cpu().numpy(), oracle.sgemm_f32(oracle.Problem(X, W, transB=True, bias=b)))
    _same_bits(x.grad.cpu().numpy(), oracle.sgemm_f32(oracle.Problem(g.cpu().numpy(), W)))


def test_native_degenerate_and_narrow_sizes():
    """The native mode's edge cases: M or N = 0 (no-op), K = 0 (C = beta C),
    alpha = 0 with beta = 0 (NaN in C and the operands ignored), a linear
    layer with K = 0 (Y = bias), and 1 x 1 x 1, single rows and columns."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    fp32 = emu.MODES["fp32"]
    dev = _gpu.device()
    C = torch.full((4, 4), 7.0, device=dev)
    emu.emu_sgemm(fp32, 0, 0, 0, 4, 4, 1.0, C, 4, C, 4, 0.0, C, 4)
    emu.emu_sgemm(fp32, 0, 0, 4, 0, 4, 1.0, C, 4, C, 4, 0.0, C, 4)
    assert emu.emu_stream_check() == 0 and torch.all(C == 7.0)
    Cold = torch.arange(16, dtype=torch.float32, device=dev).reshape(4, 4)
    C = Cold.clone()
    emu.emu_sgemm(fp32, 0, 0, 4, 4, 0, 1.0, C, 4, C, 4, 2.0, C, 4)
    assert emu.emu_stream_check() == 0 and torch.equal(C, 2 * Cold)
    A = torch.full((4, 8), float("nan"), device=dev)
    C = torch.full((4, 4), float("nan"), device=dev)
    emu.emu_sgemm(fp32, 0, 0, 4, 4, 8, 0.0, A, 8, A, 8, 0.0, C, 4)
    assert emu.emu_stream_check() == 0 and torch.all(C == 0)
    b = torch.arange(4, dtype=torch.float32, device=dev)
    Y = torch.full((3, 4), float("nan"), device=dev)
    emu.emu_linear_fwd(fp32, 3, 4, 0, Y, Y, b, Y)
    assert emu.emu_stream_check() == 0 and torch.equal(Y, b.expand(3, 4))
    rng = np.random.default_rng(44)
    for (M, N, K) in [(1, 1, 1), (1, 300, 64), (257, 1, 64), (130, 130, 1), (4, 4, 4)]:
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        _same_bits(_gpu.gpu_sgemm("fp32", A, B), oracle.sgemm_f32(oracle.Problem(A, B)))

"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances: normwise max|C - C64| / (|alpha||A||B| + |beta||C| + |bias|)
<= 2 K 2^-24 for BF16x9 and 4 K 2^-24 for TF32x3, and elementwise agreement
with the oracle's own emulated result within 1e-5 relative (floored at the
rms of the result, because accumulation orders differ).
"""
import numpy as np
import pytest

import oracle
from fp32_emulated_gemm_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
MODES = ["bf16x9", "tf32x3"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_tiny_config(mode, beta):
    """M=N=128, K=256, U[-1,1] from seed 0; beta = 0 and beta = 1."""
    A, B, Cold = W.tiny_inputs()
    C = _gpu.gpu_sgemm(mode, A, B, beta=beta, C_old=Cold)
    _gpu.compare(mode, C, oracle.Problem(A, B, beta=beta, C_old=Cold if beta else None))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tA,tB", [(False, False), (True, False), (False, True), (True, True)])
def test_ragged_all_layouts(mode, tA, tB):
    """Several tiles and a ragged tail in M, N and K, every storage order."""
    rng = np.random.default_rng(7)
    M, N, K = 300, 260, 200
    A_op = rng.standard_normal((M, K)).astype(np.float32)
    B_op = rng.standard_normal((K, N)).astype(np.float32)
    A = np.ascontiguousarray(A_op.T) if tA else A_op
    B = np.ascontiguousarray(B_op.T) if tB else B_op
    Cold = rng.standard_normal((M, N)).astype(np.float32)
    C = _gpu.gpu_sgemm(mode, A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold)
    _gpu.compare(mode, C, oracle.Problem(A, B, transA=tA, transB=tB, alpha=0.75, beta=-0.5, C_old=Cold))


@pytest.mark.parametrize("mode", MODES)
def test_split_dump_bit_exact(mode):
    """The kernels' split, dumped from shared memory, equals the oracle's
    split bit for bit (components in natural magnitude: the oracle's scaled
    component i times 2^-8i), for the K-major and the transposing path."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(3)
    R, Kc = 128, 32
    # random sign, exponent in [-60, 60], full fraction: every component used
    sign = rng.integers(0, 2, R * Kc, dtype=np.uint32) << np.uint32(31)
    ex = (rng.integers(-60, 61, R * Kc) + 127).astype(np.uint32) << np.uint32(23)
    fr = rng.integers(0, 1 << 23, R * Kc, dtype=np.uint32)
    X = (sign | ex | fr).view(np.float32).reshape(R, Kc)
    ncomp = 3 if mode == "bf16x9" else 2
    for mn_major in (0, 1):
        src = np.ascontiguousarray(X.T) if mn_major else X
        ld = src.shape[1]
        out = torch.zeros(ncomp * R * Kc * (2 if mode == "bf16x9" else 4), dtype=torch.uint8, device=_gpu.device())
        emu.emu_split_dump(emu.MODES[mode], R, Kc, _gpu.to_dev(src), ld, mn_major, out)
        assert emu.emu_stream_check() == 0
        raw = out.cpu().numpy()
        if mode == "bf16x9":
            got = raw.view(np.uint16).reshape(3, R * Kc)
            c = oracle.split_bf16x9_f32(X.ravel())
            for i in range(3):
                want = (c[i].astype(np.float64) * 2.0 ** (-8 * i)).astype(np.float32)
                assert np.array_equal(got[i], (want.view(np.uint32) >> 16).astype(np.uint16)), (mn_major, i)
        else:
            got = raw.view(np.uint32).reshape(2, R * Kc)
            hi, lo = oracle.split_tf32x3(X.ravel())
            assert np.array_equal(got[0], hi.view(np.uint32)), mn_major
            assert np.array_equal(got[1], lo.view(np.uint32)), mn_major


@pytest.mark.parametrize("mode", MODES)
def test_pet_small_forward_and_input_gradient(mode):
    """M=6144, K=256, N=1024 forward with bias, then dX = dY W; X ~ N(0,1),
    W ~ N(0,1/K), b ~ N(0,0.01), dY ~ N(0,1); checked on a row sample."""
    import fp32_emulated_gemm_gb300 as emu
    s = W.PET_SMALL
    X, Wt, b, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    rows = W.sample_rows(s.M, every=16, edge=128)
    Y = emu.linear_fwd(_gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b), mode=mode)
    dX = emu.linear_bwd_input(_gpu.to_dev(dY), _gpu.to_dev(Wt), mode=mode)
    assert emu.emu_stream_check() == 0
    _gpu.compare(mode, Y.cpu().numpy(), oracle.Problem(X, Wt, transB=True, bias=b), rows)
    _gpu.compare(mode, dX.cpu().numpy(), oracle.Problem(dY, Wt), rows)


@pytest.mark.parametrize("mode", MODES)
def test_degenerate_sizes(mode):
    import torch
    import fp32_emulated_gemm_gb300 as emu
    dev = _gpu.device()
    # M == 0 and N == 0: no-op
    C = torch.full((4, 4), 7.0, device=dev)
    emu.emu_sgemm(emu.MODES[mode], 0, 0, 0, 4, 4, 1.0, C, 4, C, 4, 0.0, C, 4)
    emu.emu_sgemm(emu.MODES[mode], 0, 0, 4, 0, 4, 1.0, C, 4, C, 4, 0.0, C, 4)
    assert emu.emu_stream_check() == 0 and torch.all(C == 7.0)
    # K == 0: C = beta C
    Cold = torch.arange(16, dtype=torch.float32, device=dev).reshape(4, 4)
    C = Cold.clone()
    emu.emu_sgemm(emu.MODES[mode], 0, 0, 4, 4, 0, 1.0, C, 4, C, 4, 2.0, C, 4)
    assert emu.emu_stream_check() == 0 and torch.equal(C, 2 * Cold)
    # alpha == 0 with beta == 0 ignores NaN in C and in the operands
    A = torch.full((4, 8), float("nan"), device=dev)
    C = torch.full((4, 4), float("nan"), device=dev)
    emu.emu_sgemm(emu.MODES[mode], 0, 0, 4, 4, 8, 0.0, A, 8, A, 8, 0.0, C, 4)
    assert emu.emu_stream_check() == 0 and torch.all(C == 0)
    # linear layer with K == 0: Y = bias
    b = torch.arange(4, dtype=torch.float32, device=dev)
    Y = torch.full((3, 4), float("nan"), device=dev)
    emu.emu_linear_fwd(emu.MODES[mode], 3, 4, 0, Y, Y, b, Y)
    assert emu.emu_stream_check() == 0 and torch.equal(Y, b.expand(3, 4))


@pytest.mark.parametrize("mode", MODES)
def test_single_element_and_narrow(mode):
    """1 x 1 x 1, a single row, a single column and K = 1."""
    rng = np.random.default_rng(5)
    for (M, N, K) in [(1, 1, 1), (1, 300, 64), (257, 1, 64), (130, 130, 1), (4, 4, 4)]:
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        C = _gpu.gpu_sgemm(mode, A, B)
        _gpu.compare(mode, C, oracle.Problem(A, B))


def test_invalid_arguments_return_status():
    import torch
    import fp32_emulated_gemm_gb300 as emu
    dev = _gpu.device()
    X = torch.zeros((8, 8), device=dev)
    with pytest.raises(emu.EmuError) as e:
        emu.emu_sgemm(0, 0, 0, -1, 8, 8, 1.0, X, 8, X, 8, 0.0, X, 8)
    assert e.value.status == 1
    with pytest.raises(emu.EmuError) as e:
        emu.emu_sgemm(0, 0, 0, 8, 8, 8, 1.0, X, 6, X, 8, 0.0, X, 8)  # lda < K
    assert e.value.status == 1
    with pytest.raises(emu.EmuError) as e:  # misaligned A (4-byte offset)
        emu.emu_sgemm(0, 0, 0, 4, 4, 4, 1.0, X.view(-1)[1:], 8, X, 8, 0.0, X, 8)
    assert e.value.status == 2
    with pytest.raises(emu.EmuError) as e:
        emu.emu_sgemm(7, 0, 0, 8, 8, 8, 1.0, X, 8, X, 8, 0.0, X, 8)
    assert e.value.status == 1
    assert emu.emu_stream_check() == 0


def test_bounded_wait_reports_timeout_and_context_survives():
    """A kernel wait that runs out (a barrier nothing completes) records
    EMU_STATUS_DEVICE_TIMEOUT instead of hanging; the CUDA context stays
    usable and the flag clears after it is reported."""
    import ctypes
    import torch
    import fp32_emulated_gemm_gb300 as emu
    lib = emu.load()
    lib.emu_selftest_wait_timeout.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    lib.emu_selftest_wait_timeout.restype = ctypes.c_int
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert emu.emu_stream_check() == 0
    assert lib.emu_selftest_wait_timeout(2_000_000, stream) == 0  # 2 ms budget
    assert emu.emu_stream_check() == 6  # EMU_STATUS_DEVICE_TIMEOUT
    assert emu.emu_stream_check() == 0  # reported once, then cleared
    # the context still computes correctly
    A, B, Cold = W.tiny_inputs()
    C = _gpu.gpu_sgemm("bf16x9", A, B)
    _gpu.compare("bf16x9", C, oracle.Problem(A, B))


@pytest.mark.parametrize("mode", MODES)
def test_weight_gradient(mode):
    """dW = dY^T X (+ beta dW) for the PET-small layer: the contraction runs
    over the 6144 tokens (split into several k-pieces); beta = 1 accumulates."""
    import fp32_emulated_gemm_gb300 as emu
    s = W.PET_SMALL
    X, _, _, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    rows = W.sample_rows(s.N, every=37, edge=8)
    dW = emu.linear_bwd_weight(_gpu.to_dev(dY), _gpu.to_dev(X), mode=mode)
    assert emu.emu_stream_check() == 0
    dW_h = dW.cpu().numpy()
    _gpu.compare(mode, dW_h, oracle.Problem(dY, X, transA=True), rows)
    old = np.random.default_rng(9).standard_normal(dW_h.shape).astype(np.float32)
    dW2 = emu.linear_bwd_weight(_gpu.to_dev(dY), _gpu.to_dev(X), mode=mode, out=_gpu.to_dev(old), beta=1.0)
    assert emu.emu_stream_check() == 0
    _gpu.compare(mode, dW2.cpu().numpy(), oracle.Problem(dY, X, transA=True, beta=1.0, C_old=old), rows)


def test_emu_linear_module_matches_fp32_layer():
    """EmuLinear (forward, input gradient, optional emulated weight gradient)
    against the same layer in float64 torch on the CPU."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    torch.manual_seed(0)
    for wg in ("fp32", "emulated"):
        lin = emu.EmuLinear(256, 512, mode="bf16x9", weight_grad=wg).cuda()
        x = torch.randn(3, 700, 256, device="cuda", requires_grad=True)
        y = lin(x)
        g = torch.randn_like(y)
        y.backward(g)
        ref = torch.nn.Linear(256, 512).double()
        with torch.no_grad():
            ref.weight.copy_(lin.weight.double().cpu())
            ref.bias.copy_(lin.bias.double().cpu())
        xr = x.detach().double().cpu().requires_grad_(True)
        yr = ref(xr)
        yr.backward(g.double().cpu())
        scale = lambda t: float(t.abs().max())
        assert float((y.detach().double().cpu() - yr).abs().max()) <= 1e-5 * scale(yr)
        assert float((x.grad.double().cpu() - xr.grad).abs().max()) <= 1e-5 * scale(xr.grad)
        assert float((lin.weight.grad.double().cpu() - ref.weight.grad).abs().max()) <= 1e-5 * scale(ref.weight.grad)
        assert float((lin.bias.grad.double().cpu() - ref.bias.grad).abs().max()) <= 1e-5 * scale(ref.bias.grad)


@pytest.mark.parametrize("mode", ["tf32x1", "bf16x6"])
def test_comparator_modes(mode):
    """The comparators (one-pass TF32, BF16x6) against their oracles: the
    tiny config with beta, a ragged problem in every storage order, and the
    PET-small forward and input gradient on a row sample."""
    import fp32_emulated_gemm_gb300 as emu
    A, B, Cold = W.tiny_inputs()
    C = _gpu.gpu_sgemm(mode, A, B, beta=1.0, C_old=Cold)
    _gpu.compare(mode, C, oracle.Problem(A, B, beta=1.0, C_old=Cold))
    rng = np.random.default_rng(8)
    M, N, K = 300, 260, 200
    A_op = rng.standard_normal((M, K)).astype(np.float32)
    B_op = rng.standard_normal((K, N)).astype(np.float32)
    for tA, tB in [(False, False), (True, False), (False, True), (True, True)]:
        Am = np.ascontiguousarray(A_op.T) if tA else A_op
        Bm = np.ascontiguousarray(B_op.T) if tB else B_op
        C = _gpu.gpu_sgemm(mode, Am, Bm, transA=tA, transB=tB)
        _gpu.compare(mode, C, oracle.Problem(Am, Bm, transA=tA, transB=tB))
    s = W.PET_SMALL
    X, Wt, b, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    rows = W.sample_rows(s.M, every=32, edge=64)
    Y = emu.linear_fwd(_gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b), mode=mode)
    dX = emu.linear_bwd_input(_gpu.to_dev(dY), _gpu.to_dev(Wt), mode=mode)
    assert emu.emu_stream_check() == 0
    _gpu.compare(mode, Y.cpu().numpy(), oracle.Problem(X, Wt, transB=True, bias=b), rows)
    _gpu.compare(mode, dX.cpu().numpy(), oracle.Problem(dY, Wt), rows)


@pytest.mark.parametrize("mode", MODES)
def test_split_k_plans_match_oracle_and_repeat_bitwise(mode, monkeypatch):
    """A long-k, few-tile GEMM under forced split-K plans (the pieces of a
    tile reduce-scatter their partials through the workspace): every plan
    meets the tolerances, and each plan gives the same bits on every run
    (the sum order is fixed by the plan, not by which piece finishes first)."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(11)
    M, N, K = 300, 260, 3000          # 2 x 2 tiles, ragged edges, 94 k-stages
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = (rng.standard_normal((K, N)) / np.sqrt(K)).astype(np.float32)
    Ad, Bd = _gpu.to_dev_padded(A, float("nan")), _gpu.to_dev_padded(B, float("nan"))
    noise = torch.empty(1 << 22, device=_gpu.device())
    for S in ("1", "2", "3", "7"):
        monkeypatch.setenv("EMU_SPLIT_K", S)
        runs = []
        for rep in range(3):
            noise.uniform_()  # other work on the GPU between runs
            C = emu.sgemm(Ad, Bd, mode=mode)
            assert emu.emu_stream_check() == 0
            runs.append(C.cpu().numpy())
        for r in runs[1:]:
            assert np.array_equal(r.view(np.uint32), runs[0].view(np.uint32)), f"split {S} not repeatable"
        _gpu.compare(mode, runs[0], oracle.Problem(A, B))

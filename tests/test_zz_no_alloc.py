"""emu_sgemm_noalloc: the GEMM for callers that cannot allocate device memory.

Some callers cannot let a library call cudaMalloc: applications that give all
device memory to their own pre-sized pool, latency-critical loops that must
not enter the driver's allocator, code that must never hit an out-of-memory
error mid-run.  For them the library offers emu_sgemm_noalloc, whose split-K
scratch is a fixed 64 MiB device array inside the library.

These tests call it through the C ABI and compare it with emu_sgemm (same
kernel, same plan, so the same bits: asserted bit for bit, which also covers
the tolerance the other GPU tests use), on two calls in a row (the shared
array keeps the previous call's contents).  This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
from fp32_emulated_gemm_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

NOT_SUPPORTED = 2


def _noalloc():
    import fp32_emulated_gemm_gb300 as emu
    f = emu.load().emu_sgemm_noalloc
    i64, i32, f32, P = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    f.argtypes = [i32, i32, i32, i64, i64, i64, f32, P, i64, P, i64, f32, P, i64, P]
    f.restype = i32
    return f


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
@pytest.mark.parametrize("case", ["split_k", "single_piece", "chained"])
def test_noalloc_matches_emu_sgemm_on_two_calls(mode, case):
    import torch
    import fp32_emulated_gemm_gb300 as emu
    if case == "chained":
        # 96 tiles of 8 k-stages on 76 pairs: a chained plan, whose cut tiles
        # pass their running sums through the scratch array
        M, N, K = 6144, 1024, 256
        assert emu.emu_plan_query(M, N, K, 76)["chain"] == 1
        rng = np.random.default_rng(23)
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
    elif case == "split_k":
        # input gradient of the PET-small layer: 24 tiles, K split into 3 pieces
        s = W.PET_SMALL
        _, Wt, _, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
        A, B = dY, Wt  # dX[M, K] = dY[M, N] W[N, K]
        M, N, K = s.M, s.K, s.N
    else:
        rng = np.random.default_rng(21)
        M, N, K = 300, 260, 200
        A = rng.standard_normal((M, K)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
    Ad, Bd = _gpu.to_dev(A), _gpu.to_dev(B)
    ref = torch.empty((M, N), device=_gpu.device())
    emu.emu_sgemm(emu.MODES[mode], 0, 0, M, N, K, 1.0, Ad, A.shape[1], Bd, B.shape[1], 0.0, ref, N)
    assert emu.emu_stream_check() == 0
    ref_h = ref.cpu().numpy()
    f = _noalloc()
    for call in range(2):
        out = torch.full((M, N), float("nan"), device=_gpu.device())
        st = f(emu.MODES[mode], 0, 0, M, N, K, 1.0, ctypes.c_void_p(Ad.data_ptr()), A.shape[1],
               ctypes.c_void_p(Bd.data_ptr()), B.shape[1], 0.0, ctypes.c_void_p(out.data_ptr()), N, _stream())
        assert st == 0, emu.emu_status_string(st)
        assert emu.emu_stream_check() == 0
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        assert np.array_equal(got.view(np.uint32), ref_h.view(np.uint32)), f"call {call}: bits differ from emu_sgemm"
        ex = oracle.elementwise_excess(got, ref_h)
        assert ex <= 1.0, f"call {call}: differs from emu_sgemm beyond 1e-5 relative (excess {ex:.3f})"
    # and against the float64 oracle on a row sample, like the other tests
    rows = W.sample_rows(M, every=97, edge=16)
    _gpu.compare(mode, got, oracle.Problem(A, B), rows, elementwise=False)


def test_noalloc_rejects_plans_beyond_its_scratch(monkeypatch):
    """Automatic plans keep split tiles to one wave of units (at most one
    partial tile per CTA pair, about 19 MiB), so a plan beyond the 64 MiB
    array is forced here: the wide-model input gradient (96 tiles, 128
    k-stages) with every tile split into 32 pieces needs 768 MiB of partial
    tiles.  The call is refused with EMU_STATUS_NOT_SUPPORTED and enqueues
    nothing."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    dev = _gpu.device()
    monkeypatch.setenv("EMU_SPLIT_K", "32")
    M, N, K = 6144, 1024, 4096  # dX = dY[6144, 4096] W[4096, 1024]
    A = torch.zeros((M, K), device=dev)
    B = torch.zeros((K, N), device=dev)
    C = torch.full((M, N), 7.0, device=dev)
    st = _noalloc()(0, 0, 0, M, N, K, 1.0, ctypes.c_void_p(A.data_ptr()), K, ctypes.c_void_p(B.data_ptr()), N,
                    0.0, ctypes.c_void_p(C.data_ptr()), N, _stream())
    assert st == NOT_SUPPORTED
    assert emu.emu_stream_check() == 0
    assert torch.all(C == 7.0)


def test_noalloc_follows_the_performant_strategy():
    """Under the performant strategy a small product requested in an emulated
    mode runs in native FP32 here too: the native kernel's bits, equal to the
    oracle's sequential SGEMM."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(26)
    M, N, K = 192, 256, 256
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    Ad, Bd = _gpu.to_dev(A), _gpu.to_dev(B)
    out = torch.full((M, N), float("nan"), device=_gpu.device())
    with emu.strategy("performant"):
        assert emu.emu_dispatch_query("bf16x9", M, N, K) == "fp32"
        st = _noalloc()(emu.MODES["bf16x9"], 0, 0, M, N, K, 1.0, ctypes.c_void_p(Ad.data_ptr()), K,
                        ctypes.c_void_p(Bd.data_ptr()), N, 0.0, ctypes.c_void_p(out.data_ptr()), N, _stream())
    assert st == 0, emu.emu_status_string(st)
    assert emu.emu_stream_check() == 0
    got = out.cpu().numpy()
    want = oracle.sgemm_f32(oracle.Problem(A, B))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))

"""Failure paths on the GPU, made without faulting it: a split-K wait that
runs out, the release of the library's buffers, and allocations that fail.

Every wait in the kernels is bounded; a timeout is recorded in a device flag
(EMU_STATUS_DEVICE_TIMEOUT from emu_stream_check) and the kernel returns.
The split-K pieces count their arrivals on counters tagged with a per-launch
epoch, so the counts a timed-out launch leaves behind cannot be taken for a
later launch's: the tests below leave such counts on every tile and then
require the next split launch's bits.  Allocation failures are injected on
the host (emu_debug_fail_allocations), never provoked on the device.
"""
import numpy as np
import pytest

import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 6
ALLOC_FAILED = 4


def _problem(seed, M=300, N=260, K=3000):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = (rng.standard_normal((K, N)) / np.sqrt(K)).astype(np.float32)
    return A, B


def _same_bits(got, want):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), \
        f"{int((got.view(np.uint32) != want.view(np.uint32)).sum())} elements differ"


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
@pytest.mark.parametrize("pieces", [2, 3])
def test_split_launch_after_a_split_timeout_is_correct(mode, pieces, monkeypatch):
    """A split launch leaves partial tiles in the stream's workspace; then
    every counter of the workspace gets one arrival and a wait for the second
    runs out (2 ms), as when a piece's partners are lost.  The next split
    launch on the same stream must give the bits it gives on a clean
    workspace and meet the tolerances."""
    import fp32_emulated_gemm_gb300 as emu
    monkeypatch.setenv("EMU_SPLIT_K", str(pieces))
    A, B = _problem(41)
    A_other, B_other = _problem(42)
    Ad, Bd = _gpu.to_dev_padded(A, float("nan")), _gpu.to_dev_padded(B, float("nan"))
    ref = emu.sgemm(Ad, Bd, mode=mode).cpu().numpy()             # a clean run
    assert emu.emu_stream_check() == 0
    emu.sgemm(_gpu.to_dev(A_other), _gpu.to_dev(B_other), mode=mode)  # other partials left behind
    assert emu.emu_stream_check() == 0
    tiles = 2 * 2
    emu.emu_selftest_split_timeout(2_000_000, tiles)
    assert emu.emu_stream_check() == DEVICE_TIMEOUT
    assert emu.emu_stream_check() == 0                            # reported once
    C = emu.sgemm(Ad, Bd, mode=mode).cpu().numpy()
    assert emu.emu_stream_check() == 0
    _same_bits(C, ref)
    p = oracle.Problem(A, B)
    _same_bits(C, oracle.gemm_tc(p, mode=mode, pieces=pieces))
    _gpu.compare(mode, C, p, label=f"after split timeout, {pieces} pieces")


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_chained_launch_after_a_timeout_is_correct(mode, monkeypatch):
    """A chained plan (80 tiles on 76 pairs) waits for one arrival on a cut
    tile's counter before it reads the published running sum.  After a
    chained launch on other inputs and a timed-out wait that leaves one
    arrival on every counter, the next chained launch on the same stream must
    give the bits of the unsplit plan."""
    import fp32_emulated_gemm_gb300 as emu
    M, N, K = 2000, 2500, 200
    monkeypatch.setenv("EMU_CHAIN", "1")
    assert emu.emu_plan_query(M, N, K, 76)["chain"] == 1
    A, B = _problem(43, M, N, K)
    A_other, B_other = _problem(44, M, N, K)
    Ad, Bd = _gpu.to_dev(A), _gpu.to_dev(B)
    emu.sgemm(_gpu.to_dev(A_other), _gpu.to_dev(B_other), mode=mode)  # other running sums left behind
    assert emu.emu_stream_check() == 0
    emu.emu_selftest_split_timeout(2_000_000, 8 * 10)
    assert emu.emu_stream_check() == DEVICE_TIMEOUT
    C = emu.sgemm(Ad, Bd, mode=mode).cpu().numpy()
    assert emu.emu_stream_check() == 0
    monkeypatch.setenv("EMU_CHAIN", "0")
    monkeypatch.setenv("EMU_SPLIT_K", "1")
    _same_bits(C, emu.sgemm(Ad, Bd, mode=mode).cpu().numpy())
    rows = np.arange(0, M, 53)
    _gpu.compare(mode, C, oracle.Problem(A, B), rows, label="chained, after a timeout")


def test_shutdown_releases_buffers_and_later_calls_allocate_again(monkeypatch):
    """emu_shutdown frees every cached workspace and pre-split buffer; the
    next split call (and a TF32x3 call that pre-splits op(B)) allocates
    again and gives the same bits."""
    import fp32_emulated_gemm_gb300 as emu
    monkeypatch.setenv("EMU_SPLIT_K", "3")
    A, B = _problem(43)
    Ad, Bd = _gpu.to_dev(A), _gpu.to_dev(B)
    before = emu.sgemm(Ad, Bd, mode="bf16x9").cpu().numpy()
    monkeypatch.delenv("EMU_SPLIT_K")
    A2, B2 = _problem(44, M=1100, N=300, K=500)                   # 5 tile rows: op(B) pre-split in TF32x3
    A2d, B2d = _gpu.to_dev(A2), _gpu.to_dev(B2)
    before_tf = emu.sgemm(A2d, B2d, mode="tf32x3").cpu().numpy()
    assert emu.emu_stream_check() == 0
    emu.emu_shutdown()
    emu.emu_shutdown()                                            # nothing left: a no-op
    monkeypatch.setenv("EMU_SPLIT_K", "3")
    _same_bits(emu.sgemm(Ad, Bd, mode="bf16x9").cpu().numpy(), before)
    monkeypatch.delenv("EMU_SPLIT_K")
    _same_bits(emu.sgemm(A2d, B2d, mode="tf32x3").cpu().numpy(), before_tf)
    assert emu.emu_stream_check() == 0


@pytest.mark.parametrize("case", ["split_workspace", "presplit_buffer"])
def test_allocation_failure_returns_status_and_enqueues_nothing(case, monkeypatch):
    """With the library's next allocation made to fail, the call that needs
    it returns EMU_STATUS_ALLOC_FAILED and leaves C untouched; the next call
    allocates and computes normally."""
    import torch
    import fp32_emulated_gemm_gb300 as emu
    if case == "split_workspace":
        monkeypatch.setenv("EMU_SPLIT_K", "2")
        A, B = _problem(45)
        mode = "bf16x9"
    else:
        A, B = _problem(46, M=1100, N=300, K=500)
        mode = "tf32x3"
    M, N = A.shape[0], B.shape[1]
    Ad, Bd = _gpu.to_dev(A), _gpu.to_dev(B)
    emu.emu_shutdown()                                            # the call must allocate
    C = torch.full((M, N), 7.0, device=_gpu.device())
    emu.emu_debug_fail_allocations(1)
    try:
        with pytest.raises(emu.EmuError) as e:
            emu.sgemm(Ad, Bd, mode=mode, C=C)
        assert e.value.status == ALLOC_FAILED
    finally:
        emu.emu_debug_fail_allocations(0)
    assert emu.emu_stream_check() == 0
    assert torch.all(C == 7.0)
    emu.sgemm(Ad, Bd, mode=mode, C=C)
    assert emu.emu_stream_check() == 0
    _gpu.compare(mode, C.cpu().numpy(), oracle.Problem(A, B), rows=np.arange(0, M, 7),
                 label=f"after allocation failure ({case})")

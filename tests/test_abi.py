"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side checks answer without touching a GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

import fp32_emulated_gemm_gb300 as emu
from fp32_emulated_gemm_gb300 import build as emu_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "emu_gemm.h")


@pytest.fixture(scope="module")
def lib():
    emu_build.build()
    return ctypes.CDLL(emu_build.LIB)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(emu_\w+)\s*\(", text, flags=re.M)))


def _declared_enum(name_prefix):
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(rf"({name_prefix}\w+)\s*=\s*(\d+)", text)}


def test_header_declares_the_boundary():
    fns = _declared_functions()
    for required in ("emu_sgemm", "emu_linear_fwd", "emu_linear_bwd_input", "emu_status_string",
                     "emu_stream_check"):
        assert required in fns


def test_library_exports_every_declared_symbol(lib):
    fns = _declared_functions()
    assert fns
    for name in fns:
        assert hasattr(lib, name), f"{name} declared in emu_gemm.h but not exported"


def test_enums_match_binding():
    modes = _declared_enum("EMU_MODE_")
    assert modes == {"EMU_MODE_BF16X9": emu.EMU_MODE_BF16X9, "EMU_MODE_TF32X3": emu.EMU_MODE_TF32X3,
                     "EMU_MODE_TF32X1": emu.EMU_MODE_TF32X1, "EMU_MODE_BF16X6": emu.EMU_MODE_BF16X6,
                     "EMU_MODE_FP32": emu.EMU_MODE_FP32}
    assert {f"EMU_MODE_{k.upper()}": v for k, v in emu.MODES.items()} == modes
    ops = _declared_enum("EMU_OP_")
    assert ops == {"EMU_OP_N": emu.EMU_OP_N, "EMU_OP_T": emu.EMU_OP_T}
    strategies = _declared_enum("EMU_STRATEGY_")
    assert strategies == {"EMU_STRATEGY_EAGER": emu.EMU_STRATEGY_EAGER,
                          "EMU_STRATEGY_PERFORMANT": emu.EMU_STRATEGY_PERFORMANT}
    assert {f"EMU_STRATEGY_{k.upper()}": v for k, v in emu.STRATEGIES.items()} == strategies
    st = _declared_enum("EMU_STATUS_")
    assert {v: k for k, v in st.items()} == emu.STATUS_NAMES


def test_status_strings(lib):
    emu.load()
    for code, name in emu.STATUS_NAMES.items():
        assert emu.emu_status_string(code) == name
    assert emu.emu_status_string(99) == "EMU_STATUS_UNKNOWN"
    assert emu.emu_version() >= 100


def test_host_checks_reject_bad_arguments_before_any_device_work(lib):
    """Argument errors are reported from the host checks alone, so they
    answer the same with or without a GPU; nothing is enqueued."""
    f = emu.load().emu_sgemm
    buf = (ctypes.c_float * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    aligned = ctypes.c_void_p((p.value + 15) & ~15)
    z = ctypes.c_void_p(0)
    assert f(0, 0, 0, -1, 4, 4, 1.0, aligned, 4, aligned, 4, 0.0, aligned, 4, z) == 1   # negative M
    assert f(5, 0, 0, 4, 4, 4, 1.0, aligned, 4, aligned, 4, 0.0, aligned, 4, z) == 1   # bad mode
    assert f(0, 3, 0, 4, 4, 4, 1.0, aligned, 4, aligned, 4, 0.0, aligned, 4, z) == 1   # bad op
    assert f(0, 0, 0, 4, 4, 4, 1.0, aligned, 2, aligned, 4, 0.0, aligned, 4, z) == 1   # lda < K
    assert f(0, 0, 0, 4, 4, 4, 1.0, None, 4, aligned, 4, 0.0, aligned, 4, z) == 1      # NULL A
    mis = ctypes.c_void_p(aligned.value + 4)
    assert f(0, 0, 0, 4, 4, 4, 1.0, mis, 4, aligned, 4, 0.0, aligned, 4, z) == 2      # misaligned A
    assert f(0, 0, 0, 4, 4, 4, 1.0, aligned, 4, aligned, 4, 0.0, aligned, 2, z) == 1   # ldc < N
    assert f(0, 0, 0, 4, 4, 4, 1.0, aligned, 4, aligned, 4, 0.0, aligned, 6, z) == 2   # ldc not a multiple of 4
    assert f(0, 0, 0, 0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, z) == 0            # M == 0: no-op


def test_no_gpu_means_error_not_fallback(lib):
    """Without a usable GPU a valid call fails loudly (no CPU fallback)."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except Exception:
        pass
    f = emu.load().emu_sgemm
    buf = (ctypes.c_float * 64)()
    aligned = ctypes.c_void_p((ctypes.cast(buf, ctypes.c_void_p).value + 15) & ~15)
    st = f(0, 0, 0, 4, 4, 4, 1.0, aligned, 4, aligned, 4, 0.0, aligned, 4, ctypes.c_void_p(0))
    assert st in (3, 5)


def test_strategy_and_dispatch_are_host_decisions(lib):
    """The strategy switch and the dispatch decision need no GPU.  Eager runs
    every product in the requested mode; performant sends small products to
    native FP32 and keeps large ones emulated; FP32 requested stays FP32;
    packing has no FP32 form."""
    assert emu.emu_get_strategy() == "eager"
    assert emu.load().emu_set_strategy(7) == 1
    for mode in ("bf16x9", "tf32x3", "tf32x1", "bf16x6", "fp32"):
        assert emu.emu_dispatch_query(mode, 64, 64, 64) == mode
        assert emu.emu_dispatch_query(mode, 16384, 16384, 16384) == mode
    with emu.strategy("performant"):
        assert emu.emu_get_strategy() == "performant"
        for mode in ("bf16x9", "tf32x3"):
            assert emu.emu_dispatch_query(mode, 64, 64, 64) == "fp32"
            assert emu.emu_dispatch_query(mode, 192, 256, 256) == "fp32"
            assert emu.emu_dispatch_query(mode, 16384, 16384, 16384) == mode
            assert emu.emu_dispatch_query(mode, 17280, 512, 512) == mode
        assert emu.emu_dispatch_query("fp32", 16384, 16384, 16384) == "fp32"
        # a larger product is never sent to native FP32 when a smaller one of
        # the same shape family stays emulated
        sizes = [64 * 2 ** i for i in range(9)]
        picks = [emu.emu_dispatch_query("bf16x9", s, s, s) for s in sizes]
        first_emulated = picks.index("bf16x9")
        assert all(p == "bf16x9" for p in picks[first_emulated:])
    assert emu.emu_get_strategy() == "eager"
    with pytest.raises(emu.EmuError):
        emu.emu_dispatch_query("bf16x9", 0, 4, 4)
    assert emu.emu_pack_bytes("fp32", 64, 64) == -1


def test_failure_hooks_check_arguments_on_the_host(lib):
    """The diagnostic and test-hook entry points validate their arguments
    before touching a device; emu_shutdown with nothing cached is a no-op."""
    L = emu.load()
    z = ctypes.c_void_p(0)
    assert L.emu_debug_fail_allocations(-1) == 1
    assert L.emu_debug_fail_allocations(0) == 0
    assert L.emu_selftest_split_timeout(0, 4, z) == 1                  # zero budget
    assert L.emu_selftest_split_timeout(11_000_000_000, 4, z) == 1     # above 10 s
    assert L.emu_selftest_split_timeout(1_000_000, 0, z) == 1          # no tiles
    assert L.emu_selftest_wait_timeout(0, z) == 1
    assert L.emu_shutdown() == 0

"""GPU parity at the full sizes of the PET-like, wide-model and stress
workloads, in the launch configuration the benchmark times, checked on
deterministic row samples the oracle can evaluate row by row."""
import numpy as np
import pytest

import oracle
from fp32_emulated_gemm_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
MODES = ["bf16x9", "tf32x3"]


def _linear_pair(mode, shape, config, rows):
    import fp32_emulated_gemm_gb300 as emu
    X, Wt, b, dY = W.linear_inputs(shape, config)
    Y = emu.linear_fwd(_gpu.to_dev(X), _gpu.to_dev(Wt), _gpu.to_dev(b), mode=mode)
    dX = emu.linear_bwd_input(_gpu.to_dev(dY), _gpu.to_dev(Wt), mode=mode)
    assert emu.emu_stream_check() == 0
    Yh, dXh = Y.cpu().numpy(), dX.cpu().numpy()
    del Y, dX
    r1 = _gpu.compare(mode, Yh, oracle.Problem(X, Wt, transB=True, bias=b), rows)
    r2 = _gpu.compare(mode, dXh, oracle.Problem(dY, Wt), rows)
    return r1, r2


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layer", ["wide_l1", "wide_l2"])
def test_wide_model_layers(mode, layer):
    """M=6144; K=1024 N=4096 and K=4096 N=1024; forward and input gradient."""
    shape = W.WIDE_L1 if layer == "wide_l1" else W.WIDE_L2
    rows = W.sample_rows(shape.M, every=128, edge=64)
    _linear_pair(mode, shape, W.CONFIG_ID["wide"], rows)


@pytest.mark.parametrize("mode", MODES)
def test_pet_large(mode):
    """M=552960, K=256, N=1024 forward and input gradient (17,280 atoms x 32)."""
    shape = W.PET_LARGE
    rows = W.sample_rows(shape.M, every=2048, edge=128)
    _linear_pair(mode, shape, W.CONFIG_ID["pet_large"], rows)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", list(W.STRESS_SIZES))
def test_stress_sweep(mode, n):
    """Square GEMMs, magnitudes 2^U[-20,20], 1% zeros/subnormals/huge values:
    the normwise bound against float64 holds; BF16x9 is also compared with
    the oracle's native FP32 SGEMM error (reported, and required to be no
    worse than 4x it at these sizes)."""
    A, B = W.stress_inputs(n)
    if n <= 1024:
        rows = np.arange(n)
    elif n <= 4096:
        rows = W.sample_rows(n, every=256, edge=8)
    else:
        rows = np.array([0, 1, n // 3, n // 2, n - 2, n - 1], dtype=np.int64)
    C = _gpu.gpu_sgemm(mode, A, B)
    p = oracle.Problem(A, B)
    res = _gpu.compare(mode, C, p, rows, elementwise=False)
    if mode == "bf16x9":
        C64, D = oracle.gemm_f64(p, rows), oracle.absdenom_f64(p, rows)
        e32 = oracle.normwise_error(oracle.sgemm_f32(p, rows), C64, D)
        assert res["normwise"] <= 4 * max(e32, 2.0 ** -24), (res["normwise"], e32)

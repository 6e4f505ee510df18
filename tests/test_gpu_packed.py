"""Weight pre-split (packed op(B)) on the GPU.

The packed planes are the kernel's own split of op(B)^T, so a product with a
packed operand must give exactly the bits of the unpacked product; the
planes themselves must equal the oracle's split (components in natural
magnitude for BF16, hi and lo for TF32).
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
    assert not diff.any(), f"{int(diff.sum())} of {diff.size} elements differ"


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tA,tB", [(False, False), (True, True), (False, True)])
def test_packed_product_equals_unpacked_bitwise(mode, tA, tB):
    import torch
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(31)
    for (M, N, K) in [(300, 260, 200), (520, 130, 1100), (64, 1000, 37)]:
        A = rng.standard_normal((K, M) if tA else (M, K)).astype(np.float32)
        B = rng.standard_normal((N, K) if tB else (K, N)).astype(np.float32)
        Ad, Bd = _gpu.to_dev_padded(A, float("nan")), _gpu.to_dev_padded(B, float("nan"))
        plain = emu.sgemm(Ad, Bd, mode=mode, transA=tA, transB=tB)
        packed = emu.pack_b(Bd, mode=mode, transB=tB)
        got = emu.sgemm_packed(Ad, packed, N, mode=mode, transA=tA)
        assert emu.emu_stream_check() == 0
        _same_bits(got.cpu().numpy(), plain.cpu().numpy())


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_pack_planes_equal_the_oracle_split(mode):
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(32)
    N, K = 70, 45                                  # Kp = 64: the tail past K must be zero
    sign = rng.integers(0, 2, N * K, dtype=np.uint32) << np.uint32(31)
    ex = (rng.integers(-60, 61, N * K) + 127).astype(np.uint32) << np.uint32(23)
    fr = rng.integers(0, 1 << 23, N * K, dtype=np.uint32)
    Bt = (sign | ex | fr).view(np.float32).reshape(N, K)      # op(B)^T, stored N x K (transB)
    packed = emu.pack_b(_gpu.to_dev(Bt), mode=mode, transB=True).cpu().numpy()
    Kp = 64
    if mode == "bf16x9":
        planes = packed.view(np.uint16).reshape(3, N, Kp)
        c = oracle.split_bf16x9_f32(Bt.ravel())
        for i in range(3):
            want = (c[i].astype(np.float64) * 2.0 ** (-8 * i)).astype(np.float32).reshape(N, K)
            assert np.array_equal(planes[i, :, :K], (want.view(np.uint32) >> 16).astype(np.uint16)), i
        assert not planes[:, :, K:].any()
    else:
        planes = packed.view(np.uint32).reshape(2, N, Kp)
        hi, lo = oracle.split_tf32x3(Bt.ravel())
        assert np.array_equal(planes[0, :, :K], hi.view(np.uint32).reshape(N, K))
        assert np.array_equal(planes[1, :, :K], lo.view(np.uint32).reshape(N, K))
        assert not planes[:, :, K:].any()


@pytest.mark.parametrize("mode", ["bf16x9", "tf32x3"])
def test_packed_linear_layer_matches_unpacked_and_oracle(mode):
    import fp32_emulated_gemm_gb300 as emu
    s = W.PET_SMALL
    X, Wt, b, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    Xd, Wd, bd, dYd = (_gpu.to_dev(a) for a in (X, Wt, b, dY))
    pw = emu.pack_weight(Wd, mode)
    Y, dX = emu.linear_fwd_packed(Xd, pw, bd), emu.linear_bwd_input_packed(dYd, pw)
    Y0, dX0 = emu.linear_fwd(Xd, Wd, bd, mode=mode), emu.linear_bwd_input(dYd, Wd, mode=mode)
    assert emu.emu_stream_check() == 0
    _same_bits(Y.cpu().numpy(), Y0.cpu().numpy())
    _same_bits(dX.cpu().numpy(), dX0.cpu().numpy())
    rows = W.sample_rows(s.M, every=64, edge=64)
    _gpu.compare(mode, Y.cpu().numpy(), oracle.Problem(X, Wt, transB=True, bias=b), rows)
    _gpu.compare(mode, dX.cpu().numpy(), oracle.Problem(dY, Wt), rows)


def test_emulinear_prepack_follows_weight_updates():
    import torch
    import fp32_emulated_gemm_gb300 as emu
    torch.manual_seed(1)
    lin = emu.EmuLinear(256, 384, mode="bf16x9", prepack=True).cuda()
    ref = emu.EmuLinear(256, 384, mode="bf16x9").cuda()
    ref.load_state_dict(lin.state_dict())
    x = torch.randn(700, 256, device="cuda")
    assert torch.equal(lin(x), ref(x))
    with torch.no_grad():                          # an optimizer step changes the weight in place
        lin.weight.mul_(0.5)
        ref.weight.mul_(0.5)
    assert torch.equal(lin(x), ref(x))
    xg = x.clone().requires_grad_(True)
    xr = x.clone().requires_grad_(True)
    lin(xg).sum().backward()
    ref(xr).sum().backward()
    assert torch.equal(xg.grad, xr.grad)


def test_packed_rejects_bad_arguments():
    import torch
    import fp32_emulated_gemm_gb300 as emu
    dev = _gpu.device()
    B = torch.zeros((8, 8), device=dev)
    buf = torch.zeros(emu.emu_pack_bytes(0, 8, 8) + 16, dtype=torch.uint8, device=dev)
    with pytest.raises(emu.EmuError):
        emu.emu_pack_b(0, 5, 8, 8, B, 8, buf)               # bad transB
    with pytest.raises(emu.EmuError):
        emu.emu_pack_b(0, 1, 8, 8, B, 4, buf)               # ldb < K
    with pytest.raises(emu.EmuError):
        emu.emu_pack_b(0, 1, 8, 8, B, 8, buf[1:])           # misaligned
    assert emu.emu_pack_bytes(9, 8, 8) == -1


@pytest.mark.parametrize("mode", ["tf32x3", "tf32x1"])
def test_automatic_pre_split_gives_the_same_bits(mode, monkeypatch):
    """TF32 products with several tile rows split op(B) ahead of the product;
    the result must not depend on it."""
    import fp32_emulated_gemm_gb300 as emu
    rng = np.random.default_rng(33)
    M, N, K = 1100, 300, 700
    A = _gpu.to_dev(rng.standard_normal((M, K)).astype(np.float32))
    B = _gpu.to_dev(rng.standard_normal((K, N)).astype(np.float32))
    auto = emu.sgemm(A, B, mode=mode).cpu().numpy()
    monkeypatch.setenv("EMU_AUTOPACK", "0")   # read once per process: use a child process
    import subprocess, sys, os
    code = ("import numpy as np, torch, fp32_emulated_gemm_gb300 as emu\n"
            "rng = np.random.default_rng(33)\n"
            "A = torch.from_numpy(rng.standard_normal((1100, 700)).astype(np.float32)).cuda()\n"
            "B = torch.from_numpy(rng.standard_normal((700, 300)).astype(np.float32)).cuda()\n"
            f"np.save('/tmp/emu_noautopack.npy', emu.sgemm(A, B, mode='{mode}').cpu().numpy())\n")
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ), capture_output=True, text=True,
                       timeout=300, cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stderr[-2000:]
    _same_bits(auto, np.load("/tmp/emu_noautopack.npy"))

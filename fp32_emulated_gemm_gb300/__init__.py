"""FP32 GEMM emulated on GB300 tensor cores (BF16x9 and TF32x3).

Thin Python binding over the C ABI of ``libemu_gemm.so`` (see
``include/emu_gemm.h``): the functions below carry the C names and only
marshal arguments (device pointers, sizes, the current CUDA stream).  Every
step of the computation runs in the library's sm_103a kernels; there is no
Python or CPU fallback, and a missing library raises at import of the first
call.

Method: NVIDIA blog "Unlocking Tensor Core performance for machine-learning
interatomic potentials", section "How Tensor Core FP32 bridges the hardware
gap" (Fig. 1 BF16x9, Fig. 2 and Eq. 1 TF32x3).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "EMU_MODE_BF16X9", "EMU_MODE_TF32X3", "EMU_MODE_TF32X1", "EMU_MODE_BF16X6", "EMU_MODE_FP32", "EMU_OP_N",
    "EMU_OP_T", "EMU_STRATEGY_EAGER", "EMU_STRATEGY_PERFORMANT",
    "EmuError",
    "emu_sgemm", "emu_linear_fwd", "emu_linear_bwd_input", "emu_linear_bwd_weight", "emu_status_string",
    "emu_stream_check", "emu_split_dump", "emu_plan_query", "emu_version",
    "emu_selftest_wait_timeout", "emu_selftest_split_timeout", "emu_shutdown", "emu_debug_fail_allocations",
    "emu_set_strategy", "emu_get_strategy", "emu_dispatch_query", "strategy",
    "emu_pack_bytes", "emu_pack_b", "emu_sgemm_packed_b", "emu_linear_fwd_packed", "emu_linear_bwd_input_packed",
    "pack_b", "sgemm_packed", "PackedWeight", "pack_weight", "linear_fwd_packed", "linear_bwd_input_packed",
    "sgemm", "linear_fwd", "linear_bwd_input", "linear_bwd_weight", "EmuLinearFunction", "EmuLinear",
    "library_path", "load",
]

EMU_MODE_BF16X9 = 0
EMU_MODE_TF32X3 = 1
EMU_MODE_TF32X1 = 2
EMU_MODE_BF16X6 = 3
EMU_MODE_FP32 = 4
EMU_OP_N = 0
EMU_OP_T = 1
EMU_STRATEGY_EAGER = 0
EMU_STRATEGY_PERFORMANT = 1
MODES = {"bf16x9": EMU_MODE_BF16X9, "tf32x3": EMU_MODE_TF32X3, "tf32x1": EMU_MODE_TF32X1,
         "bf16x6": EMU_MODE_BF16X6, "fp32": EMU_MODE_FP32}
STRATEGIES = {"eager": EMU_STRATEGY_EAGER, "performant": EMU_STRATEGY_PERFORMANT}

STATUS_NAMES = {
    0: "EMU_STATUS_SUCCESS", 1: "EMU_STATUS_INVALID_VALUE", 2: "EMU_STATUS_NOT_SUPPORTED",
    3: "EMU_STATUS_ARCH_MISMATCH", 4: "EMU_STATUS_ALLOC_FAILED", 5: "EMU_STATUS_LAUNCH_FAILED",
    6: "EMU_STATUS_DEVICE_TIMEOUT",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class EmuError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {STATUS_NAMES.get(self.status, self.status)}")


def library_path() -> str:
    return os.path.join(_HERE, "libemu_gemm.so")


def load():
    """Load libemu_gemm.so (built in-tree by build.py); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -m fp32_emulated_gemm_gb300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(path)
        i64, i32, f32, P = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        L.emu_sgemm.argtypes = [i32, i32, i32, i64, i64, i64, f32, P, i64, P, i64, f32, P, i64, P]
        L.emu_linear_fwd.argtypes = [i32, i64, i64, i64, P, P, P, P, P]
        L.emu_linear_bwd_input.argtypes = [i32, i64, i64, i64, P, P, P, P]
        L.emu_linear_bwd_weight.argtypes = [i32, i64, i64, i64, P, P, f32, P, P]
        L.emu_status_string.argtypes = [i32]
        L.emu_status_string.restype = ctypes.c_char_p
        L.emu_stream_check.argtypes = [P]
        L.emu_split_dump.argtypes = [i32, i64, i64, P, i64, i32, P, P]
        L.emu_pack_bytes.argtypes = [i32, i64, i64]
        L.emu_pack_bytes.restype = i64
        L.emu_pack_b.argtypes = [i32, i32, i64, i64, P, i64, P, P]
        L.emu_sgemm_packed_b.argtypes = [i32, i32, i64, i64, i64, f32, P, i64, P, f32, P, i64, P]
        L.emu_linear_fwd_packed.argtypes = [i32, i64, i64, i64, P, P, P, P, P]
        L.emu_linear_bwd_input_packed.argtypes = [i32, i64, i64, i64, P, P, P, P]
        for name in ("emu_pack_b", "emu_sgemm_packed_b", "emu_linear_fwd_packed", "emu_linear_bwd_input_packed"):
            getattr(L, name).restype = i32
        L.emu_plan_query.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i64), i32]
        L.emu_plan_query.restype = i32
        L.emu_plan_bounds.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i64), i32]
        L.emu_plan_bounds.restype = i32
        L.emu_version.argtypes = []
        L.emu_set_strategy.argtypes = [i32]
        L.emu_set_strategy.restype = i32
        L.emu_get_strategy.argtypes = []
        L.emu_get_strategy.restype = i32
        L.emu_dispatch_query.argtypes = [i32, i64, i64, i64, i32, ctypes.POINTER(i32)]
        L.emu_dispatch_query.restype = i32
        L.emu_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
        L.emu_selftest_split_timeout.argtypes = [ctypes.c_uint64, i64, P]
        L.emu_shutdown.argtypes = []
        L.emu_debug_fail_allocations.argtypes = [i32]
        for name in ("emu_sgemm", "emu_linear_fwd", "emu_linear_bwd_input", "emu_linear_bwd_weight",
                     "emu_stream_check", "emu_split_dump", "emu_version", "emu_selftest_wait_timeout",
                     "emu_selftest_split_timeout", "emu_shutdown", "emu_debug_fail_allocations"):
            getattr(L, name).restype = i32
        _lib = L
        return L


# ------------------------------------------------------------ C names ------
def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr() if hasattr(t, "data_ptr") else int(t))


def _check(st: int, what: str) -> None:
    if st != 0:
        raise EmuError(st, what)


def emu_sgemm(mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
    _check(load().emu_sgemm(int(mode), int(transA), int(transB), int(M), int(N), int(K), float(alpha),
                            _ptr(A), int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc),
                            ctypes.c_void_p(_stream(stream))), "emu_sgemm")


def emu_linear_fwd(mode, M, N, K, X, W, bias, Y, stream=None):
    _check(load().emu_linear_fwd(int(mode), int(M), int(N), int(K), _ptr(X), _ptr(W), _ptr(bias), _ptr(Y),
                                 ctypes.c_void_p(_stream(stream))), "emu_linear_fwd")


def emu_linear_bwd_input(mode, M, N, K, dY, W, dX, stream=None):
    _check(load().emu_linear_bwd_input(int(mode), int(M), int(N), int(K), _ptr(dY), _ptr(W), _ptr(dX),
                                       ctypes.c_void_p(_stream(stream))), "emu_linear_bwd_input")


def emu_linear_bwd_weight(mode, M, N, K, dY, X, beta, dW, stream=None):
    _check(load().emu_linear_bwd_weight(int(mode), int(M), int(N), int(K), _ptr(dY), _ptr(X), float(beta),
                                        _ptr(dW), ctypes.c_void_p(_stream(stream))), "emu_linear_bwd_weight")


def emu_status_string(status: int) -> str:
    return load().emu_status_string(int(status)).decode()


def emu_stream_check(stream=None) -> int:
    return int(load().emu_stream_check(ctypes.c_void_p(_stream(stream))))


def emu_selftest_wait_timeout(budget_ns, stream=None):
    _check(load().emu_selftest_wait_timeout(int(budget_ns), ctypes.c_void_p(_stream(stream))),
           "emu_selftest_wait_timeout")


def emu_selftest_split_timeout(budget_ns, tiles, stream=None):
    _check(load().emu_selftest_split_timeout(int(budget_ns), int(tiles), ctypes.c_void_p(_stream(stream))),
           "emu_selftest_split_timeout")


def emu_shutdown():
    _check(load().emu_shutdown(), "emu_shutdown")


def emu_debug_fail_allocations(n):
    _check(load().emu_debug_fail_allocations(int(n)), "emu_debug_fail_allocations")


def emu_split_dump(mode, R, Kc, X, ldx, mn_major, out, stream=None):
    _check(load().emu_split_dump(int(mode), int(R), int(Kc), _ptr(X), int(ldx), int(mn_major), _ptr(out),
                                 ctypes.c_void_p(_stream(stream))), "emu_split_dump")


def emu_pack_bytes(mode, N, K) -> int:
    return int(load().emu_pack_bytes(_mode(mode), int(N), int(K)))


def emu_pack_b(mode, transB, N, K, B, ldb, packed, stream=None):
    _check(load().emu_pack_b(int(mode), int(transB), int(N), int(K), _ptr(B), int(ldb), _ptr(packed),
                             ctypes.c_void_p(_stream(stream))), "emu_pack_b")


def emu_sgemm_packed_b(mode, transA, M, N, K, alpha, A, lda, packed_b, beta, C, ldc, stream=None):
    _check(load().emu_sgemm_packed_b(int(mode), int(transA), int(M), int(N), int(K), float(alpha), _ptr(A),
                                     int(lda), _ptr(packed_b), float(beta), _ptr(C), int(ldc),
                                     ctypes.c_void_p(_stream(stream))), "emu_sgemm_packed_b")


def emu_linear_fwd_packed(mode, M, N, K, X, W_packed, bias, Y, stream=None):
    _check(load().emu_linear_fwd_packed(int(mode), int(M), int(N), int(K), _ptr(X), _ptr(W_packed), _ptr(bias),
                                        _ptr(Y), ctypes.c_void_p(_stream(stream))), "emu_linear_fwd_packed")


def emu_linear_bwd_input_packed(mode, M, N, K, dY, Wt_packed, dX, stream=None):
    _check(load().emu_linear_bwd_input_packed(int(mode), int(M), int(N), int(K), _ptr(dY), _ptr(Wt_packed),
                                              _ptr(dX), ctypes.c_void_p(_stream(stream))),
           "emu_linear_bwd_input_packed")


PLAN_FIELDS = ("pipe", "tile_n", "tiles_m", "tiles_n", "k_stages", "tiles_a", "split_a", "split_b",
               "units", "pairs", "slots", "cost_x100", "chain")


def emu_plan_query(M, N, K, pairs) -> dict:
    """The launch plan emu_sgemm would use (host only; see the header)."""
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    _check(load().emu_plan_query(int(M), int(N), int(K), int(pairs), out, len(PLAN_FIELDS)), "emu_plan_query")
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


def emu_plan_bounds(M, N, K, pairs) -> list:
    """The run bounds of the chained plan emu_plan_query describes (host
    only; see the header)."""
    out = (ctypes.c_int64 * (int(pairs) + 1))()
    _check(load().emu_plan_bounds(int(M), int(N), int(K), int(pairs), out, int(pairs) + 1), "emu_plan_bounds")
    return [int(v) for v in out]


def emu_version() -> int:
    return int(load().emu_version())


def emu_set_strategy(strategy) -> None:
    """Process-wide strategy: "eager" (always the requested mode) or
    "performant" (native FP32 where emulation is predicted slower)."""
    s = STRATEGIES[strategy] if isinstance(strategy, str) else int(strategy)
    _check(load().emu_set_strategy(s), "emu_set_strategy")


def emu_get_strategy() -> str:
    v = int(load().emu_get_strategy())
    return {c: n for n, c in STRATEGIES.items()}[v]


def emu_dispatch_query(mode, M, N, K, pairs=76) -> str:
    """The mode emu_sgemm would run an M x N x K product in under the current
    strategy (host only)."""
    out = ctypes.c_int(-1)
    _check(load().emu_dispatch_query(_mode(mode), int(M), int(N), int(K), int(pairs), ctypes.byref(out)),
           "emu_dispatch_query")
    return {c: n for n, c in MODES.items()}[out.value]


class strategy:
    """Context manager: run the enclosed calls under another strategy, then
    restore the previous one (process-wide, so not for concurrent threads
    that want different strategies)."""

    def __init__(self, name):
        self.name = name
        self.prev = None

    def __enter__(self):
        self.prev = emu_get_strategy()
        emu_set_strategy(self.name)
        return self

    def __exit__(self, *exc):
        emu_set_strategy(self.prev)
        return False


# ----------------------------------------------------- tensor helpers ------
def _mode(mode):
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _f32_cuda(t, name):
    import torch
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32):
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor (unit column stride)")
    return t


def _new_c(M, N, device):
    """An M x N float32 result whose rows start on 16-byte boundaries (the
    library wants ldc to be a multiple of 4): a view of a padded buffer when
    N is not a multiple of 4."""
    import torch
    ld = (N + 3) // 4 * 4
    return torch.empty((M, ld), device=device, dtype=torch.float32)[:, :N]


def sgemm(A, B, *, mode="bf16x9", transA=False, transB=False, alpha=1.0, beta=0.0, C=None):
    """C = alpha op(A) op(B) + beta C on the current stream (C allocated when None)."""
    import torch
    _f32_cuda(A, "A"), _f32_cuda(B, "B")
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    Kb, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if Kb != K:
        raise ValueError("inner dimensions differ")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = _new_c(M, N, A.device)
    _f32_cuda(C, "C")
    emu_sgemm(_mode(mode), EMU_OP_T if transA else EMU_OP_N, EMU_OP_T if transB else EMU_OP_N, M, N, K,
              alpha, A, A.stride(0), B, B.stride(0), beta, C, C.stride(0))
    return C


def pack_b(B, *, mode="bf16x9", transB=False):
    """Packed form of op(B) (a uint8 device tensor) for sgemm_packed."""
    import torch
    _f32_cuda(B, "B")
    K, N = (B.shape[1], B.shape[0]) if transB else B.shape
    out = torch.empty(max(1, emu_pack_bytes(_mode(mode), N, K)), dtype=torch.uint8, device=B.device)
    emu_pack_b(_mode(mode), EMU_OP_T if transB else EMU_OP_N, N, K, B, B.stride(0), out)
    return out


def sgemm_packed(A, packed_b, N, *, mode="bf16x9", transA=False, alpha=1.0, beta=0.0, C=None):
    """C = alpha op(A) op(B) + beta C with op(B) given by pack_b (N columns)."""
    import torch
    _f32_cuda(A, "A")
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = _new_c(M, N, A.device)
    _f32_cuda(C, "C")
    emu_sgemm_packed_b(_mode(mode), EMU_OP_T if transA else EMU_OP_N, M, N, K, alpha, A, A.stride(0), packed_b,
                       beta, C, C.stride(0))
    return C


class PackedWeight:
    """A linear layer's weight W [N, K] split once for both passes: `fwd` for
    Y = X W^T + b and `bwd` for dX = dY W.  Valid while W is unchanged (see
    `version`, the tensor's version counter when it was packed)."""

    def __init__(self, W, mode="bf16x9"):
        _f32_cuda(W, "W")
        W = W.contiguous()
        self.mode, self.N, self.K = mode, W.shape[0], W.shape[1]
        self.version = W._version
        self.fwd = pack_b(W, mode=mode, transB=True)
        self.bwd = pack_b(W, mode=mode, transB=False)


def pack_weight(W, mode="bf16x9"):
    return PackedWeight(W, mode)


def linear_fwd_packed(X, pw: PackedWeight, bias=None, *, out=None):
    import torch
    M, K = X.shape
    Y = out if out is not None else torch.empty((M, pw.N), device=X.device, dtype=torch.float32)
    emu_linear_fwd_packed(_mode(pw.mode), M, pw.N, K, X.contiguous(), pw.fwd,
                          None if bias is None else bias.contiguous(), Y)
    return Y


def linear_bwd_input_packed(dY, pw: PackedWeight, *, out=None):
    import torch
    M, N = dY.shape
    dX = out if out is not None else torch.empty((M, pw.K), device=dY.device, dtype=torch.float32)
    emu_linear_bwd_input_packed(_mode(pw.mode), M, N, pw.K, dY.contiguous(), pw.bwd, dX)
    return dX


def linear_fwd(X, W, bias=None, *, mode="bf16x9", out=None):
    """Y = X W^T + bias (X [M,K], W [N,K], contiguous)."""
    import torch
    M, K = X.shape
    N = W.shape[0]
    Y = out if out is not None else torch.empty((M, N), device=X.device, dtype=torch.float32)
    emu_linear_fwd(_mode(mode), M, N, K, X.contiguous(), W.contiguous(),
                   None if bias is None else bias.contiguous(), Y)
    return Y


def linear_bwd_input(dY, W, *, mode="bf16x9", out=None):
    """dX = dY W (dY [M,N], W [N,K], contiguous)."""
    import torch
    M, N = dY.shape
    K = W.shape[1]
    dX = out if out is not None else torch.empty((M, K), device=dY.device, dtype=torch.float32)
    emu_linear_bwd_input(_mode(mode), M, N, K, dY.contiguous(), W.contiguous(), dX)
    return dX


def linear_bwd_weight(dY, X, *, mode="bf16x9", out=None, beta=0.0):
    """dW = dY^T X (+ beta * out) (dY [M,N], X [M,K], contiguous)."""
    import torch
    M, N = dY.shape
    K = X.shape[1]
    dW = out if out is not None else torch.empty((N, K), device=dY.device, dtype=torch.float32)
    emu_linear_bwd_weight(_mode(mode), M, N, K, dY.contiguous(), X.contiguous(), beta, dW)
    return dW


def _autograd():
    import torch

    class EmuLinearFunction(torch.autograd.Function):
        """nn.Linear with the forward and the input gradient emulated; the
        weight gradient uses plain FP32 (TF32 off), as in the blog's
        TF32Linear ("TF32x3 on Ampere GPUs"), unless weight_grad="emulated"."""

        @staticmethod
        def forward(ctx, X, W, bias, mode, weight_grad="fp32", packed=None):
            ctx.save_for_backward(X, W)
            ctx.mode = mode
            ctx.weight_grad = weight_grad
            ctx.has_bias = bias is not None
            ctx.packed = packed
            if packed is not None:
                return linear_fwd_packed(X, packed, bias)
            return linear_fwd(X, W, bias, mode=mode)

        @staticmethod
        def backward(ctx, dY):
            X, W = ctx.saved_tensors
            dY = dY.contiguous()
            dX = None
            if ctx.needs_input_grad[0]:
                dX = (linear_bwd_input_packed(dY, ctx.packed) if ctx.packed is not None
                      else linear_bwd_input(dY, W, mode=ctx.mode))
            dW = db = None
            if ctx.needs_input_grad[1] and ctx.weight_grad == "emulated":
                dW = linear_bwd_weight(dY, X, mode=ctx.mode)
            elif ctx.needs_input_grad[1]:
                prev = torch.backends.cuda.matmul.allow_tf32
                torch.backends.cuda.matmul.allow_tf32 = False
                try:
                    dW = dY.t().mm(X)
                finally:
                    torch.backends.cuda.matmul.allow_tf32 = prev
            if ctx.has_bias and ctx.needs_input_grad[2]:
                db = dY.sum(0)
            return dX, dW, db, None, None, None

    class EmuLinear(torch.nn.Linear):
        """Drop-in nn.Linear whose matmuls run on the emulated path."""

        def __init__(self, in_features, out_features, bias=True, mode="bf16x9", weight_grad="fp32",
                     prepack=False, **kw):
            """prepack=True splits the weight once and reuses the split until the
            weight changes (fixed-weight inference and molecular dynamics)."""
            super().__init__(in_features, out_features, bias=bias, **kw)
            self.mode = mode
            self.weight_grad = weight_grad
            self.prepack = prepack
            self._packed = None

        def _packed_weight(self):
            W = self.weight
            pw = self._packed
            if (pw is None or pw.version != W._version or pw.mode != self.mode or pw.N != W.shape[0]
                    or pw.K != W.shape[1] or pw.fwd.device != W.device):
                with torch.no_grad():
                    pw = PackedWeight(W.detach(), self.mode)
                pw.version = W._version
                self._packed = pw
            return pw

        def forward(self, x):
            shp = x.shape
            # (native FP32 has no packed form: prepack then has nothing to do)
            packed = self._packed_weight() if self.prepack and _mode(self.mode) != EMU_MODE_FP32 else None
            y = EmuLinearFunction.apply(x.reshape(-1, shp[-1]), self.weight, self.bias, self.mode,
                                        self.weight_grad, packed)
            return y.reshape(*shp[:-1], self.out_features)

    return EmuLinearFunction, EmuLinear


def __getattr__(name):
    if name in ("EmuLinearFunction", "EmuLinear"):
        f, m = _autograd()
        globals()["EmuLinearFunction"], globals()["EmuLinear"] = f, m
        return globals()[name]
    raise AttributeError(name)

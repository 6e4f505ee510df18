"""Seeded synthetic inputs for the emulated-GEMM workloads.

This module holds no arithmetic of the method: it only draws random FP32
matrices.  It is the one module that both the tests' oracle side and the CUDA
side use, so that both see the same inputs.

The shapes stand in for the linear layers of the PET interatomic potential in
the blog post "Unlocking Tensor Core performance for machine-learning
interatomic potentials" ("Benchmarking on PET": a 192-atom water box and a
17,280-atom supercell, each atom with about 32 neighbours, so M = atoms x 32
tokens; a 26M- and a 255M-parameter checkpoint).  No checkpoint or dataset is
used: weights are random with the layer's fan-in scaling.

Seeds: numpy ``Generator(PCG64(100 * config + tensor_id))`` with tensor ids
A/X = 0, B/W = 1, bias = 2, dY = 3, C_old = 4.  The tiny config draws A, B and
C_old in that order from one ``default_rng(0)`` stream.  "N(0, s)" reads s as
the variance.
"""
from __future__ import annotations

import dataclasses

import numpy as np

FLT_MAX = float(np.finfo(np.float32).max)

TENSOR_A, TENSOR_B, TENSOR_BIAS, TENSOR_DY, TENSOR_COLD = 0, 1, 2, 3, 4


def rng_for(config: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(100 * int(config) + int(tensor_id)))


@dataclasses.dataclass(frozen=True)
class LinearShape:
    """One linear layer: forward Y[M,N] = X[M,K] W[N,K]^T + b, input gradient dX = dY W."""
    name: str
    M: int
    K: int
    N: int


# The five workloads.
TINY = dict(M=128, N=128, K=256)
PET_SMALL = LinearShape("pet_small", M=6144, K=256, N=1024)        # 192 atoms x 32
PET_LARGE = LinearShape("pet_large", M=552960, K=256, N=1024)      # 17,280 atoms x 32
WIDE_L1 = LinearShape("wide_l1", M=6144, K=1024, N=4096)
WIDE_L2 = LinearShape("wide_l2", M=6144, K=4096, N=1024)
STRESS_SIZES = (256, 1024, 4096, 16384)

CONFIG_ID = {"tiny": 1, "pet_small": 2, "pet_large": 3, "wide": 4, "stress": 5}


def tiny_inputs():
    """A, B, C_old ~ U[-1, 1] from one seed-0 stream, in that order."""
    g = np.random.default_rng(0)
    A = g.uniform(-1.0, 1.0, size=(TINY["M"], TINY["K"])).astype(np.float32)
    B = g.uniform(-1.0, 1.0, size=(TINY["K"], TINY["N"])).astype(np.float32)
    C = g.uniform(-1.0, 1.0, size=(TINY["M"], TINY["N"])).astype(np.float32)
    return A, B, C


def linear_inputs(shape: LinearShape, config: int, with_bias: bool = True, rows: int | None = None):
    """X ~ N(0,1) [M,K], W ~ N(0,1/K) [N,K], b ~ N(0,0.01) [N], dY ~ N(0,1) [M,N].

    ``rows`` draws only the first ``rows`` rows of X and dY (same values as
    the full draw, since both are generated row-major from their own stream).
    """
    M = shape.M if rows is None else int(rows)
    X = _normal(rng_for(config, TENSOR_A), (M, shape.K), 1.0)
    W = _normal(rng_for(config, TENSOR_B), (shape.N, shape.K), 1.0 / np.sqrt(shape.K))
    b = _normal(rng_for(config, TENSOR_BIAS), (shape.N,), 0.1) if with_bias else None
    dY = _normal(rng_for(config, TENSOR_DY), (M, shape.N), 1.0)
    return X, W, b, dY


def _normal(g: np.random.Generator, shape, std: float) -> np.ndarray:
    out = np.empty(shape, np.float32)
    flat = out.reshape(-1)
    step = 1 << 24  # chunked so multi-GB draws never hold a float64 copy
    for s in range(0, flat.size, step):
        e = min(flat.size, s + step)
        flat[s:e] = g.standard_normal(e - s) * std
    return out


def stress_matrix(n: int, tensor_id: int, allow_huge: bool, zero_specials: bool = False):
    """n x n matrix: random sign, magnitude 2^u with u ~ U[-20, 20]; 1% of the
    entries replaced, in equal parts, by zeros, subnormals and (A only)
    values near FLT_MAX / (K 2^20) so that every K-term sum stays finite."""
    g = rng_for(CONFIG_ID["stress"] * 10 + int(np.log2(n)), tensor_id)
    out = np.empty((n, n), np.float32)
    flat = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat.size, step):
        e = min(flat.size, s + step)
        u = g.uniform(-20.0, 20.0, e - s)
        sign = np.where(g.random(e - s) < 0.5, -1.0, 1.0)
        flat[s:e] = sign * np.exp2(u)
    nspec = max(1, flat.size // 100)
    idx = g.choice(flat.size, size=nspec, replace=False)
    classes = 3 if allow_huge else 2
    kind = np.arange(nspec) % classes
    if zero_specials:
        flat[idx] = 0.0
        return out
    flat[idx[kind == 0]] = 0.0
    sub = idx[kind == 1]
    mant = g.integers(1, 1 << 23, size=sub.size, dtype=np.uint32)
    sgn = (g.random(sub.size) < 0.5).astype(np.uint32) << 31
    flat[sub] = (mant | sgn).view(np.float32)
    if allow_huge:
        huge = idx[kind == 2]
        v = FLT_MAX / (n * 2.0 ** 20) * (1.0 - g.uniform(0.0, 2.0 ** -8, huge.size))
        sgn = np.where(g.random(huge.size) < 0.5, -1.0, 1.0)
        flat[huge] = (sgn * v).astype(np.float32)
    return out


def stress_inputs(n: int, zero_specials: bool = False):
    A = stress_matrix(n, TENSOR_A, allow_huge=True, zero_specials=zero_specials)
    B = stress_matrix(n, TENSOR_B, allow_huge=False, zero_specials=zero_specials)
    return A, B


def sample_rows(M: int, every: int = 64, edge: int = 256) -> np.ndarray:
    """Deterministic row sample of a tall problem: every `every`-th row plus
    the first and last `edge` rows."""
    r = set(range(0, M, every))
    r.update(range(0, min(edge, M)))
    r.update(range(max(0, M - edge), M))
    return np.array(sorted(r), dtype=np.int64)

"""Seeded synthetic inputs for the block-scaled GEMM workloads.

This module draws random numbers and nothing else: it holds none of the
quantisation or GEMM arithmetic, so both the CPU oracle and the CUDA path can
take their inputs from it without sharing any of the method's code.

Every array comes from ``numpy.random.Generator(PCG64)`` seeded with
``[0xB5C0 + workload index, stream]``; stream 1 is operand A (activations or
gradients), stream 2 is operand B (weights), stream 3 is a decode activation
vector, stream 4 is an optional addend C.  The distributions follow the five
workloads of the block-scaled GEMM study:

  * ``fp8_256``    FP8 E4M3 x E4M3, M=N=K=256, both operands ~N(0,1) with a
                   0.1 % Bernoulli mask of x100 outliers.
  * ``mxfp4_1024`` MXFP4, M=N=K=1024, ~N(0,1) times a per-row factor
                   2^U(-8,8) (B's rows are its N rows, stored N x K).
  * ``ffn_up``     FP8 forward FFN-up, M=8192, K=4096, N=14336: activations
                   ~N(0,1) with 0.1 % x50 outliers, weights ~N(0, 0.02).
  * ``dgrad``      FP8 backward dgrad, M=8192, K=14336, N=4096: gradients
                   Laplace(0, 1e-3) times a per-row 2^U(-12,0), weights
                   ~N(0, 0.02).
  * ``decode``     MXFP4 decode, M in {1,16}, K=8192, N=28672: weights
                   ~N(0, 0.02), activations ~N(0,1) (rounded to BF16 by the
                   caller).

Operand B is always returned in its stored orientation, N x K (K contiguous),
which is the column-major K x N matrix of the GEMM.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 0xB5C0

WORKLOADS = {
    # name: (index, M, N, K)
    "fp8_256": (0, 256, 256, 256),
    "mxfp4_1024": (1, 1024, 1024, 1024),
    "ffn_up": (2, 8192, 14336, 4096),
    "dgrad": (3, 8192, 4096, 14336),
    "decode": (4, 16, 28672, 8192),
}


def rng(index: int, stream: int) -> np.random.Generator:
    """The generator for one matrix of one workload."""
    return np.random.Generator(np.random.PCG64([SEED_BASE + index, stream]))


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def with_outliers(g: np.random.Generator, x: np.ndarray, p: float, factor: float) -> np.ndarray:
    """Multiply an i.i.d. Bernoulli(p) subset of the entries by ``factor``."""
    mask = g.random(x.shape, dtype=np.float32) < np.float32(p)
    x[mask] *= np.float32(factor)
    return x


def row_factor_pow2_uniform(g: np.random.Generator, rows: int, lo: float, hi: float) -> np.ndarray:
    """A per-row magnitude 2^U(lo, hi) (float32, one value per row)."""
    u = g.uniform(lo, hi, size=rows)
    return np.exp2(u).astype(np.float32)


def laplace(g: np.random.Generator, shape, scale: float) -> np.ndarray:
    return g.laplace(0.0, scale, size=shape).astype(np.float32)


def make(name: str, m: int | None = None, n: int | None = None, k: int | None = None,
         rows_a: int | None = None):
    """Return ``(A, B)`` float32 source matrices of a workload.

    A is M x K and B is N x K.  ``m``, ``n``, ``k`` override the workload's
    sizes (same distributions, smaller or ragged shapes for parity tests).
    ``rows_a`` is an alias for ``m`` used by the decode workload.
    """
    idx, M, N, K = WORKLOADS[name]
    M = m if m is not None else (rows_a if rows_a is not None else M)
    N = n if n is not None else N
    K = k if k is not None else K
    ga, gb = rng(idx, 1), rng(idx, 2)
    if name == "fp8_256":
        A = with_outliers(ga, normal(ga, (M, K)), 0.001, 100.0)
        B = with_outliers(gb, normal(gb, (N, K)), 0.001, 100.0)
    elif name == "mxfp4_1024":
        A = normal(ga, (M, K)) * row_factor_pow2_uniform(ga, M, -8.0, 8.0)[:, None]
        B = normal(gb, (N, K)) * row_factor_pow2_uniform(gb, N, -8.0, 8.0)[:, None]
    elif name == "ffn_up":
        A = with_outliers(ga, normal(ga, (M, K)), 0.001, 50.0)
        B = normal(gb, (N, K), 0.02)
    elif name == "dgrad":
        A = laplace(ga, (M, K), 1e-3) * row_factor_pow2_uniform(ga, M, -12.0, 0.0)[:, None]
        B = normal(gb, (N, K), 0.02)
    elif name == "decode":
        gx = rng(idx, 3)
        A = normal(gx, (M, K))
        B = normal(gb, (N, K), 0.02)
    else:  # pragma: no cover - guarded by the WORKLOADS lookup above
        raise KeyError(name)
    return np.ascontiguousarray(A, dtype=np.float32), np.ascontiguousarray(B, dtype=np.float32)


def addend(name: str, m: int, n: int) -> np.ndarray:
    """An optional FP32 addend C (M x N), ~N(0,1)."""
    idx = WORKLOADS[name][0]
    return normal(rng(idx, 4), (m, n))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even) and return uint16 bits.

    Used to hand BF16 source activations to both sides; finite inputs only.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)

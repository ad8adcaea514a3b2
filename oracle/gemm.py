"""Block-scaled GEMM in FP64 (CPU oracle; test infrastructure only).

D = sum_k (s_A a_k)(s_B b_k) + C with the codes a, b decoded from their bit
fields and the scales applied per K block:

* FP8 ("FP8 GEMM on CDNA4", §3.3 and §4.4): the scales are FP32 and constant
  over a 128-wide K tile, so D = sum_t (s_A,t * s_B,t) * P_t + C where
  P_t = sum_{k in tile t} a_k b_k.  For E4M3 x E4M3 every P_t is exact in FP64:
  products are multiples of 2^-18 below 2^17.6, so 128 of them need at most
  43 significant bits.  s_A,t * s_B,t is a product of two FP32 values and is
  exact in FP64.  Only the multiplication by P_t and the sum over tiles round
  (relative error ~1e-16, far below the comparison tolerance).
* MXFP4 ("Rubin FP4 GEMM deep dive", §2.2 and §3.1): every element is an E2M1
  value times an E8M0 power of two, exact in FP64; D = (s_A a)(s_B b)^T + C.
* MXFP8 (the same K-blocked rule with FP8 E4M3 / E5M2 elements): every
  element is an FP8 value times an E8M0 power of two, exact in FP64.

Both also return the per-element bound  Bnd_ij = sum_k |s_A a_k s_B b_k|,
used by the tolerance |D_gpu - D| <= 1e-4 * Bnd + 1e-6.

Operand layouts follow the pages ("FP8 GEMM on CDNA4", §3.1; "Rubin FP4 GEMM
deep dive", §3.1): A is M x K row-major, B is K x N column-major, i.e. stored
as N rows of K contiguous values.
"""
from __future__ import annotations

import numpy as np

from . import formats

TILE = 128


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def gemm_fp8(A: np.ndarray, fa: str, sA: np.ndarray, ga: str,
             B: np.ndarray, fb: str, sB: np.ndarray, gb: str,
             C: np.ndarray | None = None, rows=None):
    """FP8 block-scaled GEMM.

    A: uint8 codes M x K; B: uint8 codes N x K.
    sA: "tile" -> [ceil(M/128)][ceil(K/128)]; "row" -> [ceil(K/128)][M].
    sB: "tile" -> [ceil(N/128)][ceil(K/128)]; "row" -> [ceil(K/128)][N].
    rows: optional array of row indices of D to compute (sampling large shapes).
    Returns (D, Bnd) as float64 arrays of shape (len(rows) or M) x N.
    """
    M, K = A.shape
    N = B.shape[0]
    ri = np.arange(M) if rows is None else np.asarray(rows)
    a = formats.decode_array(A[ri], fa)
    b = formats.decode_array(B, fb)
    D = np.zeros((len(ri), N), dtype=np.float64)
    Bnd = np.zeros((len(ri), N), dtype=np.float64)
    for t in range(_cdiv(K, TILE)):
        ks = slice(t * TILE, min((t + 1) * TILE, K))
        P = a[:, ks] @ b[:, ks].T
        Pabs = np.abs(a[:, ks]) @ np.abs(b[:, ks]).T
        sa = (sA[ri // TILE, t] if ga == "tile" else sA[t, ri]).astype(np.float64)
        sb = (sB[np.arange(N) // TILE, t] if gb == "tile" else sB[t, :]).astype(np.float64)
        S = sa[:, None] * sb[None, :]
        D += S * P
        Bnd += np.abs(S) * Pabs
    if C is not None:
        D += np.asarray(C, dtype=np.float64)[ri]
    return D, Bnd


def mxfp4_values(packed: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Real values s * a of a packed MXFP4 matrix (rows x K) with row-major
    E8M0 scales (rows x K/32), exact in FP64."""
    codes = formats.unpack_e2m1(packed)
    vals = formats.decode_array(codes, "e2m1")
    scale = formats.decode_e8m0_array(sf)
    R, K = vals.shape
    return (vals.reshape(R, K // 32, 32) * scale[:, :, None]).reshape(R, K)


def gemm_mxfp4(A: np.ndarray, sfA: np.ndarray, B: np.ndarray, sfB: np.ndarray,
               C: np.ndarray | None = None, rows=None):
    """MXFP4 GEMM. A: packed M x K/2, sfA M x K/32; B: packed N x K/2,
    sfB N x K/32 (scales row-major).  Returns (D, Bnd) in FP64."""
    M = A.shape[0]
    ri = np.arange(M) if rows is None else np.asarray(rows)
    a = mxfp4_values(A[ri], sfA[ri])
    b = mxfp4_values(B, sfB)
    D = a @ b.T
    Bnd = np.abs(a) @ np.abs(b).T
    if C is not None:
        D += np.asarray(C, dtype=np.float64)[ri]
    return D, Bnd


def mx_values(codes: np.ndarray, fmt: str, sf: np.ndarray) -> np.ndarray:
    """Real values s * a of an MX matrix (rows x K): FP8 codes one per byte
    (fmt "e4m3" / "e5m2") or packed E2M1 (fmt "e2m1"), with row-major E8M0
    scales (rows x K/32), exact in FP64."""
    if fmt == "e2m1":
        return mxfp4_values(codes, sf)
    vals = formats.decode_array(codes, fmt)
    scale = formats.decode_e8m0_array(sf)
    R, K = vals.shape
    return (vals.reshape(R, K // 32, 32) * scale[:, :, None]).reshape(R, K)


def gemm_mxfp8(A: np.ndarray, fa: str, sfA: np.ndarray, B: np.ndarray, fb: str, sfB: np.ndarray,
               C: np.ndarray | None = None, rows=None):
    """MXFP8 GEMM. A: FP8 codes M x K (format fa), sfA M x K/32; B: FP8 codes
    N x K (format fb), sfB N x K/32 (scales row-major).  Returns (D, Bnd) in
    FP64."""
    M = A.shape[0]
    ri = np.arange(M) if rows is None else np.asarray(rows)
    a = mx_values(A[ri], fa, sfA[ri])
    b = mx_values(B, fb, sfB)
    D = a @ b.T
    Bnd = np.abs(a) @ np.abs(b).T
    if C is not None:
        D += np.asarray(C, dtype=np.float64)[ri]
    return D, Bnd


def within_tolerance(D_gpu: np.ndarray, D_ref: np.ndarray, Bnd: np.ndarray,
                     bf16: bool = False):
    """Elementwise check of |D_gpu - D_ref| <= 1e-4 * Bnd + 1e-6, plus
    8e-3 * |D_ref| for BF16 outputs (their own rounding).  Returns
    (ok: bool, worst ratio err / allowed)."""
    err = np.abs(np.asarray(D_gpu, dtype=np.float64) - D_ref)
    allowed = 1e-4 * Bnd + 1e-6
    if bf16:
        allowed = allowed + 8e-3 * np.abs(D_ref)
    ratio = err / allowed
    return bool(np.all(err <= allowed)), float(np.max(ratio)) if ratio.size else 0.0

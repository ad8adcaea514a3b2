"""Quantisers of the block-scaled GEMM (CPU oracle; test infrastructure only).

FP8 per-tile quantiser - "FP8 GEMM on CDNA4", §3.3 and §4.2:
  the scale of a tile is its largest magnitude divided by the format's largest
  value (448 for E4M3), every element is divided by the scale and stored as
  FP8, and the GEMM multiplies the accumulated result by s_A * s_B (§4.4).
  The tile is the granularity the page settles on (§3.3, §6); the workloads add
  a 1 x 128 granularity for activations.

MXFP4 quantiser - "Rubin FP4 GEMM deep dive", §4.2 steps 1-3 and §2.2:
  per block of 32 elements along K, take the largest magnitude, divide by 6
  (the E2M1 maximum), round that to the nearest power of two and store it as
  an E8M0 code, divide the elements by the power of two, round to E2M1 and
  pack two codes per byte, first element in the low nibble.

MXFP8 quantiser - the same MX rule (§2.2: 32 elements along K share one E8M0
  scale; §4.2 steps 1-3) with FP8 elements: the block maximum is divided by the
  FP8 format's largest value (448 for E4M3, 57344 for E5M2) instead of 6, and
  the scaled elements are rounded to that FP8 format; one code per byte.  The
  pages give the rule for E2M1 only; taking it unchanged for FP8 elements is a
  reading (the "smaller formats share the block structure" of §2.2).

NVFP4 quantiser - "Rubin FP4 GEMM deep dive", §5.3 (smaller blocks, 16
  elements, give finer scales at twice the scale storage) and §2.2 (the block
  scale is kept in a higher-precision format such as FP8): per block of 16
  elements along K, v = max_abs / 6 (FP32), the scale code is v / g rounded to
  E4M3 (RNE, saturating at 448; g is an FP32 tensor scale, 1 by default, that
  keeps v / g inside E4M3's range), the block's scale is s = fl32(E4M3(code)
  * g), and each element is RNE_satfinite_E2M1(fl32(x / s)); a block whose s
  is 0 stores all-zero codes.  The tensor scale g is not on the pages: it is
  the reading that lets an E4M3 scale cover data of any magnitude (the
  dynamic-range concern of §3.2); the GEMM multiplies its sum by g_A * g_B.

FP4 with 16-bit block scales - "Rubin FP4 GEMM deep dive", §3.2: where the
  power-of-two E8M0 scale is too coarse, the block scale may be kept in FP16
  or BF16 at twice the scale bytes.  Per block of 32 elements along K (the MX
  block of §2.2): v = max_abs / 6 (FP32, round to nearest), the scale is v
  rounded to nearest (ties to even) in BF16 or FP16, saturating at the
  format's largest finite value; every element is
  RNE_satfinite_E2M1(fl32(x / s)) by IEEE division; a block whose scale is 0
  stores all-zero codes.  Scales are stored K-block major, [K/32][rows] of
  16-bit codes, so one K block's scales are contiguous.  The rounding of v,
  the saturation and the layout are readings; the page fixes only the
  format of the scale.

Readings where the pages leave a step open (also listed in the design notes):
  * the scale is s = max_abs / fmt_max computed in FP32 with round-to-nearest,
    and the element is q = RNE_satfinite(x / s) with an IEEE FP32 division
    (not a multiplication by 1/s);
  * fmt_max is the format's own maximum: 448 for E4M3, 57344 for E5M2; any
    other positive value may be passed (e.g. 448 for E5M2);
  * an all-zero group (or one whose FP32 scale underflows to 0) gets s = 1.0;
  * "nearest power of two" is nearest in linear distance on v = max_abs / 6
    (FP32); a tie (v = 1.5 * 2^e) goes to the larger power; v = 0 gives
    E8M0 code 127 (1.0); codes are clamped to [0, 254].
"""
from __future__ import annotations

import math

import numpy as np

from . import formats

TILE = 128        # FP8 scale tile along both dimensions (and along K for 1x128)
MX_BLOCK = 32     # MXFP4 block along K
NV_BLOCK = 16     # NVFP4 block along K


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def fmt_max_default(fmt: str) -> float:
    return formats.max_finite(fmt)


def fp8_scale(amax: np.float32, fmt_max: float) -> np.float32:
    """s = max_abs / fmt_max in FP32 (round to nearest); 1.0 if that is 0."""
    s = np.float32(amax) / np.float32(fmt_max)
    if s == 0:
        s = np.float32(1.0)
    return np.float32(s)


def quantize_fp8(x: np.ndarray, fmt: str, gran: str, fmt_max: float | None = None):
    """Quantise a row-major float32 matrix (rows x cols, cols = K) to FP8.

    gran = "tile"  : one scale per 128 x 128 tile, scales[ceil(R/128)][ceil(C/128)]
    gran = "row"   : one scale per 1 x 128 run of a row, stored K-tile major,
                     scales[ceil(C/128)][R]
    Ragged edge tiles cover what is left.  Returns (codes uint8 R x C,
    scales float32).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    fm = fmt_max_default(fmt) if fmt_max is None else float(fmt_max)
    codes = np.empty((R, C), dtype=np.uint8)
    if gran == "tile":
        scales = np.empty((_cdiv(R, TILE), _cdiv(C, TILE)), dtype=np.float32)
        for ti in range(scales.shape[0]):
            for tj in range(scales.shape[1]):
                blk = x[ti * TILE:(ti + 1) * TILE, tj * TILE:(tj + 1) * TILE]
                s = fp8_scale(np.max(np.abs(blk)), fm)
                scales[ti, tj] = s
                codes[ti * TILE:(ti + 1) * TILE, tj * TILE:(tj + 1) * TILE] = \
                    formats.encode(blk / s, fmt)
    elif gran == "row":
        scales = np.empty((_cdiv(C, TILE), R), dtype=np.float32)
        for tj in range(scales.shape[0]):
            blk = x[:, tj * TILE:(tj + 1) * TILE]
            amax = np.max(np.abs(blk), axis=1)
            s = np.array([fp8_scale(a, fm) for a in amax], dtype=np.float32)
            scales[tj, :] = s
            codes[:, tj * TILE:(tj + 1) * TILE] = formats.encode(blk / s[:, None], fmt)
    else:
        raise ValueError(gran)
    return codes, scales


def e8m0_nearest_pow2(v: np.float32) -> int:
    """E8M0 code of the power of two nearest to v (linear distance, ties up)."""
    v = float(np.float32(v))
    if v == 0.0:
        return 127
    f, x = math.frexp(v)            # v = f * 2^x, 0.5 <= f < 1, exact
    lower = math.ldexp(1.0, x - 1)  # 2^floor(log2 v)
    upper = 2.0 * lower
    e = (x - 1) if (v - lower) < (upper - v) else x
    return int(min(max(e + 127, 0), 254))


def quantize_mxfp4(x: np.ndarray):
    """Quantise a row-major float32 matrix (rows x K, K % 32 == 0) to MXFP4.

    Returns (packed uint8 R x K/2, sf uint8 R x K/32) with the scale factors in
    the canonical row-major layout.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    if K % MX_BLOCK:
        raise ValueError("K must be a multiple of 32")
    nb = K // MX_BLOCK
    sf = np.empty((R, nb), dtype=np.uint8)
    codes = np.empty((R, K), dtype=np.uint8)
    blocks = x.reshape(R, nb, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    v = amax / np.float32(6.0)                     # FP32, round to nearest
    for r in range(R):
        for b in range(nb):
            sf[r, b] = e8m0_nearest_pow2(v[r, b])
    pow2 = np.ldexp(1.0, -(sf.astype(np.int64) - 127))    # 2^-E, exact in FP64
    scaled = blocks.astype(np.float64) * pow2[:, :, None]  # exact
    codes[:] = formats.encode(scaled.reshape(R, K), "e2m1")
    return formats.pack_e2m1(codes), sf


def quantize_mxfp8(x: np.ndarray, fmt: str, fmt_max: float | None = None):
    """Quantise a row-major float32 matrix (rows x K, K % 32 == 0) to MXFP8:
    fmt "e4m3" or "e5m2" elements, one E8M0 scale per 32 elements along K.

    Per block: v = max_abs / fmt_max in FP32 (round to nearest), E = the power
    of two nearest to v (same reading as MXFP4: linear distance, ties up,
    v = 0 -> code 127, codes clamped to [0, 254]), element = RNE_satfinite of
    x * 2^-E (exact in FP64) in the FP8 format.  Returns (codes uint8 R x K,
    sf uint8 R x K/32) with row-major scale factors.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    if K % MX_BLOCK:
        raise ValueError("K must be a multiple of 32")
    if fmt not in ("e4m3", "e5m2"):
        raise ValueError(fmt)
    fm = np.float32(fmt_max_default(fmt) if fmt_max is None else fmt_max)
    nb = K // MX_BLOCK
    blocks = x.reshape(R, nb, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    v = amax / fm                                  # FP32, round to nearest
    sf = np.empty((R, nb), dtype=np.uint8)
    for r in range(R):
        for b in range(nb):
            sf[r, b] = e8m0_nearest_pow2(v[r, b])
    pow2 = np.ldexp(1.0, -(sf.astype(np.int64) - 127))    # 2^-E, exact in FP64
    scaled = blocks.astype(np.float64) * pow2[:, :, None]  # exact
    codes = formats.encode(scaled.reshape(R, K), fmt)
    return codes.astype(np.uint8), sf


def quantize_nvfp4(x: np.ndarray, tensor_scale: float = 1.0):
    """Quantise a row-major float32 matrix (rows x K, K % 16 == 0) to NVFP4:
    E2M1 elements, one E4M3 scale per 16 elements along K, an FP32 tensor
    scale g.  Returns (packed uint8 R x K/2, sf uint8 R x K/16 E4M3 codes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    if K % NV_BLOCK:
        raise ValueError("K must be a multiple of 16")
    g = np.float32(tensor_scale)
    if not (np.isfinite(g) and g > 0):
        raise ValueError("tensor_scale must be positive and finite")
    nb = K // NV_BLOCK
    blocks = x.reshape(R, nb, NV_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    v = amax / np.float32(6.0)                          # FP32, round to nearest
    u = v / g                                           # FP32, round to nearest
    sf = formats.encode(u, "e4m3").astype(np.uint8)     # RNE, saturating at 448
    s = (formats.decode_array(sf, "e4m3").astype(np.float32) * g).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s)
    q = (blocks / safe[:, :, None]).astype(np.float32)  # IEEE FP32 division
    codes = formats.encode(q.reshape(R, K), "e2m1").reshape(R, nb, NV_BLOCK)
    codes[s == 0] = 0
    return formats.pack_e2m1(codes.reshape(R, K).astype(np.uint8)), sf


def quantize_fp4_bs16(x: np.ndarray, scale_fmt: str = "bf16"):
    """Quantise a row-major float32 matrix (rows x K, K % 32 == 0) to E2M1
    elements with one 16-bit ("bf16" or "f16") scale per 32 along K.

    Returns (packed uint8 R x K/2, sf uint16 [K/32][R] scale codes)."""
    if scale_fmt not in ("bf16", "f16"):
        raise ValueError(scale_fmt)
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, K = x.shape
    if K % MX_BLOCK:
        raise ValueError("K must be a multiple of 32")
    nb = K // MX_BLOCK
    blocks = x.reshape(R, nb, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    v = amax / np.float32(6.0)                                # FP32, round to nearest
    sf = formats.encode(v, scale_fmt)                         # RNE, satfinite, uint16
    s = formats.decode_array(sf, scale_fmt).astype(np.float32)   # exact
    safe = np.where(s == 0, np.float32(1.0), s)
    q = (blocks / safe[:, :, None]).astype(np.float32)        # IEEE FP32 division
    codes = formats.encode(q.reshape(R, K), "e2m1").reshape(R, nb, MX_BLOCK)
    codes[s == 0] = 0
    return formats.pack_e2m1(codes.reshape(R, K).astype(np.uint8)), np.ascontiguousarray(sf.T)


def sf_to_tcgen05_layout(sf: np.ndarray, pad: int = 127) -> np.ndarray:
    """Rearrange row-major E8M0 scales [R][KB] into the storage order the
    block-scaled tensor-core MMA reads them in (not from the pages; NVIDIA's
    documented 128-row x 4-scale atom): atoms of 512 bytes, ordered by
    (row block of 128, group of 4 K-blocks); inside an atom the byte of row r,
    K-block c is at (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4).
    Padding bytes (rows beyond R, K-blocks beyond KB) hold `pad`: 127 (E8M0
    1.0) for E8M0 scales, 0 for E4M3 scales.
    """
    R, KB = sf.shape
    rb, cb = _cdiv(R, 128), _cdiv(KB, 4)
    out = np.full(rb * cb * 512, pad, dtype=np.uint8)
    r = np.arange(R)[:, None]
    c = np.arange(KB)[None, :]
    off = ((r // 128) * cb + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    out[off] = sf
    return out

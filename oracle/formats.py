"""Number formats of the block-scaled GEMM, decoded from their bit fields.

Test infrastructure (see the package docstring): imported only by tests, the
smoke check and the bench's CPU baseline.

Formats and where the pages define them:

* FP8 E4M3 - 1 sign, 4 exponent, 3 mantissa bits; largest finite value 448
  ("FP8 GEMM on CDNA4", §1.3 and §3.3).  It is the "fn" variant: no infinity,
  exponent 1111 with mantissa 111 is NaN, so 448 = 1.75 * 2^8 is the maximum
  (the page's 448, and torch.float8_e4m3fn in "FP8 MMA internals on Hopper").
* FP8 E5M2 - 1 sign, 5 exponent, 2 mantissa bits ("FP8 GEMM on CDNA4", §1.3):
  IEEE-like, bias 15, exponent 11111 is Inf (mantissa 0) or NaN; max 57344.
* FP4 E2M1 - 1 sign, 2 exponent, 1 mantissa bit; magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6} ("Rubin FP4 GEMM deep dive", §2.1), max 6 (§4.2).
* E8M0 - 8 exponent bits, no mantissa, powers of two only ("Rubin FP4 GEMM deep
  dive", §2.2); bias 127, code 0xFF is NaN (the OCP MX convention; the page
  says only "8-bit exponent, 0-bit mantissa").
* BF16 and FP16 - the 16-bit block-scale formats that "Rubin FP4 GEMM deep
  dive", §3.2 offers where E8M0 is too coarse: BF16 is 1 sign, 8 exponent
  (bias 127), 7 mantissa bits; FP16 is 1 sign, 5 exponent (bias 15), 10
  mantissa bits; both IEEE-style (subnormals at exponent 0, the all-ones
  exponent is Inf / NaN).

Encoders round to the nearest representable value; a value exactly half way
between two neighbours goes to the one whose code is even (the code's last bit
is the mantissa's last bit, so this is IEEE round-half-to-even).  Magnitudes
beyond the largest finite value saturate to it ("satfinite").  The sign bit is
the input's sign bit, so -0.0 and negative values that round to zero give the
negative-zero code.
"""
from __future__ import annotations

import functools
import math
from fractions import Fraction

import numpy as np

NAN = float("nan")


# ----------------------------------------------------------------- decoders --
def decode_e4m3(code: int) -> float:
    """E4M3 (fn): bias 7, subnormals at exponent 0, S.1111.111 is NaN."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return NAN
    if e == 0:
        return s * m * 2.0 ** (-3) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def decode_e5m2(code: int) -> float:
    """E5M2: bias 15, subnormals at exponent 0, exponent 31 is Inf / NaN."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 2) & 0x1F
    m = code & 0x3
    if e == 0x1F:
        return s * math.inf if m == 0 else NAN
    if e == 0:
        return s * m * 2.0 ** (-2) * 2.0 ** (1 - 15)
    return s * (1.0 + m / 4.0) * 2.0 ** (e - 15)


def decode_e2m1(code: int) -> float:
    """E2M1 (4-bit code): bias 1, subnormal at exponent 0, no Inf or NaN."""
    s = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


def decode_e8m0(code: int) -> float:
    """E8M0: the power of two 2^(code-127); 0xFF is NaN."""
    if code == 0xFF:
        return NAN
    return 2.0 ** (code - 127)


def _decode_ieee16(code: int, ebits: int) -> float:
    mbits = 15 - ebits
    bias = (1 << (ebits - 1)) - 1
    s = -1.0 if (code >> 15) & 1 else 1.0
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == (1 << ebits) - 1:
        return s * math.inf if m == 0 else NAN
    if e == 0:
        return s * m * 2.0 ** (-mbits) * 2.0 ** (1 - bias)
    return s * (1.0 + m / 2.0 ** mbits) * 2.0 ** (e - bias)


def decode_bf16(code: int) -> float:
    """BF16: bias 127, 7 mantissa bits, subnormals at exponent 0."""
    return _decode_ieee16(code, 8)


def decode_f16(code: int) -> float:
    """FP16: bias 15, 10 mantissa bits, subnormals at exponent 0."""
    return _decode_ieee16(code, 5)


FORMATS = {
    # name: (decoder, code bits)
    "e4m3": (decode_e4m3, 8),
    "e5m2": (decode_e5m2, 8),
    "e2m1": (decode_e2m1, 4),
    "bf16": (decode_bf16, 16),
    "f16": (decode_f16, 16),
}

# The largest finite magnitude of each element format, read off the decoder.
def max_finite(fmt: str) -> float:
    dec, bits = FORMATS[fmt]
    vals = [dec(c) for c in range(1 << bits)]
    return max(v for v in vals if math.isfinite(v))


@functools.lru_cache(maxsize=None)
def _decode_table_cached(fmt: str) -> np.ndarray:
    dec, bits = FORMATS[fmt]
    t = np.array([dec(c) for c in range(1 << bits)], dtype=np.float64)
    t.setflags(write=False)
    return t


def decode_table(fmt: str) -> np.ndarray:
    """float64 value of every code of a format (index = code)."""
    return _decode_table_cached(fmt)


@functools.lru_cache(maxsize=None)
def _positive_ladder(fmt: str):
    """Sorted (value, code) pairs of the non-negative finite codes."""
    dec, bits = FORMATS[fmt]
    sign = 1 << (bits - 1)
    pairs = []
    for c in range(sign):          # codes with the sign bit clear
        v = dec(c)
        if math.isfinite(v):
            pairs.append((v, c))
    pairs.sort()
    vals = np.array([p[0] for p in pairs], dtype=np.float64)
    codes = np.array([p[1] for p in pairs], dtype=np.int64)
    return vals, codes


# ----------------------------------------------------------------- encoders --
def encode(x, fmt: str) -> np.ndarray:
    """Round float32 values to the nearest code of ``fmt`` (ties to the even
    code), saturating to the largest finite magnitude.

    Works on the exact binary value of each input: the midpoint between two
    neighbouring codes is exactly representable in FP64, so each decision is
    an exact comparison.  NaN inputs give the format's NaN code (E4M3 0x7F,
    E5M2 0x7F); E2M1 has no NaN and NaN inputs are rejected, and so are NaN
    inputs to the 16-bit scale formats (a scale is never NaN).
    Returns uint8 codes (E2M1 codes in the low nibble, unpacked), or uint16
    codes for BF16 / FP16.
    """
    dec, bits = FORMATS[fmt]
    sign_bit = 1 << (bits - 1)
    x = np.asarray(x, dtype=np.float32)
    xd = x.astype(np.float64)
    mag = np.abs(xd)
    vals, codes = _positive_ladder(fmt)
    vmax = vals[-1]
    nan = np.isnan(xd)
    if fmt not in ("e4m3", "e5m2") and nan.any():
        raise ValueError(f"{fmt}: NaN input")
    m = np.where(nan, 0.0, np.minimum(mag, vmax))
    # v[i] <= m < v[i+1]
    i = np.searchsorted(vals, m, side="right") - 1
    i = np.clip(i, 0, len(vals) - 1)
    lo_v = vals[i]
    hi_i = np.minimum(i + 1, len(vals) - 1)
    hi_v = vals[hi_i]
    mid = (lo_v + hi_v) / 2.0            # exact: one more bit than the codes
    lo_c = codes[i]
    hi_c = codes[hi_i]
    pick_hi = (m > mid) | ((m == mid) & (hi_c % 2 == 0) & (hi_i != i))
    out = np.where(pick_hi, hi_c, lo_c)
    out = np.where(m >= vmax, codes[-1], out)
    neg = np.signbit(x)
    out = np.where(neg, out | sign_bit, out)
    if fmt in ("e4m3", "e5m2"):
        out = np.where(nan, 0x7F, out)
    return out.astype(np.uint16 if bits == 16 else np.uint8)


def encode_one_exact(value: Fraction, fmt: str) -> int:
    """Brute-force reference for a single value given as an exact rational:
    scan every finite code, take the nearest, break ties toward the even code.
    Used by the tests to check ``encode`` on hand-built midpoints."""
    dec, bits = FORMATS[fmt]
    best = None
    for c in range(1 << bits):
        v = dec(c)
        if not math.isfinite(v):
            continue
        if (v < 0) != (value < 0) and v != 0:
            continue
        if v == 0 and (c >> (bits - 1)) != (1 if value < 0 else 0):
            continue
        d = abs(Fraction(v) - value)
        key = (d, c % 2)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


# ------------------------------------------------------------------ packing --
def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: the first element in the
    low nibble, the second in the high nibble ("Rubin FP4 GEMM deep dive", §4.2
    step 3)."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0
    lo = codes[..., 0::2] & 0xF
    hi = codes[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def decode_array(codes: np.ndarray, fmt: str) -> np.ndarray:
    """float64 values of an array of (unpacked) codes."""
    return decode_table(fmt)[np.asarray(codes, dtype=np.int64)]


def decode_e8m0_array(codes: np.ndarray) -> np.ndarray:
    table = np.array([decode_e8m0(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.int64)]

"""Pins of the oracle's FP4-with-16-bit-block-scales functions ("Rubin FP4
GEMM deep dive", §3.2: FP16/BF16 block scales where E8M0 is too coarse).

Each check is tied to something other than the oracle itself: the IEEE bit
layouts (read back through numpy / torch reinterpretation and casts), blocks
worked by hand, the page's "twice the scale bytes", exact rational
arithmetic, and a hand-built case where the per-block FP32 promotion rounds."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats
from oracle import gemm as og
from oracle import quantize as oq


def test_f16_decoder_matches_ieee_half_for_every_code():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = formats.decode_array(codes, "f16")
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_bf16_decoder_matches_the_top_half_of_fp32_for_every_code():
    codes = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (codes << 16).view(np.float32).astype(np.float64)
    got = formats.decode_array(codes, "bf16")
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert formats.max_finite("bf16") == float(np.float32(3.3895313892515355e38))
    assert formats.max_finite("f16") == 65504.0


def _wide_f32(n, lo, hi, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal(n) * np.exp2(g.uniform(lo, hi, n))).astype(np.float32)


def test_f16_encoder_matches_the_ieee_cast_inside_the_range():
    x = _wide_f32(200_000, -30, 16, 1)
    # the exact midpoints between neighbouring FP16 values, and one FP32 ulp either side
    h = np.arange(0x0001, 0x7BFF, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = (np.arange(0x0001, 0x7BFF, 37, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    mid = ((h + nxt) / 2).astype(np.float32)
    x = np.concatenate([x, mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))])
    x = x[np.abs(x) <= 65504]
    assert np.array_equal(formats.encode(x, "f16"), x.astype(np.float16).view(np.uint16))
    # beyond the largest finite value the scale saturates (reading), not Inf
    assert formats.encode(np.array([70000.0, -1e9], np.float32), "f16").tolist() == [0x7BFF, 0xFBFF]


def test_bf16_encoder_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    x = _wide_f32(200_000, -120, 120, 2)
    # FP32 values whose low 16 bits are exactly the half way point (0x8000), and its neighbours
    u = (np.random.default_rng(3).integers(0x00800000, 0x7F000000, 5000, dtype=np.uint32) & 0xFFFF0000) | 0x8000
    ties = u.view(np.float32)
    x = np.concatenate([x, ties, -ties, np.nextafter(ties, np.float32(0))])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(formats.encode(x, "bf16"), ref)


@pytest.mark.parametrize("fmt,value", [("bf16", Fraction(7, 6)), ("f16", Fraction(7, 6)),
                                       ("f16", Fraction(2049, 2048) / 3), ("bf16", Fraction(-257, 256))])
def test_16bit_encoder_against_exact_rational_search(fmt, value):
    v32 = np.float32(float(value))
    assert int(formats.encode(np.array([v32]), fmt)[0]) == formats.encode_one_exact(Fraction(float(v32)), fmt)


@pytest.mark.parametrize("fmt,scale_code,scale,elems", [
    # max 7 -> v = fl32(7/6) = 1.0010101 0101...b; BF16 keeps 7 fraction bits and the next
    # bit is 0: s = 1 + 21/128 = 1.1640625.  7/s = 6.013 -> saturates to 6; 3.5/s = 3.007
    # -> 3; 1/s = 0.859 -> 1 (above the 0.75 midpoint); -0.6/s = -0.515 -> -0.5
    ("bf16", 0x3F95, 1.1640625, [7, 5, 2, 9, 0]),
    # FP16 keeps 10 fraction bits: 1.0010101010|1010...b rounds up, s = 1 + 171/1024;
    # 7/s = 5.998 -> 6; 3.5/s = 2.999 -> 3; 1/s = 0.857 -> 1; -0.6/s = -0.514 -> -0.5
    ("f16", 0x3C00 | 171, 1.1669921875, [7, 5, 2, 9, 0]),
])
def test_quantiser_hand_worked_block(fmt, scale_code, scale, elems):
    x = np.zeros((1, 32), np.float32)
    x[0, :4] = [7.0, 3.5, 1.0, -0.6]
    q, sf = oq.quantize_fp4_bs16(x, fmt)
    assert sf.shape == (1, 1) and int(sf[0, 0]) == scale_code
    assert formats.decode_array(sf, fmt)[0, 0] == scale
    codes = formats.unpack_e2m1(q)[0]
    assert codes[:5].tolist() == elems
    assert (codes[5:] == 0).all()


def test_quantiser_ties_go_to_the_even_code_at_unit_scale():
    # block maximum 6 -> v = 1 exactly -> s = 1: the elements are cast unscaled
    x = np.zeros((1, 32), np.float32)
    x[0, :6] = [6.0, 2.5, 5.0, 0.25, 1.25, 1.75]
    for fmt in ("bf16", "f16"):
        q, sf = oq.quantize_fp4_bs16(x, fmt)
        assert formats.decode_array(sf, fmt)[0, 0] == 1.0
        # 2.5 -> 2 (code 4), 5 -> 4 (code 6), 0.25 -> 0, 1.25 -> 1 (code 2), 1.75 -> 2 (code 4)
        assert formats.unpack_e2m1(q)[0, :6].tolist() == [7, 4, 6, 0, 2, 4]


def test_quantiser_zero_saturated_and_underflowing_blocks():
    x = np.zeros((3, 64), np.float32)
    x[1, 32:40] = 420000.0 * np.array([1, -1, 0.5, 0.25, 0, 0, 0, 0])
    x[2, :32] = 1e-9
    q, sf = oq.quantize_fp4_bs16(x, "f16")
    # an all-zero block: scale code 0, codes 0
    assert int(sf[0, 0]) == 0 and (formats.unpack_e2m1(q)[0] == 0).all()
    # v = 70000 saturates to FP16's 65504; 420000 / 65504 = 6.41 saturates to 6
    assert int(sf[1, 1]) == 0x7BFF
    assert formats.unpack_e2m1(q)[1, 32:34].tolist() == [7, 15]
    # v = 1.7e-10 underflows FP16 (below 2^-25): scale 0, the block stores zero codes
    assert int(sf[0, 2]) == 0 and (formats.unpack_e2m1(q)[2, :32] == 0).all()
    q2, sf2 = oq.quantize_fp4_bs16(x, "bf16")     # BF16 keeps FP32's exponent range
    assert int(sf2[0, 2]) != 0 and (formats.unpack_e2m1(q2)[2, :32] == 7).all()


def test_16bit_scales_cost_twice_the_e8m0_scale_bytes():
    # "Rubin FP4 GEMM deep dive" §3.2: for a K = 4096 row, 128 bytes of E8M0 scales
    # against 2048 bytes of data; FP16 / BF16 scales take twice that
    x = np.random.default_rng(4).standard_normal((2, 4096)).astype(np.float32)
    q, sf = oq.quantize_fp4_bs16(x, "bf16")
    _, sf8 = oq.quantize_mxfp4(x)
    assert q[0].nbytes == 2048 and sf8[0].nbytes == 128
    assert sf[:, 0].nbytes == 2 * sf8[0].nbytes == 256


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_quantiser_reconstruction_bound(fmt):
    g = np.random.default_rng(5)
    x = (g.standard_normal((64, 512)) * np.exp2(g.uniform(-8, 8, (64, 1)))).astype(np.float32)
    q, sf = oq.quantize_fp4_bs16(x, fmt)
    vals = og.fp4_bs16_values(q, sf, fmt).reshape(64, 16, 32)
    s = formats.decode_array(sf.T, fmt)[:, :, None]
    blocks = x.reshape(64, 16, 32).astype(np.float64)
    amax = np.max(np.abs(blocks), axis=2, keepdims=True)
    # E2M1 steps are at most 2 (4 -> 6), so the error is at most s inside the range;
    # a scale rounded down by up to one part in 2^8 (BF16) pushes the maximum past 6 s
    assert np.all(np.abs(blocks - vals) <= s + amax * 2.0 ** -7)


def _exact_gemm(qa, sfa, qb, sfb, fmt):
    a = formats.decode_array(formats.unpack_e2m1(qa), "e2m1")
    b = formats.decode_array(formats.unpack_e2m1(qb), "e2m1")
    sa = formats.decode_array(sfa, fmt)
    sb = formats.decode_array(sfb, fmt)
    M, K = a.shape
    N = b.shape[0]
    D = np.empty((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            D[i, j] = sum(Fraction(a[i, k]) * Fraction(sa[k // 32, i]) * Fraction(b[j, k]) *
                          Fraction(sb[k // 32, j]) for k in range(K))
    return D


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_gemm_against_exact_rational_sums(fmt):
    g = np.random.default_rng(6)
    A = (g.standard_normal((3, 96)) * np.exp2(g.uniform(-4, 4, (3, 96)))).astype(np.float32)
    B = (g.standard_normal((5, 96)) * np.exp2(g.uniform(-4, 4, (5, 96)))).astype(np.float32)
    qa, sfa = oq.quantize_fp4_bs16(A, fmt)
    qb, sfb = oq.quantize_fp4_bs16(B, fmt)
    C = g.standard_normal((3, 5)).astype(np.float32)
    D, bnd = og.gemm_fp4_bs16(qa, sfa, qb, sfb, fmt, C=C)
    E = _exact_gemm(qa, sfa, qb, sfb, fmt)
    for i in range(3):
        for j in range(5):
            exact = E[i, j] + Fraction(float(C[i, j]))
            assert abs(Fraction(D[i, j]) - exact) <= Fraction(2.0 ** -50) * (abs(exact) + 1)
    # a transposed B (the classic layout mistake) is caught: N x K stored, used as K x N
    assert not np.allclose(og.gemm_fp4_bs16(qa, sfa, qb, sfb, fmt)[0],
                           og.gemm_fp4_bs16(qa, sfa, qb[::-1], sfb[:, ::-1], fmt)[0])


def test_gemm_closed_form_all_ones():
    K = 256
    qa = formats.pack_e2m1(np.full((2, K), 2, np.uint8))       # E2M1 code 2 = 1.0
    qb = formats.pack_e2m1(np.full((3, K), 2, np.uint8))
    sfa = np.full((K // 32, 2), 0x4000, np.uint16)             # BF16 2.0
    sfb = np.full((K // 32, 3), 0x3F40, np.uint16)             # BF16 0.75
    D, bnd = og.gemm_fp4_bs16(qa, sfa, qb, sfb, "bf16")
    assert (D == K * 2.0 * 0.75).all() and (bnd == D).all()
    E = og.gemm_fp4_bs16_bits(qa, sfa, qb, sfb, [0, 1], [2, 0], "bf16")
    assert (E == K * 1.5).all()


def test_block_promotion_rounds_in_fp32():
    # block 0: a = [4, 4], b = [2, 2] -> P0 = 16, s_A s_B = 2^10 * 2^10 -> acc = 2^24;
    # block 1: a = [1], b = [0.5], unit scales -> fma(1, 0.5, 2^24) = 2^24 + 0.5, which
    # FP32 rounds to 2^24 (the spacing there is 2).  The exact sum keeps the 0.5.
    ca = np.zeros((1, 64), np.uint8)
    cb = np.zeros((1, 64), np.uint8)
    ca[0, :2] = 6        # 4.0
    cb[0, :2] = 4        # 2.0
    ca[0, 32] = 2        # 1.0
    cb[0, 32] = 1        # 0.5
    qa, qb = formats.pack_e2m1(ca), formats.pack_e2m1(cb)
    sfa = np.array([[0x4480], [0x3F80]], np.uint16)            # BF16 2^10, 1.0
    sfb = np.array([[0x4480], [0x3F80]], np.uint16)
    D, _ = og.gemm_fp4_bs16(qa, sfa, qb, sfb, "bf16")
    assert D[0, 0] == 2.0 ** 24 + 0.5
    E = og.gemm_fp4_bs16_bits(qa, sfa, qb, sfb, [0], [0], "bf16")
    assert E[0] == 2.0 ** 24

"""Pins of the oracle's quantisers: hand-worked groups, closed forms, invariants."""
import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import formats, quantize

FACTS = {r[0]: r[1] for r in read_golden("format_facts.txt")}


def test_fp8_tile_hand_worked():
    # max_abs 896 -> s = 896/448 = 2 (exact); elements halve before the cast
    x = np.zeros((3, 5), np.float32)
    x[0, :3] = [896.0, 1.0, -3.0]
    q, s = quantize.quantize_fp8(x, "e4m3", "tile")
    assert s.shape == (1, 1) and s[0, 0] == 2.0
    # 448 -> 0x7E, 0.5 -> 0x30, -1.5 -> 0xBC
    assert list(q[0, :3]) == [0x7E, 0x30, 0xBC]
    assert (q[1:] == 0).all()


def test_fp8_zero_tile_scale_is_one():
    q, s = quantize.quantize_fp8(np.zeros((130, 7), np.float32), "e4m3", "tile")
    assert s.shape == (2, 1) and (s == 1.0).all() and (q == 0).all()


def test_fp8_scale_is_fp32_quotient():
    g = np.random.default_rng(3)
    x = (g.standard_normal((256, 384)) * 3).astype(np.float32)
    q, s = quantize.quantize_fp8(x, "e4m3", "tile")
    for ti in range(2):
        for tj in range(3):
            amax = np.abs(x[ti*128:(ti+1)*128, tj*128:(tj+1)*128]).max()
            # FP32 round-to-nearest of the exact quotient
            exact = float(amax) / 448.0
            assert s[ti, tj] == np.float32(exact) or \
                abs(float(s[ti, tj]) - exact) <= 0.5 * float(np.spacing(np.float32(exact)))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("gran", ["tile", "row"])
def test_fp8_invariants(fmt, gran):
    # every code is the nearest value to x/s; the max of each group maps to +-fmt_max
    g = np.random.default_rng(11)
    R, C = 200, 300          # ragged in both directions
    x = g.standard_normal((R, C)).astype(np.float32) * np.exp2(g.uniform(-6, 6, (R, 1))).astype(np.float32)
    q, s = quantize.quantize_fp8(x, fmt, gran)
    vals = formats.decode_array(q, fmt)
    if gran == "tile":
        assert s.shape == (2, 3)
        S = np.repeat(np.repeat(s, 128, 0), 128, 1)[:R, :C]
    else:
        assert s.shape == (3, R)
        S = np.repeat(s.T, 128, 1)[:, :C]
    y = x.astype(np.float64) / S.astype(np.float64)
    # nearest: no finite code value is closer to x/s than the chosen one
    ladder = np.array(sorted(v for v in formats.decode_table(fmt) if np.isfinite(v) and v >= 0))
    ay = np.minimum(np.abs(y), ladder[-1]).ravel()
    best = np.min(np.abs(ladder[None, :] - ay[:, None]), axis=1)
    assert np.all(np.abs(np.abs(vals).ravel() - ay) <= best * (1 + 1e-12))
    assert np.all(np.sign(vals) * np.sign(y) >= 0)
    fmax = formats.max_finite(fmt)
    assert np.isclose(np.abs(vals).max(), fmax)


def test_fp8_custom_fmt_max_for_e5m2():
    x = np.array([[896.0, -1.0]], np.float32)
    q, s = quantize.quantize_fp8(x, "e5m2", "row", fmt_max=448.0)
    assert s[0, 0] == 2.0
    assert formats.decode_e5m2(int(q[0, 0])) == 448.0


def test_e8m0_nearest_power_of_two():
    E = lambda v: quantize.e8m0_nearest_pow2(np.float32(v)) - 127
    assert E(1.0) == 0
    assert E(1.49) == 0 and E(1.5) == 1 and E(1.51) == 1     # tie goes up
    assert E(0.74) == -1 and E(0.75) == 0
    assert E(3.0) == 2 and E(2.99) == 1
    assert E(2.0 ** -130) == -127                            # clamped to code 0
    assert quantize.e8m0_nearest_pow2(np.float32(0.0)) == 127


def test_mxfp4_hand_worked():
    # a 32-block with max 6 -> v = 1 -> scale 2^0; max 9 -> v = 1.5 -> 2^1 (tie up);
    # max 8.9 -> v = 1.483 -> 2^0 and 8.9 saturates to 6; max 12 -> 2^1
    x = np.zeros((4, 32), np.float32)
    x[0, :4] = [6.0, 1.0, -0.5, 0.2]
    x[1, :2] = [9.0, -2.5]
    x[2, :2] = [8.9, 0.75]
    x[3, :2] = [-12.0, 5.0]
    packed, sf = quantize.quantize_mxfp4(x)
    assert list(sf[:, 0]) == [127, 128, 127, 128]
    codes = formats.unpack_e2m1(packed)
    vals = formats.decode_array(codes, "e2m1")
    assert list(vals[0, :4]) == [6.0, 1.0, -0.5, 0.0]        # 0.2 -> 0 (below 0.25)
    assert list(vals[1, :2]) == [4.0, -1.0]                  # 9/2 = 4.5 -> 4 (nearest), -1.25 -> -1 (tie to even)
    assert list(vals[2, :2]) == [6.0, 1.0]                   # 0.75 -> 1 (tie to even code 2)
    assert list(vals[3, :2]) == [-6.0, 2.0]                  # 5/2 = 2.5 -> 2 (tie to even)


def test_mxfp4_zero_block_and_sizes():
    K = 4096
    x = np.zeros((2, K), np.float32)
    x[1, 100] = 3.0
    packed, sf = quantize.quantize_mxfp4(x)
    assert sf.shape[1] == int(FACTS["mx_scale_bytes_per_row_k4096"])
    assert packed.shape[1] == int(FACTS["mx_data_bytes_per_row_k4096"])
    assert K // sf.shape[1] == int(FACTS["mx_block"])
    assert (sf[0] == 127).all() and (packed[0] == 0).all()


def test_mxfp4_reconstruction_bound():
    # every element is within half an E2M1 step (times the scale) of its source,
    # or clipped at 6 * scale; the block max never exceeds 9 * 2^E before clipping
    g = np.random.default_rng(5)
    x = (g.standard_normal((64, 256)) * np.exp2(g.uniform(-8, 8, (64, 1)))).astype(np.float32)
    packed, sf = quantize.quantize_mxfp4(x)
    vals = formats.decode_array(formats.unpack_e2m1(packed), "e2m1")
    scale = np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=1)
    y = x / scale
    assert np.all(np.abs(y).reshape(64, 8, 32).max(axis=2) <= 9.0)
    clipped = np.abs(y) > 6.0
    assert np.all(np.abs(vals[clipped]) == 6.0)
    step = np.where(np.abs(y) < 2, 0.5, np.where(np.abs(y) < 4, 1.0, 2.0))
    assert np.all(np.abs(vals - y)[~clipped] <= step[~clipped] / 2)


def test_tcgen05_layout_is_a_permutation():
    g = np.random.default_rng(1)
    sf = g.integers(0, 255, size=(130, 9), dtype=np.uint8)
    out = quantize.sf_to_tcgen05_layout(sf)
    assert out.size == 2 * 3 * 512
    # each source byte lands in exactly one place and the rest is padding (127)
    assert sorted(out.tolist()) == sorted(sf.ravel().tolist() + [127] * (out.size - sf.size))


def test_tcgen05_layout_hand_placed_bytes():
    # The tensor core's scale-factor atom (NVIDIA's PTX ISA, tcgen05 block
    # scaling; the same 128 x 4 tile as cuBLAS's block-scaling layout): 512
    # bytes per 128 rows x 4 K-blocks, stored as [32][4][4] = (row mod 32,
    # row / 32 within the 128, K-block mod 4); atoms ordered row block major.
    # Each expected offset below is worked out by hand from that description.
    R, KB = 256, 8                 # 2 row blocks x 2 atoms along K
    placed = {                     # (row, K-block): offset in bytes
        (0, 0): 0, (1, 0): 16, (31, 0): 496, (32, 0): 4, (96, 0): 12,
        (0, 1): 1, (0, 3): 3, (33, 2): 22, (127, 3): 511,
        (0, 4): 512, (5, 6): 594,          # second atom of row block 0
        (128, 0): 1024,                    # first atom of row block 1
        (200, 7): 1675,                    # 1536 + 8*16 + 2*4 + 3
    }
    sf = np.zeros((R, KB), np.uint8)
    for n, (r, c) in enumerate(placed):
        sf[r, c] = n + 1
    out = quantize.sf_to_tcgen05_layout(sf)
    assert out.size == 4 * 512
    for n, off in enumerate(placed.values()):
        assert out[off] == n + 1, (off, out[off])
    assert np.count_nonzero(out) == len(placed)


def test_mxfp8_hand_worked_e4m3():
    # E4M3 max 448.  Block max 448 -> v = 1 -> 2^0; 672 -> v = 1.5 -> tie -> 2^1;
    # 600 -> v = 1.34 -> 2^0 (600 saturates to 448); 0 -> code 127.
    x = np.zeros((4, 32), np.float32)
    x[0, :3] = [448.0, -1.0, 0.3]
    x[1, :3] = [672.0, -336.0, 2.0]
    x[2, :2] = [600.0, 17.0]
    codes, sf = quantize.quantize_mxfp8(x, "e4m3")
    assert list(sf[:, 0]) == [127, 128, 127, 127]
    vals = formats.decode_array(codes, "e4m3")
    assert list(vals[0, :3]) == [448.0, -1.0, 0.3125]        # 0.3 -> 0.3125 (1.25 * 2^-2)
    # after dividing by 2: 336 is half way between 320 and 352 and -168 half
    # way between -160 and -176; both go to the even mantissa
    assert list(vals[1, :3]) == [320.0, -160.0, 1.0]
    # 17 is half way between 16 and 18: even mantissa -> 16
    assert list(vals[2, :2]) == [448.0, 16.0]
    assert (vals[3] == 0).all()


def test_mxfp8_hand_worked_e5m2_and_fmt_max():
    # E5M2 max 57344: block max 57344 -> 2^0; 3 * 57344 / 2 = 86016 -> tie -> 2^1
    x = np.zeros((2, 32), np.float32)
    x[0, :2] = [57344.0, 3.0]
    x[1, :2] = [86016.0, -5.0]
    packed, sf = quantize.quantize_mxfp8(x, "e5m2")
    assert list(sf[:, 0]) == [127, 128]
    vals = formats.decode_array(packed, "e5m2")
    assert list(vals[0, :2]) == [57344.0, 3.0]
    assert list(vals[1, :2]) == [40960.0, -2.5]              # 43008 -> 40960 (tie to even), -2.5 exact
    # fmt_max = 448 for E5M2 maps the block maximum to 448 instead
    _, sf448 = quantize.quantize_mxfp8(x, "e5m2", fmt_max=448.0)
    assert list(sf448[:, 0]) == [127 + 7, 127 + 8]           # 57344 / 448 = 128 = 2^7; 86016/448 = 192 -> 2^8 (tie up)


def test_mxfp8_reconstruction_bound():
    # each element is within half an FP8 step (times the scale) of its source,
    # or clipped at fmt_max * scale; scaled block maxima stay below 1.5 * fmt_max
    g = np.random.default_rng(6)
    x = (g.standard_normal((64, 256)) * np.exp2(g.uniform(-12, 12, (64, 1)))).astype(np.float32)
    for fmt, mant in (("e4m3", 3), ("e5m2", 2)):
        codes, sf = quantize.quantize_mxfp8(x, fmt)
        fm = formats.max_finite(fmt)
        vals = formats.decode_array(codes, fmt)
        scale = np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=1)
        y = x.astype(np.float64) / scale
        assert np.all(np.abs(y).reshape(64, 8, 32).max(axis=2) <= 1.5 * fm)
        clipped = np.abs(y) > fm
        assert np.all(np.abs(vals[clipped]) == fm)
        # spacing of the format at |y| (normal range), never below the subnormal step
        emin = -6 if fmt == "e4m3" else -14
        e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** emin)))
        step = np.exp2(e - mant)
        assert np.all(np.abs(vals - y)[~clipped] <= step[~clipped] / 2)


def test_mxfp8_zero_block_and_sizes():
    K = 4096
    x = np.zeros((2, K), np.float32)
    x[1, 100] = 3.0
    codes, sf = quantize.quantize_mxfp8(x, "e4m3")
    assert codes.shape == (2, K) and sf.shape == (2, K // int(FACTS["mx_block"]))
    assert (sf[0] == 127).all() and (codes[0] == 0).all()


# ------------------------------------------------------------------ NVFP4
def _nv_block(vals):
    x = np.zeros((1, 16), np.float32)
    x[0, :len(vals)] = vals
    return x


def _nv_codes(packed):
    return formats.unpack_e2m1(packed)[0]


def test_nvfp4_hand_worked_unit_scale():
    # max 6 -> v = 1 -> E4M3 1.0 (0x38), s = 1: elements rounded directly,
    # ties to the even E2M1 code (1.25 -> 1, 5 -> 4, 0.25 -> 0, 0.75 -> 1)
    x = _nv_block([6, -3, 1.25, 5, 0.25, 0.75, -0.75, 2.5, 3.5])
    p, sf = quantize.quantize_nvfp4(x)
    assert sf[0, 0] == 0x38
    vals = formats.decode_array(_nv_codes(p), "e2m1")[:9]
    assert list(vals) == [6, -3, 1, 4, 0, 1, -1, 2, 4]


def test_nvfp4_scale_rounds_to_e4m3_and_elements_divide():
    # max 7: v = 7/6 = 1.1666..; the E4M3 neighbours are 1.125 and 1.25, so
    # the scale is 1.125 (0x39); 7 / 1.125 = 6.22 saturates to 6;
    # 2.8125 / 1.125 = 2.5 ties to 2 (even), 3.375 / 1.125 = 3
    x = _nv_block([7, 2.8125, -3.375])
    p, sf = quantize.quantize_nvfp4(x)
    assert sf[0, 0] == 0x39
    vals = formats.decode_array(_nv_codes(p), "e2m1")[:3]
    assert list(vals) == [6, 2, -3]


def test_nvfp4_scale_saturates_and_subnormal_scales():
    # max 6000: v = 1000 > 448 -> scale 448 (0x7E); 6000 / 448 saturates to 6
    p, sf = quantize.quantize_nvfp4(_nv_block([6000, 896]))
    assert sf[0, 0] == 0x7E
    assert list(formats.decode_array(_nv_codes(p), "e2m1")[:2]) == [6, 2]
    # max 0.006: v = 0.001 lies between E4M3 subnormals 0 and 2^-9 (nearer
    # 2^-9) -> code 0x01; 0.006 / 2^-9 = 3.07 -> 3
    p, sf = quantize.quantize_nvfp4(_nv_block([0.006]))
    assert sf[0, 0] == 0x01
    assert formats.decode_array(_nv_codes(p), "e2m1")[0] == 3


def test_nvfp4_zero_and_underflowing_blocks():
    x = np.zeros((2, 32), np.float32)
    x[1, 16:] = 1e-5              # v = 1.7e-6 rounds to E4M3 zero: s = 0
    x[1, 0] = 0.5
    p, sf = quantize.quantize_nvfp4(x)
    assert sf.shape == (2, 2) and p.shape == (2, 16)
    assert sf[0, 0] == 0 and sf[0, 1] == 0 and sf[1, 1] == 0
    codes = formats.unpack_e2m1(p)
    assert not codes[0].any() and not codes[1, 16:].any()
    assert formats.decode_array(codes[1, :1], "e2m1")[0] == 6   # 0.5 / (0.5/6 -> E4M3) = 6


def test_nvfp4_tensor_scale_is_a_power_of_two_shift():
    # with g = 2^-7 every block scale code equals the g = 1 code of x * 2^7,
    # and the element codes are identical (all steps scale exactly)
    g = np.random.default_rng(3)
    x = (g.standard_normal((16, 128)) * 0.02).astype(np.float32)
    p1, sf1 = quantize.quantize_nvfp4(x, tensor_scale=2.0 ** -7)
    p2, sf2 = quantize.quantize_nvfp4(x * np.float32(2.0 ** 7))
    assert np.array_equal(p1, p2) and np.array_equal(sf1, sf2)


def test_nvfp4_reconstruction_bound():
    g = np.random.default_rng(4)
    x = (g.standard_normal((64, 256)) * np.exp2(g.uniform(-4, 4, (64, 1)))).astype(np.float32)
    p, sf = quantize.quantize_nvfp4(x, tensor_scale=2.0 ** -3)
    vals = formats.decode_array(formats.unpack_e2m1(p), "e2m1").reshape(64, 16, 16)
    s = (formats.decode_array(sf, "e4m3") * 2.0 ** -3)[:, :, None]
    blocks = x.reshape(64, 16, 16).astype(np.float64)
    amax = np.max(np.abs(blocks), axis=2, keepdims=True)
    # E2M1 steps are at most 2 (4 -> 6): error <= s; a scale rounded down by
    # up to 1/16 can push the maximum past 6 s by at most amax / 16
    assert np.all(np.abs(blocks - vals * s) <= s + amax / 16 + 1e-30)


def test_tcgen05_layout_pad_byte():
    sf = np.arange(5 * 3, dtype=np.uint8).reshape(5, 3) + 1
    out = quantize.sf_to_tcgen05_layout(sf, pad=0)
    assert out.size == 512 and np.count_nonzero(out) == 15
    assert sorted(out[out != 0]) == sorted(sf.ravel())

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

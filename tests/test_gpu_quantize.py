"""Quantiser parity: codes and scales bit-exact against the CPU oracle."""
import numpy as np
import pytest

import synth
from helpers import device, special_f32_values, to_dev
from oracle import formats, quantize as oq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("gran", ["tile", "row"])
@pytest.mark.parametrize("shape", [(256, 256), (200, 300), (1, 16), (129, 4100)])
def test_fp8_quantize_bit_exact(fmt, gran, shape):
    import fp4_gemm_gb300 as bsg
    dev = device()
    g = np.random.default_rng(hash((fmt, gran, shape)) % 2**32)
    x = (g.standard_normal(shape) * np.exp2(g.uniform(-10, 10, (shape[0], 1)))).astype(np.float32)
    x[g.random(shape) < 0.001] *= 100
    q, s = bsg.bsg_quantize_fp8(to_dev(x, dev), fmt, gran)
    oq_, os_ = oq.quantize_fp8(x, fmt, gran)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(q.cpu().numpy(), oq_)


def test_fp8_quantize_bf16_source_and_fmt_max():
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    x, _ = synth.make("dgrad", m=130, n=1, k=640)
    xb = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    xt = to_dev(xb, dev).to(torch.bfloat16)
    for fmt, fm in (("e5m2", 0.0), ("e5m2", 448.0), ("e4m3", 0.0)):
        q, s = bsg.bsg_quantize_fp8(xt, fmt, "tile", fmt_max=fm)
        oq_, os_ = oq.quantize_fp8(xb, fmt, "tile", fmt_max=None if fm == 0 else fm)
        assert np.array_equal(s.cpu().numpy(), os_)
        assert np.array_equal(q.cpu().numpy(), oq_)


def test_fp8_strided_source():
    import fp4_gemm_gb300 as bsg
    dev = device()
    g = np.random.default_rng(3)
    big = g.standard_normal((64, 520)).astype(np.float32)
    xt = to_dev(big, dev)[:, 4:504]          # leading dimension 520, 500 columns
    q, s = bsg.bsg_quantize_fp8(xt, "e4m3", "row")
    oq_, os_ = oq.quantize_fp8(big[:, 4:504], "e4m3", "row")
    assert np.array_equal(s.cpu().numpy(), os_) and np.array_equal(q.cpu().numpy(), oq_)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_cast_every_rounding_class(fmt):
    # one row per 127 test values plus the format max, so every row's scale is 1.0
    import fp4_gemm_gb300 as bsg
    dev = device()
    fmax = formats.max_finite(fmt)
    v = special_f32_values()
    v = v[np.isfinite(v)]
    rows = -(-v.size // 127)
    x = np.zeros((rows, 128), np.float32)
    x[:, 0] = fmax
    flat = np.zeros(rows * 127, np.float32)
    flat[: v.size] = v
    x[:, 1:] = flat.reshape(rows, 127)
    # values above the format max would change the scale: saturate them by hand
    x[:, 1:] = np.clip(x[:, 1:], -fmax, fmax)
    q, s = bsg.bsg_quantize_fp8(to_dev(x, dev), fmt, "row")
    assert (s.cpu().numpy() == 1.0).all()
    assert np.array_equal(q.cpu().numpy(), formats.encode(x, fmt))


def test_e2m1_cast_every_rounding_class():
    import fp4_gemm_gb300 as bsg
    dev = device()
    v = special_f32_values()
    v = np.clip(v[np.isfinite(v)], -6.0, 6.0)
    rows = -(-v.size // 31)
    x = np.zeros((rows, 32), np.float32)
    x[:, 0] = 6.0
    flat = np.zeros(rows * 31, np.float32)
    flat[: v.size] = v
    x[:, 1:] = flat.reshape(rows, 31)
    q, sf = bsg.bsg_quantize_mxfp4(to_dev(x, dev), "rowmajor")
    assert (sf.cpu().numpy() == 127).all()
    assert np.array_equal(q.cpu().numpy(), formats.pack_e2m1(formats.encode(x, "e2m1")))


@pytest.mark.parametrize("shape", [(1024, 1024), (130, 96), (1, 32), (16, 8192)])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_mxfp4_quantize_bit_exact(shape, src):
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    g = np.random.default_rng(shape[0] * 7 + shape[1])
    x = (g.standard_normal(shape) * np.exp2(g.uniform(-8, 8, (shape[0], 1)))).astype(np.float32)
    x[0, :32] = 0.0                              # an all-zero block
    if src == "bf16":
        x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    xt = to_dev(x, dev)
    if src == "bf16":
        xt = xt.to(torch.bfloat16)
    op, osf = oq.quantize_mxfp4(x)
    q, sf = bsg.bsg_quantize_mxfp4(xt, "rowmajor")
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(q.cpu().numpy(), op)
    q2, sf2 = bsg.bsg_quantize_mxfp4(xt, "tcgen05")
    assert np.array_equal(q2.cpu().numpy(), op)
    assert np.array_equal(sf2.cpu().numpy(), oq.sf_to_tcgen05_layout(osf))
    sf3 = bsg.bsg_sf_to_tcgen05(sf)
    assert np.array_equal(sf3.cpu().numpy(), oq.sf_to_tcgen05_layout(osf))


def test_e8m0_rounding_boundaries():
    # block maxima that put v = max/6 exactly on, just below and just above 1.5 * 2^e
    import fp4_gemm_gb300 as bsg
    dev = device()
    vs = []
    for e in range(-20, 20):
        mid = np.float32(1.5 * 2.0 ** e)
        vs += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf)),
               np.float32(2.0 ** e)]
    vs += [np.float32(2.0 ** -140), np.float32(1e-45), np.float32(3e38)]
    maxima = np.array(vs, np.float32) * np.float32(6.0)
    maxima = maxima[np.isfinite(maxima)]
    x = np.zeros((maxima.size, 32), np.float32)
    x[:, 3] = -maxima
    x[:, 7] = maxima / np.float32(3.0)
    op, osf = oq.quantize_mxfp4(x)
    q, sf = bsg.bsg_quantize_mxfp4(to_dev(x, dev), "rowmajor")
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(q.cpu().numpy(), op)


def _division_stress(fmt, gran, seed):
    """Groups whose amax spans the FP32 range, filled with values whose
    quotient by the group scale lies next to an FP8 rounding midpoint, so a
    quotient off by one FP32 ulp would change the code."""
    g = np.random.default_rng(seed)
    fm = oq.fmt_max_default(fmt)
    table = np.unique(np.abs(formats.decode_table(fmt)[np.isfinite(formats.decode_table(fmt))]))
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    exps = [-126, -110, -95, -88, -81, -80, -79, -60, -20, -1, 0, 1, 20, 60, 79, 80, 81, 100, 120, 127]
    amaxes = [np.float32(np.ldexp(1.0 + g.random(), e)) if e < 127 else np.float32(3.0e38) for e in exps]
    groups = len(amaxes)
    if gran == "tile":
        x = np.zeros((128, 128 * groups), np.float32)
        views = [np.zeros(128 * 128, np.float32) for _ in range(groups)]
    else:
        x = np.zeros((groups, 128 * 3), np.float32)
        views = [x[i, 128 * (i % 3):128 * (i % 3 + 1)] for i in range(groups)]
    for v, amax in zip(views, amaxes):
        s = oq.fp8_scale(amax, fm)
        n = v.size
        m = mids[g.integers(0, mids.size, n)] * np.where(g.random(n) < 0.5, -1, 1).astype(np.float32)
        with np.errstate(over="ignore", under="ignore"):
            vals = (m * s).astype(np.float32)
            step = g.integers(-2, 3, n)
            vals = np.where(step > 0, np.nextafter(vals, np.float32(np.inf)), vals)
            vals = np.where(step < 0, np.nextafter(vals, np.float32(-np.inf)), vals).astype(np.float32)
        vals = np.clip(vals, -amax, amax)
        vals[: 4] = [amax, -0.0, 0.0, np.float32(1e-45)]
        vals[4: 8] = -np.float32(np.ldexp(1.0, -140)), np.float32(np.ldexp(1.0, -126)), -amax, amax / 3
        v[:] = vals
    if gran == "tile":
        for i, v in enumerate(views):
            x[:, 128 * i:128 * (i + 1)] = v.reshape(128, 128)
    return x


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("gran", ["tile", "row"])
def test_fp8_division_next_to_rounding_midpoints(fmt, gran):
    # Every element is divided by its group's scale in FP32 and then rounded
    # to FP8; these inputs put the FP32 quotient next to FP8 midpoints over
    # scales from 2^-126 to 2^127, including signed zeros and subnormals.
    import fp4_gemm_gb300 as bsg
    dev = device()
    x = _division_stress(fmt, gran, 11 if gran == "tile" else 12)
    q, s = bsg.bsg_quantize_fp8(to_dev(x, dev), fmt, gran)
    oq_, os_ = oq.quantize_fp8(x, fmt, gran)
    assert np.array_equal(s.cpu().numpy(), os_)
    got = q.cpu().numpy()
    bad = np.argwhere(got != oq_)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"

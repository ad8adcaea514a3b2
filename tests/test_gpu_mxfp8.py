"""MXFP8 parity: the MX quantiser with FP8 elements bit-exact against the
oracle, and the block-scaled FP8 GEMM within the stated tolerance:
|D - D_ref| <= 1e-4 * sum_k |s_A a_k s_B b_k| + 1e-6 (BF16 output: + 8e-3 |D_ref|)."""
import numpy as np
import pytest

import synth
from helpers import device, report, special_f32_values, to_dev
from oracle import formats
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(256, 256), (130, 96), (1, 32), (200, 4128)])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_mxfp8_quantize_bit_exact(fmt, shape, src):
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    g = np.random.default_rng(shape[0] * 11 + shape[1] + (fmt == "e5m2"))
    x = (g.standard_normal(shape) * np.exp2(g.uniform(-12, 12, (shape[0], 1)))).astype(np.float32)
    x[g.random(shape) < 0.002] *= 60
    x[0, :32] = 0.0                              # an all-zero block
    if src == "bf16":
        x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    xt = to_dev(x, dev)
    if src == "bf16":
        xt = xt.to(torch.bfloat16)
    oc, osf = oq.quantize_mxfp8(x, fmt)
    q, sf = bsg.bsg_quantize_mx(xt, fmt, "rowmajor")
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(q.cpu().numpy(), oc)
    q2, sf2 = bsg.bsg_quantize_mx(xt, fmt, "tcgen05")
    assert np.array_equal(q2.cpu().numpy(), oc)
    assert np.array_equal(sf2.cpu().numpy(), oq.sf_to_tcgen05_layout(osf))


def test_mxfp8_quantize_custom_fmt_max():
    import fp4_gemm_gb300 as bsg
    dev = device()
    x, _ = synth.make("dgrad", m=64, n=1, k=512)
    for fmt, fm in (("e5m2", 448.0), ("e4m3", 240.0)):
        oc, osf = oq.quantize_mxfp8(x, fmt, fmt_max=fm)
        q, sf = bsg.bsg_quantize_mx(to_dev(x, dev), fmt, "rowmajor", fmt_max=fm)
        assert np.array_equal(sf.cpu().numpy(), osf) and np.array_equal(q.cpu().numpy(), oc)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mxfp8_cast_every_rounding_class(fmt):
    # every 32-block starts with the format maximum, so its scale is 2^0 and
    # the other 31 values go through the cast unscaled
    import fp4_gemm_gb300 as bsg
    dev = device()
    fmax = formats.max_finite(fmt)
    v = special_f32_values()
    v = v[np.isfinite(v) & (np.abs(v) <= fmax)]
    nblk = -(-v.size // 31)
    nblk += (-nblk) % 8                          # whole rows of 8 blocks
    body = np.zeros(nblk * 31, np.float32)
    body[:v.size] = v
    blocks = np.zeros((nblk, 32), np.float32)
    blocks[:, 0] = fmax
    blocks[:, 1:] = body.reshape(nblk, 31)
    x = blocks.reshape(-1, 256)
    q, sf = bsg.bsg_quantize_mx(to_dev(x, dev), fmt, "rowmajor")
    assert (sf.cpu().numpy() == 127).all()
    oc, osf = oq.quantize_mxfp8(x, fmt)
    assert (osf == 127).all()
    assert np.array_equal(q.cpu().numpy(), oc)


def _run(A, B, fa, fb, out, C=None, rows=None):
    import fp4_gemm_gb300 as bsg
    dev = device()
    qa, sfa = bsg.bsg_quantize_mx(to_dev(A, dev), fa, "tcgen05")
    qb, sfb = bsg.bsg_quantize_mx(to_dev(B, dev), fb, "tcgen05")
    Ct = None if C is None else to_dev(C, dev)
    D = bsg.bsg_gemm(qa, fa, sfa, "mx", qb, fb, sfb, "mx", C=Ct, out=out)
    assert bsg.bsg_device_error() == 0
    oca, osa = oq.quantize_mxfp8(A, fa)
    ocb, osb = oq.quantize_mxfp8(B, fb)
    assert np.array_equal(qa.cpu().numpy(), oca) and np.array_equal(qb.cpu().numpy(), ocb)
    Dref, bnd = og.gemm_mxfp8(oca, fa, osa, ocb, fb, osb, C=C, rows=rows)
    Dg = D.float().cpu().numpy()
    if rows is not None:
        Dg = Dg[rows]
    return og.within_tolerance(Dg, Dref, bnd, bf16=out == "bf16")


def test_mxfp8_256_cube():
    A, B = synth.make("fp8_256")
    report("mxfp8 256", *_run(A, B, "e4m3", "e4m3", "f32"))


@pytest.mark.parametrize("M,N,K", [(200, 300, 288), (1, 256, 128), (129, 257, 32), (384, 520, 1056),
                                   (130, 128, 96)])
@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_mxfp8_ragged(M, N, K, fa, fb):
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    report(f"mxfp8 {M}x{N}x{K} {fa}x{fb}", *_run(A, B, fa, fb, "f32"))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_mxfp8_with_addend(out):
    A, B = synth.make("ffn_up", m=512, n=768, k=1024)
    C = synth.addend("ffn_up", 512, 768)
    report(f"mxfp8 + C {out}", *_run(A, B, "e4m3", "e4m3", out, C=C))


@pytest.mark.parametrize("N,out", [(1001, "bf16"), (1002, "f32")])
def test_mxfp8_output_pitch_not_16_bytes(N, out):
    A, B = synth.make("ffn_up", m=300, n=N, k=256)
    report(f"mxfp8 pitch N={N}", *_run(A, B, "e4m3", "e4m3", out))


def test_mxfp8_many_tiles_persistent():
    # more 128 x 256 tiles than SMs: every CTA walks several tiles, and the
    # accumulator is handed between MMA and epilogue many times
    A, B = synth.make("ffn_up", m=2048, n=4096, k=512)
    rows = np.r_[0:3, 127:130, 1000:1003, 2045:2048]
    report("mxfp8 persistent", *_run(A, B, "e4m3", "e4m3", "bf16", rows=rows))


def test_mxfp8_long_k_e5m2():
    A, B = synth.make("dgrad", m=256, n=512, k=4096)
    report("mxfp8 long K", *_run(A, B, "e5m2", "e4m3", "f32"))

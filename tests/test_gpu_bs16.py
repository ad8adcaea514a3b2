"""FP4 with BF16 / FP16 block scales ("Rubin FP4 GEMM deep dive", §3.2):
the quantiser bit-exact against the oracle, and the block-promoted GEMM bit
for bit against the oracle's step-by-step emulation (every partial and every
scale product is exact, so only the per-block FMAs round) and within the
stated tolerance |D - D_ref| <= 1e-4 * sum_k |s_A a_k s_B b_k| + 1e-6 of the
exact FP64 GEMM (BF16 output: + 8e-3 |D_ref|)."""
import numpy as np
import pytest

import synth
from helpers import device, report, special_f32_values, to_dev
from oracle import formats
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _q(x, scale, src="f32"):
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    xt = to_dev(x, dev)
    if src == "bf16":
        xt = xt.to(torch.bfloat16)
    q, sf = bsg.bsg_quantize_fp4_bs16(xt, scale)
    assert bsg.bsg_device_error() == 0
    return q, sf


def _sf_host(sf):
    return sf.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("scale", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(256, 256), (130, 96), (1, 32), (200, 4128), (37, 288)])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantiser_bit_exact(scale, shape, src):
    g = np.random.default_rng(shape[0] * 7 + shape[1] + (scale == "f16"))
    x = (g.standard_normal(shape) * np.exp2(g.uniform(-14, 14, (shape[0], 1)))).astype(np.float32)
    x[g.random(shape) < 0.002] *= 60
    x[0, :32] = 0.0                              # an all-zero block
    if src == "bf16":
        x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    q, sf = _q(x, scale, src)
    oc, osf = oq.quantize_fp4_bs16(x, scale)
    assert np.array_equal(_sf_host(sf), osf)
    assert np.array_equal(q.cpu().numpy(), oc)


@pytest.mark.parametrize("scale", ["bf16", "f16"])
def test_quantiser_every_rounding_class_at_unit_scale(scale):
    # every block starts with 6.0, so v = 1 and s = 1 exactly: the other 31
    # values go through the E2M1 cast unscaled (ties, saturation, signs)
    v = special_f32_values()
    v = v[np.isfinite(v) & (np.abs(v) <= 6.0)]
    nblk = -(-v.size // 31)
    nblk += (-nblk) % 8
    body = np.zeros(nblk * 31, np.float32)
    body[:v.size] = v
    blocks = np.zeros((nblk, 32), np.float32)
    blocks[:, 0] = 6.0
    blocks[:, 1:] = body.reshape(nblk, 31)
    x = blocks.reshape(-1, 256)
    q, sf = _q(x, scale)
    one = 0x3F80 if scale == "bf16" else 0x3C00
    assert (_sf_host(sf) == one).all()
    oc, osf = oq.quantize_fp4_bs16(x, scale)
    assert np.array_equal(q.cpu().numpy(), oc)


def test_quantiser_fp16_saturation_and_underflow():
    x = np.zeros((4, 128), np.float32)
    x[0, :32] = 420000.0 * np.linspace(-1, 1, 32)       # v = 70000 > 65504
    x[1, 32:64] = 1e-9                                  # v below FP16's smallest subnormal
    x[2, 64:96] = 3e-6 * np.linspace(-1, 1, 32)         # an FP16 subnormal scale
    x[3, 96:] = 65504.0 * 6                             # exactly the largest FP16 scale
    for scale in ("f16", "bf16"):
        q, sf = _q(x, scale)
        oc, osf = oq.quantize_fp4_bs16(x, scale)
        assert np.array_equal(_sf_host(sf), osf) and np.array_equal(q.cpu().numpy(), oc)


def _gemm(A, B, scale, out, C=None):
    import fp4_gemm_gb300 as bsg
    dev = device()
    qa, sfa = _q(A, scale)
    qb, sfb = _q(B, scale)
    Ct = None if C is None else to_dev(C, dev)
    D = bsg.bsg_gemm(qa, "e2m1", sfa, scale, qb, "e2m1", sfb, scale, C=Ct, out=out, K=A.shape[1])
    assert bsg.bsg_device_error() == 0
    oqa, osa = oq.quantize_fp4_bs16(A, scale)
    oqb, osb = oq.quantize_fp4_bs16(B, scale)
    assert np.array_equal(qa.cpu().numpy(), oqa) and np.array_equal(qb.cpu().numpy(), oqb)
    assert np.array_equal(_sf_host(sfa), osa) and np.array_equal(_sf_host(sfb), osb)
    return D.float().cpu().numpy().astype(np.float64), (oqa, osa, oqb, osb)


@pytest.mark.parametrize("M,N,K", [(200, 300, 256), (1, 256, 128), (129, 257, 384), (384, 520, 1024),
                                   (256, 512, 4096)])
@pytest.mark.parametrize("scale", ["bf16", "f16"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_bit_exact_and_within_tolerance(M, N, K, scale, out):
    A, B = synth.make("mxfp4_1024", m=M, n=N, k=K)
    C = synth.addend("mxfp4_1024", M, N) if out == "f32" else None
    D, (oqa, osa, oqb, osb) = _gemm(A, B, scale, out, C)
    Dref, bnd = og.gemm_fp4_bs16(oqa, osa, oqb, osb, scale, C=C)
    report(f"bs16 {M}x{N}x{K} {scale} {out}", *og.within_tolerance(D, Dref, bnd, bf16=out == "bf16"))
    i, j = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    if M * N > 40000:                            # bit-exact on a sample of large shapes
        g = np.random.default_rng(M + N + K)
        pick = g.choice(M * N, 40000, replace=False)
        i, j = i.ravel()[pick], j.ravel()[pick]
    E = og.gemm_fp4_bs16_bits(oqa, osa, oqb, osb, i.ravel(), j.ravel(), scale, C=C, out=out)
    assert np.array_equal(D[i.ravel(), j.ravel()], E)


def test_gemm_many_tiles_persistent():
    # more 128 x 256 tiles than SMs: every CTA walks several tiles
    M, N, K = 2048, 4096, 512
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    D, (oqa, osa, oqb, osb) = _gemm(A, B, "bf16", "bf16")
    rows = np.r_[0:3, 127:130, 1000:1003, 2045:2048]
    Dref, bnd = og.gemm_fp4_bs16(oqa, osa, oqb, osb, "bf16", rows=rows)
    report("bs16 persistent", *og.within_tolerance(D[rows], Dref, bnd, bf16=True))
    i, j = np.meshgrid(rows, np.arange(0, N, 7), indexing="ij")
    E = og.gemm_fp4_bs16_bits(oqa, osa, oqb, osb, i.ravel(), j.ravel(), "bf16", out="bf16")
    assert np.array_equal(D[i.ravel(), j.ravel()], E)


def test_gemm_ffn_up_full_size_sampled():
    # The FFN-up shape (M=8192, K=4096, N=14336) with BF16 block scales and BF16
    # output, launched as the benchmark launches it; each row of an operand is
    # quantised on its own, so the oracle quantises the sampled rows only.
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    _, M, N, K = synth.WORKLOADS["ffn_up"]
    A, B = synth.make("ffn_up")
    qa, sfa = bsg.bsg_quantize_fp4_bs16(to_dev(A, dev), "bf16")
    qb, sfb = bsg.bsg_quantize_fp4_bs16(to_dev(B, dev), "bf16")
    D = bsg.bsg_gemm(qa, "e2m1", sfa, "bf16", qb, "e2m1", sfb, "bf16", out="bf16", K=K)
    assert bsg.bsg_device_error() == 0
    g = np.random.default_rng(8192)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], g.integers(0, M, 28)]))
    cols = np.unique(np.concatenate([[0, 255, 256, N - 1], g.integers(0, N, 60)]))
    oqa, osa = oq.quantize_fp4_bs16(A[rows], "bf16")
    oqb, osb = oq.quantize_fp4_bs16(B[cols], "bf16")
    rt, ct = torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)
    assert np.array_equal(qa.index_select(0, rt).cpu().numpy(), oqa)
    assert np.array_equal(sfa.index_select(1, rt).cpu().numpy().view(np.uint16), osa)
    assert np.array_equal(qb.index_select(0, ct).cpu().numpy(), oqb)
    Dg = D.index_select(0, rt).index_select(1, ct).float().cpu().numpy().astype(np.float64)
    Dref, bnd = og.gemm_fp4_bs16(oqa, osa, oqb, osb, "bf16")
    report("bs16 ffn_up full size", *og.within_tolerance(Dg, Dref, bnd, bf16=True))
    i, j = np.meshgrid(np.arange(len(rows)), np.arange(len(cols)), indexing="ij")
    E = og.gemm_fp4_bs16_bits(oqa, osa, oqb, osb, i.ravel(), j.ravel(), "bf16", out="bf16")
    assert np.array_equal(Dg, E.reshape(len(rows), len(cols)))

"""MXFP4 GEMM parity (general and decode-shaped) against the oracle."""
import numpy as np
import pytest

import synth
from helpers import device, report, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _run(A, B, out, C=None, a_bf16=False, rows=None):
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    if a_bf16:
        A = synth.bf16_bits_to_f32(synth.to_bf16_bits(A))
    At = to_dev(A, dev)
    if a_bf16:
        At = At.to(torch.bfloat16)
    pa, fa = bsg.bsg_quantize_mxfp4(At, "tcgen05")
    pb, fb = bsg.bsg_quantize_mxfp4(to_dev(B, dev), "tcgen05")
    Ct = None if C is None else to_dev(C, dev)
    D = bsg.bsg_gemm(pa, "e2m1", fa, "mx", pb, "e2m1", fb, "mx", C=Ct, out=out)
    assert bsg.bsg_device_error() == 0
    opa, ofa = oq.quantize_mxfp4(A)
    opb, ofb = oq.quantize_mxfp4(B)
    assert np.array_equal(pa.cpu().numpy(), opa) and np.array_equal(pb.cpu().numpy(), opb)
    Dref, bnd = og.gemm_mxfp4(opa, ofa, opb, ofb, C=C, rows=rows)
    Dg = D.float().cpu().numpy()
    if rows is not None:
        Dg = Dg[rows]
    return og.within_tolerance(Dg, Dref, bnd, bf16=out == "bf16")


def test_mxfp4_1024_config():
    A, B = synth.make("mxfp4_1024")
    report("mxfp4_1024", *_run(A, B, "f32"))


@pytest.mark.parametrize("M,N,K", [(130, 200, 96), (64, 128, 32), (300, 260, 800)])
def test_mxfp4_ragged(M, N, K):
    A, B = synth.make("mxfp4_1024", m=M, n=N, k=K)
    report(f"mxfp4 {M}x{N}x{K}", *_run(A, B, "f32"))


def test_mxfp4_bf16_with_addend():
    A, B = synth.make("mxfp4_1024", m=256, n=384, k=512)
    C = synth.addend("mxfp4_1024", 256, 384)
    report("mxfp4 bf16+C", *_run(A, B, "bf16", C=C))


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32])
@pytest.mark.parametrize("N,K", [(1000, 1024), (4096, 8192), (384, 96), (2048, 2304), (1536, 768)])
def test_decode_path(M, N, K):
    A, B = synth.make("decode", m=M, n=N, k=K)
    report(f"decode M={M} N={N} K={K}", *_run(A, B, "bf16", a_bf16=True))


def test_decode_with_addend_fp32_twice():
    # the workspace is left zeroed: a second call reuses it and matches again
    A, B = synth.make("decode", m=16, n=2048, k=4096)
    C = synth.addend("decode", 16, 2048)
    report("decode + C (1)", *_run(A, B, "f32", C=C, a_bf16=True))
    report("decode + C (2)", *_run(A, B, "f32", C=C, a_bf16=True))


@pytest.mark.parametrize("M", [1, 16, 32])
def test_decode_full_size_sampled_columns(M):
    # The decode benchmark shape (N=28672, K=8192), launched exactly as the
    # benchmark launches it; the oracle checks a sample of output columns
    # (weight rows) that covers tile edges and split-K segment boundaries.
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    N, K = 28672, 8192
    A, B = synth.make("decode", m=M, n=N, k=K)
    A = synth.bf16_bits_to_f32(synth.to_bf16_bits(A))
    pa, fa = bsg.bsg_quantize_mxfp4(to_dev(A, dev).to(torch.bfloat16), "tcgen05")
    pb, fb = bsg.bsg_quantize_mxfp4(to_dev(B, dev), "tcgen05")
    D = bsg.bsg_gemm(pa, "e2m1", fa, "mx", pb, "e2m1", fb, "mx", out="bf16")
    assert bsg.bsg_device_error() == 0
    rng = np.random.default_rng(7)
    cols = np.unique(np.concatenate([np.arange(0, 4), np.arange(124, 132), np.arange(N - 4, N),
                                     np.arange(128, N, 128 * 37), rng.integers(0, N, 256)]))
    opa, ofa = oq.quantize_mxfp4(A)
    opb, ofb = oq.quantize_mxfp4(B[cols])
    assert np.array_equal(pa.cpu().numpy(), opa)
    assert np.array_equal(pb.cpu().numpy()[cols], opb)
    Dref, bnd = og.gemm_mxfp4(opa, ofa, opb, ofb)
    Dg = D.float().cpu().numpy()[:, cols]
    report(f"decode full size M={M} ({cols.size} columns)", *og.within_tolerance(Dg, Dref, bnd, bf16=True))


# Shapes with at least half as many 128 x 256 tiles as SMs take the large
# block-scaled kernel: ragged M and N, an N whose last tile holds one 128-row
# scale block (1900), K tails that leave a partial stage and a partial atom.
@pytest.mark.parametrize("M,N,K,out,addend", [(2000, 2000, 288, "f32", False),
                                              (1300, 1900, 1056, "bf16", True)])
def test_mxfp4_large_kernel_ragged(M, N, K, out, addend):
    A, B = synth.make("mxfp4_1024", m=M, n=N, k=K)
    C = synth.addend("mxfp4_1024", M, N) if addend else None
    rows = np.unique(np.concatenate([np.arange(0, M, 7), [M - 1]]))
    report(f"mxfp4 large {M}x{N}x{K}", *_run(A, B, out, C=C, rows=rows))


def test_mxfp4_large_kernel_ffn_up_shape_sampled():
    import fp4_gemm_gb300 as bsg
    dev = device()
    _, M, N, K = synth.WORKLOADS["ffn_up"]
    A, B = synth.make("ffn_up")
    pa, fa = bsg.bsg_quantize_mxfp4(to_dev(A, dev), "tcgen05")
    pb, fb = bsg.bsg_quantize_mxfp4(to_dev(B, dev), "tcgen05")
    D = bsg.bsg_gemm(pa, "e2m1", fa, "mx", pb, "e2m1", fb, "mx", out="bf16")
    assert bsg.bsg_device_error() == 0
    g = np.random.default_rng(13)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], g.integers(0, M, 28)]))
    cols = np.unique(np.concatenate([[0, 255, 256, N - 1], g.integers(0, N, 60)]))
    opa, ofa = oq.quantize_mxfp4(A[rows])      # MX scales are per row: rows quantise alone
    opb, ofb = oq.quantize_mxfp4(B[cols])
    Dref, bnd = og.gemm_mxfp4(opa, ofa, opb, ofb)
    report("mxfp4 ffn_up sampled", *og.within_tolerance(D.float().cpu().numpy()[np.ix_(rows, cols)],
                                                        Dref, bnd, bf16=True))


# ---- activations quantised on the fly (bsg_gemm_mxfp4_act): the result must
# be bit for bit that of bsg_quantize_mxfp4 followed by bsg_gemm, whose
# parity with the oracle the tests above establish; one case also goes to the
# oracle directly.

def _fused_and_separate(A, B, out, C=None, src="bf16", pad=0):
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    M, K = A.shape
    xt = to_dev(A, dev)
    if src == "bf16":
        xt = xt.to(torch.bfloat16)
    if pad:   # rows padded in memory: the activations are a strided view
        buf = torch.zeros((M, K + pad), dtype=xt.dtype, device=dev)
        buf[:, :K] = xt
        xt = buf[:, :K]
    pb, fb = bsg.bsg_quantize_mxfp4(to_dev(B, dev), "tcgen05")
    Ct = None if C is None else to_dev(C, dev)
    Df = bsg.bsg_gemm_mxfp4_act(xt, pb, fb, C=Ct, out=out)
    assert bsg.bsg_device_error() == 0
    pa, fa = bsg.bsg_quantize_mxfp4(xt.contiguous(), "tcgen05")
    Ds = bsg.bsg_gemm(pa, "e2m1", fa, "mx", pb, "e2m1", fb, "mx", C=Ct, out=out)
    assert bsg.bsg_device_error() == 0
    return Df.float().cpu().numpy(), Ds.float().cpu().numpy()


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32, 64])
@pytest.mark.parametrize("N,K", [(1000, 1024), (4096, 8192), (384, 96), (2048, 2304)])
@pytest.mark.parametrize("src", ["bf16", "f32"])
def test_act_quantised_on_the_fly_equals_separate(M, N, K, src):
    A, B = synth.make("decode", m=M, n=N, k=K)
    Df, Ds = _fused_and_separate(A, B, "bf16", src=src)
    assert np.array_equal(Df, Ds)


@pytest.mark.parametrize("M", [1, 16])
def test_act_quantised_on_the_fly_strided_rows_addend_repeated(M):
    # padded rows (scalar loads), an FP32 addend and FP32 output; three calls
    # in a row reuse the workspace (its counters must come back to zero)
    A, B = synth.make("decode", m=M, n=2048, k=4096)
    C = synth.addend("decode", M, 2048)
    first = None
    for _ in range(3):
        Df, Ds = _fused_and_separate(A, B, "f32", C=C, src="bf16", pad=8)
        assert np.array_equal(Df, Ds)
        if first is None:
            first = Df
        assert np.array_equal(Df, first)


def test_act_quantised_on_the_fly_full_decode_shape_against_oracle():
    # the decode benchmark shape (M=16, K=8192, N=28672), BF16 activations:
    # all outputs equal the two-call path, sampled columns are within the
    # oracle's tolerance
    N, K, M = 28672, 8192, 16
    A, B = synth.make("decode", m=M, n=N, k=K)
    A = synth.bf16_bits_to_f32(synth.to_bf16_bits(A))
    Df, Ds = _fused_and_separate(A, B, "bf16", src="bf16")
    assert np.array_equal(Df, Ds)
    rng = np.random.default_rng(11)
    cols = np.unique(np.concatenate([np.arange(0, 4), np.arange(124, 132), np.arange(N - 4, N),
                                     rng.integers(0, N, 128)]))
    opa, ofa = oq.quantize_mxfp4(A)
    opb, ofb = oq.quantize_mxfp4(B[cols])
    Dref, bnd = og.gemm_mxfp4(opa, ofa, opb, ofb)
    report("fused decode full size", *og.within_tolerance(Df[:, cols], Dref, bnd, bf16=True))

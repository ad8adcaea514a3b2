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
@pytest.mark.parametrize("N,K", [(1000, 1024), (4096, 8192), (384, 96)])
def test_decode_path(M, N, K):
    A, B = synth.make("decode", m=M, n=N, k=K)
    report(f"decode M={M} N={N} K={K}", *_run(A, B, "bf16", a_bf16=True))


def test_decode_with_addend_fp32_twice():
    # the workspace is left zeroed: a second call reuses it and matches again
    A, B = synth.make("decode", m=16, n=2048, k=4096)
    C = synth.addend("decode", 16, 2048)
    report("decode + C (1)", *_run(A, B, "f32", C=C, a_bf16=True))
    report("decode + C (2)", *_run(A, B, "f32", C=C, a_bf16=True))

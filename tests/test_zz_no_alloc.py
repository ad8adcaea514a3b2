"""The allocation-free decode entry point, called through the C ABI.

Callers that cannot allocate device memory (a plug-in handed only its input
and output buffers, a decode loop that must keep cudaMalloc out of its steady
state) use bsg_gemm_decode_noalloc, which runs the decode-shaped MXFP4 GEMM on
scratch compiled into the library.  Its results must match bsg_gemm's (the
caller-workspace entry point) within the tolerance of the other GEMM tests,
and the oracle's, on two calls in a row: the second call reuses the scratch
the first one left.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import synth
from helpers import device, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _inputs(M, N, K):
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    X, W = synth.make("decode", m=M, n=N, k=K)
    X = synth.bf16_bits_to_f32(synth.to_bf16_bits(X))
    px, fx = bsg.bsg_quantize_mxfp4(to_dev(X, dev).to(torch.bfloat16), "tcgen05")
    pw, fw = bsg.bsg_quantize_mxfp4(to_dev(W, dev), "tcgen05")
    opx, ofx = oq.quantize_mxfp4(X)
    opw, ofw = oq.quantize_mxfp4(W)
    # the oracle's result is only the oracle's if both sides hold the same operands
    assert np.array_equal(px.cpu().numpy(), opx) and np.array_equal(pw.cpu().numpy(), opw)
    assert np.array_equal(fx.cpu().numpy(), oq.sf_to_tcgen05_layout(ofx))
    assert np.array_equal(fw.cpu().numpy(), oq.sf_to_tcgen05_layout(ofw))
    Dref, bnd = og.gemm_mxfp4(opx, ofx, opw, ofw)
    return px, fx, pw, fw, Dref, bnd


@pytest.mark.parametrize("M,N,K,out", [(16, 28672, 8192, "bf16"), (1, 4096, 4096, "f32"),
                                       (32, 2048, 1024, "bf16")])
def test_noalloc_matches_workspace_entry_point(M, N, K, out):
    import torch
    import fp4_gemm_gb300 as bsg
    lib = bsg.load_library()
    px, fx, pw, fw, Dref, bnd = _inputs(M, N, K)
    ref = bsg.bsg_gemm(px, "e2m1", fx, "mx", pw, "e2m1", fw, "mx", out=out)
    dtype = torch.float32 if out == "f32" else torch.bfloat16
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        D = torch.full((M, N), float("nan"), dtype=dtype, device=px.device)
        st = lib.bsg_gemm_decode_noalloc(M, N, K, px.data_ptr(), fx.data_ptr(), pw.data_ptr(),
                                         fw.data_ptr(), None, D.data_ptr(),
                                         bsg.DTYPE[out], stream)
        assert st == 0, bsg.bsg_status_string(st)
        assert bsg.bsg_device_error() == 0
        Dh = D.float().cpu().numpy()
        ok, worst = og.within_tolerance(Dh, ref.float().cpu().numpy(), bnd, bf16=out == "bf16")
        assert ok, f"call {call} vs bsg_gemm: worst err/allowed {worst:.3g}"
        ok, worst = og.within_tolerance(Dh, Dref, bnd, bf16=out == "bf16")
        assert ok, f"call {call} vs the oracle: worst err/allowed {worst:.3g}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    import fp4_gemm_gb300 as bsg
    lib = bsg.load_library()
    device()
    M, N, K = 32, 65536, 8192
    assert bsg.bsg_gemm_workspace_size(M, N, K, "e2m1", "e2m1") > 8 << 20
    # rejected on the host before anything touches the (dummy) pointers
    st = lib.bsg_gemm_decode_noalloc(M, N, K, 256, 256, 256, 256, None, 256, 1, None)
    assert bsg.STATUS[st] == "BSG_ERR_WORKSPACE"
    st = lib.bsg_gemm_decode_noalloc(64, N, K, 256, 256, 256, 256, None, 256, 1, None)
    assert bsg.STATUS[st] == "BSG_ERR_UNSUPPORTED"

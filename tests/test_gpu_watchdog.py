"""Failure detection without a GPU fault: a kernel whose only wait is on a
barrier that nothing arrives on runs out of the library's bounded wait (2 s),
reports BSG_ERR_TIMEOUT through bsg_device_error, and leaves the context
usable for the next launches."""
import time

import numpy as np
import pytest

import synth
from helpers import device, report, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import fp4_gemm_gb300 as bsg
    dev = device()
    assert bsg.bsg_device_error() == 0
    t0 = time.perf_counter()
    bsg.bsg_check_wait_timeout()
    assert bsg.bsg_device_error() == 5          # BSG_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert 1.5 < waited < 30.0                   # the 2 s limit ended the wait
    assert bsg.bsg_device_error() == 0           # read and cleared
    # the context still runs kernels correctly
    A, B = synth.make("fp8_256")
    qa, sa = bsg.bsg_quantize_fp8(to_dev(A, dev), "e4m3", "tile")
    qb, sb = bsg.bsg_quantize_fp8(to_dev(B, dev), "e4m3", "tile")
    D = bsg.bsg_gemm(qa, "e4m3", sa, "tile", qb, "e4m3", sb, "tile", out="f32")
    assert bsg.bsg_device_error() == 0
    oqa, osa = oq.quantize_fp8(A, "e4m3", "tile")
    oqb, osb = oq.quantize_fp8(B, "e4m3", "tile")
    Dref, bnd = og.gemm_fp8(oqa, "e4m3", osa, "tile", oqb, "e4m3", osb, "tile")
    report("after timeout", *og.within_tolerance(D.cpu().numpy(), Dref, bnd))

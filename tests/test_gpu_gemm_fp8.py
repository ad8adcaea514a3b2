"""FP8 GEMM parity against the oracle within the stated tolerance:
|D - D_ref| <= 1e-4 * sum_k |s_A a_k s_B b_k| + 1e-6 (BF16 output: + 8e-3 |D_ref|)."""
import numpy as np
import pytest

import synth
from helpers import device, report, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _run(A, B, fa, fb, ga, gb, out, C=None, rows=None):
    import fp4_gemm_gb300 as bsg
    dev = device()
    qa, sa = bsg.bsg_quantize_fp8(to_dev(A, dev), fa, ga)
    qb, sb = bsg.bsg_quantize_fp8(to_dev(B, dev), fb, gb)
    Ct = None if C is None else to_dev(C, dev)
    D = bsg.bsg_gemm(qa, fa, sa, ga, qb, fb, sb, gb, C=Ct, out=out)
    assert bsg.bsg_device_error() == 0
    oqa, osa = oq.quantize_fp8(A, fa, ga)
    oqb, osb = oq.quantize_fp8(B, fb, gb)
    assert np.array_equal(qa.cpu().numpy(), oqa) and np.array_equal(qb.cpu().numpy(), oqb)
    Dref, bnd = og.gemm_fp8(oqa, fa, osa, ga, oqb, fb, osb, gb, C=C, rows=rows)
    Dg = D.float().cpu().numpy()
    if rows is not None:
        Dg = Dg[rows]
    return og.within_tolerance(Dg, Dref, bnd, bf16=out == "bf16")


def test_fp8_256_config():
    # E4M3 x E4M3, 256^3, 128x128 scales, FP32 out, 0.1 % x100 outliers
    A, B = synth.make("fp8_256")
    report("fp8_256", *_run(A, B, "e4m3", "e4m3", "tile", "tile", "f32"))


@pytest.mark.parametrize("M,N,K", [(200, 300, 272), (1, 256, 128), (129, 257, 16), (384, 520, 1040)])
@pytest.mark.parametrize("ga,gb", [("row", "tile"), ("tile", "row"), ("row", "row")])
def test_fp8_ragged(M, N, K, ga, gb):
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    report(f"ragged {M}x{N}x{K}", *_run(A, B, "e4m3", "e4m3", ga, gb, "f32"))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fp8_ffn_up_small_bf16_with_addend(out):
    A, B = synth.make("ffn_up", m=512, n=768, k=1024)
    C = synth.addend("ffn_up", 512, 768)
    report("ffn_up small", *_run(A, B, "e4m3", "e4m3", "row", "tile", out, C=C))


def test_fp8_dgrad_small_e5m2():
    # long-K accumulation: E5M2 gradients x E4M3 weights, 128x128 scales
    A, B = synth.make("dgrad", m=256, n=512, k=4096)
    report("dgrad small", *_run(A, B, "e5m2", "e4m3", "tile", "tile", "f32"))


def test_fp8_many_tiles_persistent():
    # more output tiles than SMs: every CTA walks several tiles
    A, B = synth.make("ffn_up", m=2048, n=4096, k=256)
    rows = np.r_[0:3, 1000:1003, 2045:2048]
    report("persistent", *_run(A, B, "e4m3", "e4m3", "row", "tile", "bf16", rows=rows))


def test_fp8_pair_path_ragged_bf16_addend():
    # enough 256 x 256 tiles for the CTA-pair kernel; M, N ragged (odd number
    # of 128-row blocks), rows sampled across both CTAs of a pair and the edges
    M, N, K = 4100, 2000, 384
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    C = synth.addend("ffn_up", M, N)
    rows = np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 2048, 4095, 4096, 4099])
    report("pair ragged", *_run(A, B, "e4m3", "e4m3", "row", "tile", "bf16", C=C, rows=rows))


def test_fp8_pair_path_e5m2_fp32():
    M, N, K = 2560, 2048, 1024
    A, B = synth.make("dgrad", m=M, n=N, k=K)
    rows = np.r_[0:4, 126:130, 254:258, 2556:2560]
    report("pair e5m2", *_run(A, B, "e5m2", "e4m3", "tile", "tile", "f32", rows=rows))


@pytest.mark.parametrize("M,N,K,out", [(200, 300, 272, "bf16"), (129, 257, 16, "bf16"),
                                       (130, 1001, 384, "f32")])
def test_fp8_output_pitch_not_16_bytes(M, N, K, out):
    # D's row pitch is not a multiple of 16 bytes: no TMA store; the staged
    # tile is copied out with bounds checks
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    C = synth.addend("ffn_up", M, N)
    report(f"pitch {M}x{N}x{K} {out}", *_run(A, B, "e4m3", "e4m3", "row", "tile", out, C=C))


@pytest.mark.parametrize("N,out", [(2004, "bf16"), (2001, "f32")])
def test_fp8_pair_path_output_pitch_not_16_bytes(N, out):
    M, K = 4100, 256
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    rows = np.array([0, 127, 128, 255, 256, 2047, 2048, 4095, 4096, 4099])
    report(f"pair pitch N={N} {out}", *_run(A, B, "e4m3", "e4m3", "row", "tile", out, rows=rows))

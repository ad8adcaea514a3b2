"""The FP8 GEMM with its output quantised in the epilogue (bsg_gemm_quantized).

Expected values: the oracle's step-by-step emulation of the promoted FP8 GEMM
(gemm_fp8_bits, FP32 result including the addend) quantised by the oracle's
1x128 FP8 quantiser ("FP8 GEMM on CDNA4" section 3.3) - codes and scales bit
for bit.  Where only some rows / column blocks are checked, whole 128-column
groups are emulated, since a group's scale depends on all of its elements."""
import numpy as np
import pytest

import synth
from helpers import device, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, ga, gb, fa="e4m3", workload="ffn_up"):
    import fp4_gemm_gb300 as bsg
    dev = device()
    A, B = synth.make(workload, m=M, n=N, k=K)
    qa, sa = bsg.bsg_quantize_fp8(to_dev(A, dev), fa, ga)
    qb, sb = bsg.bsg_quantize_fp8(to_dev(B, dev), "e4m3", gb)
    return A, B, qa, sa, qb, sb


def _expected(A, B, fa, ga, gb, rows, blocks, N, qfmt, fmt_max=None, C=None, a_rows_only=False):
    """Oracle codes / scales for rows x (128-column blocks) of the output."""
    if a_rows_only:   # quantise just the sampled rows of A (1x128 scales are per row)
        qa, sa = oq.quantize_fp8(A[rows], fa, ga)
        lrows = np.arange(len(rows))
    else:
        qa, sa = oq.quantize_fp8(A, fa, ga)
        lrows = np.asarray(rows)
    qb, sb = oq.quantize_fp8(B, "e4m3", gb)
    cols = np.concatenate([np.arange(b * 128, min(N, (b + 1) * 128)) for b in blocks])
    i, j = np.meshgrid(lrows, cols, indexing="ij")
    Csub = None
    if C is not None:
        Csub = np.zeros((qa.shape[0], N), np.float32)
        Csub[lrows] = C[rows]
    R = og.gemm_fp8_bits(qa, fa, sa, ga, qb, "e4m3", sb, gb, i.ravel(), j.ravel(), C=Csub, out="f32")
    R = R.astype(np.float32).reshape(len(rows), len(cols))
    codes, scales = oq.quantize_fp8(R, qfmt, "row", fmt_max)
    return cols, codes, scales


def _check(Dq, sD, rows, blocks, cols, codes, scales):
    Dq = Dq.cpu().numpy()
    sD = sD.cpu().numpy()
    assert np.array_equal(Dq[np.ix_(rows, cols)], codes)
    assert np.array_equal(sD[np.ix_(blocks, rows)], scales)


@pytest.mark.parametrize("M,N,K,ga,gb,qfmt,addend", [
    (200, 300, 272, "row", "tile", "e4m3", False),    # N % 16 != 0: bounds-checked store
    (200, 304, 272, "row", "tile", "e4m3", True),     # TMA store
    (129, 257, 16, "tile", "row", "e5m2", False),
    (264, 520, 1040, "row", "row", "e4m3", True),
    (130, 384, 512, "tile", "tile", "e5m2", True),
])
def test_fused_quant_bit_exact(M, N, K, ga, gb, qfmt, addend):
    import fp4_gemm_gb300 as bsg
    A, B, qa, sa, qb, sb = _inputs(M, N, K, ga, gb)
    C = synth.addend("ffn_up", M, N) if addend else None
    Dq, sD = bsg.bsg_gemm_quantized(qa, "e4m3", sa, ga, qb, "e4m3", sb, gb,
                                    C=None if C is None else to_dev(C, device()), qfmt=qfmt)
    assert bsg.bsg_device_error() == 0
    rows = np.arange(M)
    blocks = np.arange((N + 127) // 128)
    cols, codes, scales = _expected(A, B, "e4m3", ga, gb, rows, blocks, N, qfmt, C=C)
    _check(Dq, sD, rows, blocks, cols, codes, scales)


def test_fused_quant_dgrad_e5m2_operand_and_custom_max():
    import fp4_gemm_gb300 as bsg
    M, N, K = 160, 272, 1024
    A, B, qa, sa, qb, sb = _inputs(M, N, K, "tile", "tile", fa="e5m2", workload="dgrad")
    Dq, sD = bsg.bsg_gemm_quantized(qa, "e5m2", sa, "tile", qb, "e4m3", sb, "tile", qfmt="e4m3",
                                    fmt_max=240.0)
    assert bsg.bsg_device_error() == 0
    rows, blocks = np.arange(M), np.arange(3)
    cols, codes, scales = _expected(A, B, "e5m2", "tile", "tile", rows, blocks, N, "e4m3", fmt_max=240.0)
    _check(Dq, sD, rows, blocks, cols, codes, scales)


def test_fused_quant_zero_rows_get_unit_scale():
    import fp4_gemm_gb300 as bsg
    M, N, K = 256, 256, 256
    A, B = synth.make("ffn_up", m=M, n=N, k=K)
    A[5] = 0.0
    A[130:140] = 0.0
    dev = device()
    qa, sa = bsg.bsg_quantize_fp8(to_dev(A, dev), "e4m3", "row")
    qb, sb = bsg.bsg_quantize_fp8(to_dev(B, dev), "e4m3", "tile")
    Dq, sD = bsg.bsg_gemm_quantized(qa, "e4m3", sa, "row", qb, "e4m3", sb, "tile")
    assert bsg.bsg_device_error() == 0
    Dq, sD = Dq.cpu().numpy(), sD.cpu().numpy()
    for r in (5, 130, 139):
        assert not Dq[r].any() and np.all(sD[:, r] == 1.0)
    rows, blocks = np.arange(M), np.arange(2)
    cols, codes, scales = _expected(A, B, "e4m3", "row", "tile", rows, blocks, N, "e4m3")
    assert np.array_equal(Dq, codes) and np.array_equal(sD, scales)


def test_fused_quant_pair_kernel_sampled():
    import fp4_gemm_gb300 as bsg
    M, N, K = 4100, 2000, 384
    A, B, qa, sa, qb, sb = _inputs(M, N, K, "row", "tile")
    Dq, sD = bsg.bsg_gemm_quantized(qa, "e4m3", sa, "row", qb, "e4m3", sb, "tile")
    assert bsg.bsg_device_error() == 0
    rows = np.array([0, 1, 127, 128, 255, 256, 2047, 2048, 4095, 4096, 4099])
    blocks = np.arange((N + 127) // 128)
    cols, codes, scales = _expected(A, B, "e4m3", "row", "tile", rows, blocks, N, "e4m3",
                                    a_rows_only=True)
    _check(Dq, sD, rows, blocks, cols, codes, scales)


def test_fused_quant_ffn_up_full_size_sampled():
    # the FFN-up benchmark shape, launched as bench.py's fused-quantiser
    # workload launches it; sampled rows x three 128-column groups
    import fp4_gemm_gb300 as bsg
    _, M, N, K = synth.WORKLOADS["ffn_up"]
    A, B, qa, sa, qb, sb = _inputs(M, N, K, "row", "tile")
    Dq, sD = bsg.bsg_gemm_quantized(qa, "e4m3", sa, "row", qb, "e4m3", sb, "tile")
    assert bsg.bsg_device_error() == 0
    g = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], g.integers(0, M, 12)]))
    blocks = np.array([0, 61, N // 128 - 1])
    qb_sub_rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])
    # B's 128x128 scales are per block of 128 rows: quantise only those blocks
    cols_local, codes, scales = _expected(A, B[qb_sub_rows], "e4m3", "row", "tile", rows,
                                          np.arange(len(blocks)), len(qb_sub_rows), "e4m3",
                                          a_rows_only=True)
    cols = (blocks[:, None] * 128 + np.arange(128)[None, :]).ravel()
    Dq, sD = Dq.cpu().numpy(), sD.cpu().numpy()
    assert np.array_equal(Dq[np.ix_(rows, cols)], codes)
    assert np.array_equal(sD[np.ix_(blocks, rows)], scales)


def test_fused_output_feeds_the_next_gemm():
    # FFN up with the fused quantiser, then FFN down on its codes and scales:
    # the second GEMM reads them as an activation operand with 1x128 scales
    import fp4_gemm_gb300 as bsg
    dev = device()
    M, H, D = 192, 384, 256
    A, W1 = synth.make("ffn_up", m=M, n=H, k=D)
    _, W2 = synth.make("ffn_up", m=1, n=D, k=H)
    qa, sa = bsg.bsg_quantize_fp8(to_dev(A, dev), "e4m3", "row")
    q1, s1 = bsg.bsg_quantize_fp8(to_dev(W1, dev), "e4m3", "tile")
    q2, s2 = bsg.bsg_quantize_fp8(to_dev(W2, dev), "e4m3", "tile")
    Hq, sH = bsg.bsg_gemm_quantized(qa, "e4m3", sa, "row", q1, "e4m3", s1, "tile")
    Y = bsg.bsg_gemm(Hq, "e4m3", sH, "row", q2, "e4m3", s2, "tile", out="f32")
    assert bsg.bsg_device_error() == 0
    # oracle chain: exact-emulated hidden layer, oracle quantiser, then the
    # second GEMM emulated bit for bit
    cols, hcodes, hscales = _expected(A, W1, "e4m3", "row", "tile", np.arange(M), np.arange(3), H,
                                      "e4m3")
    oq2, os2 = oq.quantize_fp8(W2, "e4m3", "tile")
    i, j = np.meshgrid(np.arange(M), np.arange(D), indexing="ij")
    Yref = og.gemm_fp8_bits(hcodes, "e4m3", hscales, "row", oq2, "e4m3", os2, "tile",
                            i.ravel(), j.ravel(), out="f32").reshape(M, D)
    assert np.array_equal(Y.cpu().numpy().astype(np.float64), Yref)


def test_fused_quant_rejects_what_it_does_not_do():
    import fp4_gemm_gb300 as bsg
    A, B, qa, sa, qb, sb = _inputs(128, 128, 128, "row", "tile")
    with pytest.raises(bsg.BsgError) as e:
        bsg.bsg_gemm_quantized(qa, "e4m3", sa, "row", qb, "e4m3", sb, "tile", qfmt="e2m1")
    assert e.value.status == 2   # BSG_ERR_UNSUPPORTED
    with pytest.raises(bsg.BsgError) as e:
        bsg.bsg_gemm_quantized(qa, "e4m3", sa, "row", qb, "e4m3", sb, "tile", fmt_max=-1.0)
    assert e.value.status == 1   # BSG_ERR_INVALID_ARG

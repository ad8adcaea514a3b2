"""NVFP4 (E2M1 elements, E4M3 scales per 16 along K, FP32 tensor scale):
quantiser bit-exact against the oracle, GEMM within the stated tolerance
|D - D_ref| <= 1e-4 * sum_k |s_A a_k s_B b_k| + 1e-6 (BF16: + 8e-3 |D_ref|)."""
import numpy as np
import pytest

import synth
from helpers import device, report, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _bf16_tensor(x, dev):
    import torch
    bits = synth.to_bf16_bits(x)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)


@pytest.mark.parametrize("rows,cols", [(1, 16), (7, 48), (200, 272), (130, 1024)])
@pytest.mark.parametrize("g", [1.0, 2.0 ** -7, 0.0123])
@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantize_nvfp4_bit_exact(rows, cols, g, src):
    import fp4_gemm_gb300 as bsg
    dev = device()
    rng = np.random.default_rng(rows * 1000 + cols)
    x = (rng.standard_normal((rows, cols)) * np.exp2(rng.uniform(-10, 6, (rows, 1)))).astype(np.float32)
    x[0, :16] = 0.0                                         # a zero block
    if cols >= 48:
        x[-1, 16:32] *= np.float32(1e-6)                     # a block whose scale underflows
        x[-1, 32:48] = np.float32(6000.0)                    # a block whose scale saturates
    xt = _bf16_tensor(x, dev) if src == "bf16" else to_dev(x, dev)
    xr = synth.bf16_bits_to_f32(synth.to_bf16_bits(x)) if src == "bf16" else x
    op, osf = oq.quantize_nvfp4(xr, tensor_scale=g)
    p, sf = bsg.bsg_quantize_nvfp4(xt, "rowmajor", tensor_scale=g)
    assert bsg.bsg_device_error() == 0
    assert np.array_equal(p.cpu().numpy(), op)
    assert np.array_equal(sf.cpu().numpy(), osf)
    p2, sf2 = bsg.bsg_quantize_nvfp4(xt, "tcgen05", tensor_scale=g)
    assert np.array_equal(p2.cpu().numpy(), op)
    assert np.array_equal(sf2.cpu().numpy(), oq.sf_to_tcgen05_layout(osf, pad=0))


def _gemm(M, N, K, ga=1.0, gb=2.0 ** -6, out="f32", addend=False, via_bsg_gemm=False, rows=None,
          cols=None, workload="ffn_up"):
    import fp4_gemm_gb300 as bsg
    dev = device()
    A, B = synth.make(workload, m=M, n=N, k=K)
    qa, sa = bsg.bsg_quantize_nvfp4(to_dev(A, dev), tensor_scale=ga)
    qb, sb = bsg.bsg_quantize_nvfp4(to_dev(B, dev), tensor_scale=gb)
    C = synth.addend(workload, M, N) if addend else None
    Ct = None if C is None else to_dev(C, dev)
    alpha = float(np.float32(ga) * np.float32(gb))
    if via_bsg_gemm:
        assert alpha == 1.0
        D = bsg.bsg_gemm(qa, "e2m1", sa, "nv", qb, "e2m1", sb, "nv", C=Ct, out=out)
    else:
        D = bsg.bsg_gemm_nvfp4(qa, sa, qb, sb, alpha=alpha, C=Ct, out=out)
    assert bsg.bsg_device_error() == 0
    D = D.float().cpu().numpy()
    ri = np.arange(M) if rows is None else np.asarray(rows)
    ci = np.arange(N) if cols is None else np.asarray(cols)
    pa, fa = oq.quantize_nvfp4(A[ri], tensor_scale=ga)      # scales are per row: rows quantise alone
    pb, fb = oq.quantize_nvfp4(B[ci], tensor_scale=gb)
    Csub = None if C is None else C[np.ix_(ri, ci)]
    Dref, bnd = og.gemm_nvfp4(pa, fa, pb, fb, alpha=alpha, C=Csub)
    return og.within_tolerance(D[np.ix_(ri, ci)], Dref, bnd, bf16=out == "bf16")


@pytest.mark.parametrize("M,N,K", [(200, 300, 288), (1, 256, 128), (129, 257, 96), (384, 520, 1056)])
@pytest.mark.parametrize("out,addend", [("f32", False), ("bf16", True)])
def test_nvfp4_gemm_ragged(M, N, K, out, addend):
    report(f"nvfp4 {M}x{N}x{K} {out}", *_gemm(M, N, K, out=out, addend=addend))


def test_nvfp4_gemm_through_bsg_gemm():
    report("nvfp4 via bsg_gemm", *_gemm(256, 384, 512, ga=1.0, gb=1.0, via_bsg_gemm=True))


def test_nvfp4_gemm_1024_cube_wide_rows():
    report("nvfp4 1024^3", *_gemm(1024, 1024, 1024, ga=2.0 ** -2, gb=2.0 ** -2, workload="mxfp4_1024"))


def test_nvfp4_gemm_ffn_up_full_size_sampled():
    _, M, N, K = synth.WORKLOADS["ffn_up"]
    g = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], g.integers(0, M, 28)]))
    cols = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 60)]))
    report("nvfp4 ffn_up sampled", *_gemm(M, N, K, ga=1.0, gb=2.0 ** -6, out="bf16", rows=rows, cols=cols))


@pytest.mark.parametrize("M,N,K,out,addend", [(2000, 2000, 288, "f32", False),
                                              (1300, 1900, 1056, "bf16", True)])
def test_nvfp4_large_kernel_ragged(M, N, K, out, addend):
    # at least half as many 128 x 256 tiles as SMs: the large block-scaled
    # kernel (three stages of four scale atoms), partial last stage and atom
    rows = np.unique(np.concatenate([np.arange(0, M, 7), [M - 1]]))
    report(f"nvfp4 large {M}x{N}x{K}", *_gemm(M, N, K, ga=2.0 ** -1, gb=2.0 ** -6, out=out,
                                              addend=addend, rows=rows))


def test_nvfp4_large_kernel_through_bsg_gemm():
    report("nvfp4 large via bsg_gemm", *_gemm(1536, 2048, 512, ga=1.0, gb=1.0, via_bsg_gemm=True,
                                              rows=np.arange(0, 1536, 5)))


# Decode shapes (M <= 32) take the swap-AB kernel that streams the weights
# once and splits K evenly over the SMs: ragged N, N below one 128-row tile,
# K tails that leave a partial 128-byte chunk (K % 256 != 0), split tiles.
@pytest.mark.parametrize("M", [1, 7, 16, 17, 32])
@pytest.mark.parametrize("N,K", [(1000, 1024), (4096, 8192), (384, 96), (2048, 2304)])
def test_nvfp4_decode(M, N, K):
    report(f"nvfp4 decode {M}x{N}x{K}", *_gemm(M, N, K, ga=1.0, gb=2.0 ** -6, out="bf16",
                                              addend=M % 2 == 1, workload="decode"))


@pytest.mark.parametrize("M", [1, 16, 32])
def test_nvfp4_decode_through_bsg_gemm(M):
    report(f"nvfp4 decode via bsg_gemm M={M}", *_gemm(M, 2048, 4096, ga=1.0, gb=1.0, out="f32", addend=True,
                                                     via_bsg_gemm=True, workload="decode"))


def test_nvfp4_decode_full_size_sampled_columns():
    # the decode benchmark shape (N = 28672, K = 8192) at M = 16; the oracle
    # checks output columns (weight rows) at tile edges, split boundaries and
    # random places
    N, K = 28672, 8192
    rng = np.random.default_rng(11)
    cols = np.unique(np.concatenate([np.arange(0, 4), np.arange(124, 132), np.arange(N - 4, N),
                                     np.arange(128, N, 128 * 37), rng.integers(0, N, 256)]))
    report(f"nvfp4 decode full size ({cols.size} columns)",
           *_gemm(16, N, K, ga=1.0, gb=2.0 ** -6, out="bf16", cols=cols, workload="decode"))


def test_nvfp4_decode_workspace_errors():
    # a workspace that is given but too small is an error; none at all lets
    # the call fall back to the general kernel
    import ctypes
    import fp4_gemm_gb300 as bsg
    import torch
    dev = device()
    M, N, K = 16, 4096, 8192
    need = bsg.bsg_gemm_workspace_size(M, N, K, "e2m1", "e2m1")
    assert need > 0
    A, B = synth.make("decode", m=M, n=N, k=K)
    qa, sa = bsg.bsg_quantize_nvfp4(to_dev(A, dev))
    qb, sb = bsg.bsg_quantize_nvfp4(to_dev(B, dev), tensor_scale=2.0 ** -6)
    D = torch.empty((M, N), dtype=torch.float32, device=dev)
    small = torch.zeros(64, dtype=torch.uint8, device=dev)
    lib = bsg.load_library()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert lib.bsg_gemm_nvfp4_ws(M, N, K, p(qa), p(sa), p(qb), p(sb), 2.0 ** -6, None, p(D), 0, p(small), 64,
                                 None) == 6
    D1 = bsg.bsg_gemm_nvfp4(qa, sa, qb, sb, alpha=2.0 ** -6)
    assert lib.bsg_gemm_nvfp4(M, N, K, p(qa), p(sa), p(qb), p(sb), 2.0 ** -6, None, p(D), 0, None) == 0
    torch.cuda.synchronize()
    assert bsg.bsg_device_error() == 0
    # decode-shaped and general kernels agree within the tolerance
    pa, fa = oq.quantize_nvfp4(A)
    pb, fb = oq.quantize_nvfp4(B, tensor_scale=2.0 ** -6)
    Dref, bnd = og.gemm_nvfp4(pa, fa, pb, fb, alpha=2.0 ** -6)
    for X in (D1, D):
        report("nvfp4 decode / general", *og.within_tolerance(X.float().cpu().numpy(), Dref, bnd))

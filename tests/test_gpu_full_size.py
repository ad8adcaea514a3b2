"""Parity at the full benchmark sizes, launched the way the benchmark launches
them, on sampled outputs the oracle computes one by one.

* FP8 dgrad, M=8192, K=14336, N=4096: E5M2 gradients with 128x128 scales x
  E4M3 weights with 128x128 scales, FP32 out.  112 K tiles per output tile,
  i.e. 112 promotions ("FP8 MMA internals on Hopper": a chained tensor-core
  accumulator drops small terms, hence the per-K-tile promotion of "FP8 GEMM
  on CDNA4" section 4.4).  Checked three ways on sampled 128-row blocks of A
  and 128-column blocks of D: the tile quantiser's codes and scales bit-exact,
  D within |D - D_ref| <= 1e-4 * sum|s_A a s_B b| + 1e-6, and D bit-exact
  against the oracle's step-by-step emulation of the promoted GEMM.
* MXFP8 FFN-up, M=8192, K=4096, N=14336: E4M3 elements with one E8M0 scale per
  32 along K (the MX rule of "Rubin FP4 GEMM deep dive" section 4.2 with FP8
  elements), scales in the tensor core's atom order, BF16 out.  Codes and
  scale atoms of sampled blocks bit-exact; D within tolerance (+ 8e-3 |D_ref|
  for the BF16 rounding).

A 128 x 128 FP8 tile, and every row of an MX operand, is quantised on its own,
so the oracle quantises only the sampled blocks and gets the same codes as a
quantisation of the whole matrix."""
import numpy as np
import pytest

import synth
from helpers import device, report, to_dev
from oracle import gemm as og
from oracle import quantize as oq

pytestmark = pytest.mark.gpu


def _blocks_rows(blocks, offs):
    return (np.asarray(blocks)[:, None] * 128 + np.asarray(offs)[None, :]).ravel()


@pytest.fixture(scope="module")
def dgrad_run():
    import fp4_gemm_gb300 as bsg
    dev = device()
    _, M, N, K = synth.WORKLOADS["dgrad"]
    A, B = synth.make("dgrad")
    qa, sa = bsg.bsg_quantize_fp8(to_dev(A, dev), "e5m2", "tile")
    qb, sb = bsg.bsg_quantize_fp8(to_dev(B, dev), "e4m3", "tile")
    ws = bsg.workspace_for(M, N, K, "e5m2", "e4m3", dev)
    D = bsg.bsg_gemm(qa, "e5m2", sa, "tile", qb, "e4m3", sb, "tile", out="f32", workspace=ws, K=K)
    assert bsg.bsg_device_error() == 0
    rblk = np.array([0, 29, M // 128 - 1])          # sampled 128-row blocks of A
    cblk = np.array([0, 13, N // 128 - 1])          # sampled 128-column blocks of D
    rows = _blocks_rows(rblk, np.arange(128))
    cols = _blocks_rows(cblk, np.arange(128))
    rows_t = __import__("torch").from_numpy(rows).to(dev)
    cols_t = __import__("torch").from_numpy(cols).to(dev)
    out = {
        "A": A[rows], "B": B[cols], "M": M, "N": N, "K": K, "rblk": rblk, "cblk": cblk,
        "qa": qa.index_select(0, rows_t).cpu().numpy(),
        "sa": sa.cpu().numpy()[rblk], "qb": qb.index_select(0, cols_t).cpu().numpy(),
        "sb": sb.cpu().numpy()[cblk],
        "D": D.index_select(0, rows_t).index_select(1, cols_t).cpu().numpy().astype(np.float64),
    }
    del A, B
    return out


def test_dgrad_full_size_tile_quantiser_bit_exact_sampled(dgrad_run):
    r = dgrad_run
    oqa, osa = oq.quantize_fp8(r["A"], "e5m2", "tile")
    oqb, osb = oq.quantize_fp8(r["B"], "e4m3", "tile")
    assert np.array_equal(r["sa"], osa) and np.array_equal(r["qa"], oqa)
    assert np.array_equal(r["sb"], osb) and np.array_equal(r["qb"], oqb)


def test_dgrad_full_size_within_tolerance_sampled(dgrad_run):
    r = dgrad_run
    oqa, osa = oq.quantize_fp8(r["A"], "e5m2", "tile")
    oqb, osb = oq.quantize_fp8(r["B"], "e4m3", "tile")
    g = np.random.default_rng(14336)
    sel = np.unique(np.concatenate([[0, 127, 128, 255, 256, 383], g.integers(0, 384, 26)]))
    Dref, bnd = og.gemm_fp8(oqa, "e5m2", osa, "tile", oqb, "e4m3", osb, "tile", rows=sel)
    report("dgrad full size", *og.within_tolerance(r["D"][sel], Dref, bnd))


def test_dgrad_full_size_bit_exact_sampled(dgrad_run):
    r = dgrad_run
    oqa, osa = oq.quantize_fp8(r["A"], "e5m2", "tile")
    oqb, osb = oq.quantize_fp8(r["B"], "e4m3", "tile")
    g = np.random.default_rng(112)
    sel_r = np.unique(np.concatenate([[0, 127, 128, 383], g.integers(0, 384, 12)]))
    sel_c = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, 383], g.integers(0, 384, 5)]))
    i, j = np.meshgrid(sel_r, sel_c, indexing="ij")
    E = og.gemm_fp8_bits(oqa, "e5m2", osa, "tile", oqb, "e4m3", osb, "tile", i.ravel(), j.ravel(),
                         out="f32")
    assert np.array_equal(r["D"][np.ix_(sel_r, sel_c)], E.reshape(len(sel_r), len(sel_c)))


def test_mxfp8_ffn_up_full_size_sampled():
    import torch
    import fp4_gemm_gb300 as bsg
    dev = device()
    _, M, N, K = synth.WORKLOADS["ffn_up"]
    A, B = synth.make("ffn_up")
    qa, sfa = bsg.bsg_quantize_mx(to_dev(A, dev), "e4m3", "tcgen05")
    qb, sfb = bsg.bsg_quantize_mx(to_dev(B, dev), "e4m3", "tcgen05")
    D = bsg.bsg_gemm(qa, "e4m3", sfa, "mx", qb, "e4m3", sfb, "mx", out="bf16")
    assert bsg.bsg_device_error() == 0
    rblk = np.array([0, 41, M // 128 - 1])
    cblk = np.array([0, 77, N // 128 - 1])
    rows = _blocks_rows(rblk, np.arange(128))
    cols = _blocks_rows(cblk, np.arange(128))
    oca, osa = oq.quantize_mxfp8(A[rows], "e4m3")
    ocb, osb = oq.quantize_mxfp8(B[cols], "e4m3")
    assert np.array_equal(qa.index_select(0, torch.from_numpy(rows).to(dev)).cpu().numpy(), oca)
    assert np.array_equal(qb.index_select(0, torch.from_numpy(cols).to(dev)).cpu().numpy(), ocb)
    # a 128-row block's scales are one contiguous run of 512-byte atoms
    atoms = K // 32 // 4 * 512
    sfa_h, sfb_h = sfa.cpu().numpy(), sfb.cpu().numpy()
    for n, b in enumerate(rblk):
        assert np.array_equal(sfa_h[b * atoms:(b + 1) * atoms],
                              oq.sf_to_tcgen05_layout(osa[n * 128:(n + 1) * 128]))
    for n, b in enumerate(cblk):
        assert np.array_equal(sfb_h[b * atoms:(b + 1) * atoms],
                              oq.sf_to_tcgen05_layout(osb[n * 128:(n + 1) * 128]))
    g = np.random.default_rng(4096)
    sel = np.unique(np.concatenate([[0, 127, 128, 255, 256, 383], g.integers(0, 384, 26)]))
    Dref, bnd = og.gemm_mxfp8(oca, "e4m3", osa, ocb, "e4m3", osb, rows=sel)
    Dg = D.index_select(0, torch.from_numpy(rows[sel]).to(dev)).index_select(
        1, torch.from_numpy(cols).to(dev)).float().cpu().numpy()
    report("mxfp8 ffn_up full size", *og.within_tolerance(Dg, Dref, bnd, bf16=True))

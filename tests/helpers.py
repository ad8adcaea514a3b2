"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest


def device():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fp4_gemm_gb300 as bsg
    bsg.load_library()
    return torch.device("cuda:0")


def to_dev(x, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def special_f32_values():
    """FP32 bit patterns that exercise every rounding decision of a cast to
    an 8- or 4-bit float: every exponent, both signs, all 16 combinations of
    the top four mantissa bits with several patterns below them (zero, one
    ulp, half, half plus one ulp, all ones)."""
    exps = np.arange(0, 255, dtype=np.uint32)          # finite exponents
    tops = np.arange(16, dtype=np.uint32) << 19
    lows = np.array([0, 1, 0x3FFFF, 0x40000, 0x40001, 0x7FFFF, 0x20000, 0x60000], dtype=np.uint32)
    pats = (exps[:, None, None] << 23) | tops[None, :, None] | lows[None, None, :]
    pats = pats.ravel()
    pats = np.concatenate([pats, pats | np.uint32(0x80000000)])
    return pats.view(np.float32)


def report(name, ok, worst):
    assert ok, f"{name}: outside tolerance, worst err/allowed = {worst:.3g}"

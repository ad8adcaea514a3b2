"""The C-ABI library builds, loads on a machine without a GPU, and exports
every symbol include/bsg.h declares.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "bsg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsg_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("bsg_quantize_fp8", "bsg_quantize_mxfp4", "bsg_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from fp4_gemm_gb300 import build
    lib_path = build.build()
    lib = ctypes.CDLL(lib_path)
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_host_side_helpers_without_gpu():
    import fp4_gemm_gb300 as bsg
    bsg.load_library()
    assert bsg.bsg_status_string(0) == "BSG_OK"
    assert bsg.bsg_status_string(6) == "BSG_ERR_WORKSPACE"
    assert bsg.bsg_scale_bytes(256, 512, "tile") == 2 * 4 * 4
    assert bsg.bsg_scale_bytes(256, 512, "row") == 256 * 4 * 4
    assert bsg.bsg_scale_bytes(130, 96, "mx", "rowmajor") == 130 * 3
    assert bsg.bsg_scale_bytes(130, 96, "mx", "tcgen05") == 2 * 1 * 512
    assert bsg.bsg_scale_bytes(10, 48, "mx", "rowmajor") == 0      # K not a multiple of 32


def test_invalid_arguments_rejected_before_launch():
    import fp4_gemm_gb300 as bsg
    lib = bsg.load_library()
    # null pointers / bad sizes / bad enums return an error status without a GPU
    assert lib.bsg_quantize_fp8(None, 0, 4, 4, 4, 0, 0, 0.0, None, None, None) == 1
    assert lib.bsg_quantize_fp8(8, 0, 4, 4, 4, 2, 0, 0.0, 16, 16, None) == 2     # E2M1 not FP8
    assert lib.bsg_quantize_fp8(16, 0, 4, 4, 4, 0, 0, -1.0, 16, 16, None) == 1   # negative fmt_max
    assert lib.bsg_quantize_mxfp4(16, 0, 4, 40, 40, 16, 16, 0, None) == 1       # K % 32
    assert lib.bsg_gemm(0, 4, 4, 16, 0, 16, 0, 16, 0, 16, 0, None, 16, 0, None, 0, None) == 1
    assert lib.bsg_gemm(4, 4, 32, 24, 0, 16, 0, 16, 0, 16, 0, None, 16, 0, None, 0, None) == 3
    assert lib.bsg_gemm(4, 4, 32, 16, 0, 16, 0, 16, 2, 16, 2, None, 16, 0, None, 0, None) == 2
    assert lib.bsg_sf_to_tcgen05(None, 1, 1, None, None) == 1

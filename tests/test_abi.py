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


def test_newer_entry_points_reject_bad_arguments_before_launch():
    import fp4_gemm_gb300 as bsg
    lib = bsg.load_library()
    f32 = 0
    e4m3, e5m2, e2m1 = 0, 1, 2
    tile, row, mx, nv = 0, 1, 2, 3
    # bsg_gemm_quantized: null output, E2M1 output format, mixed-in MX
    # scales, fmt_max above 2^64, K % 16, misaligned scales
    args = [256, 256, 256, 16, e4m3, 16, row, 16, e4m3, 16, tile, None]
    assert lib.bsg_gemm_quantized(*args, e4m3, 0.0, None, 16, None) == 1
    assert lib.bsg_gemm_quantized(*args, e2m1, 0.0, 16, 16, None) == 2
    assert lib.bsg_gemm_quantized(256, 256, 256, 16, e4m3, 16, mx, 16, e4m3, 16, mx, None,
                                  e4m3, 0.0, 16, 16, None) == 2
    assert lib.bsg_gemm_quantized(*args, e5m2, 2.0 ** 65, 16, 16, None) == 1
    assert lib.bsg_gemm_quantized(256, 256, 24, 16, e4m3, 16, row, 16, e4m3, 16, tile, None,
                                  e4m3, 0.0, 16, 16, None) == 1
    assert lib.bsg_gemm_quantized(*args, e4m3, 0.0, 16, 18, None) == 3
    # bsg_quantize_nvfp4: null, cols % 16, bad tensor scale, misaligned codes
    assert lib.bsg_quantize_nvfp4(None, f32, 4, 32, 32, 1.0, 16, 16, 0, None) == 1
    assert lib.bsg_quantize_nvfp4(16, f32, 4, 40, 40, 1.0, 16, 16, 0, None) == 1
    assert lib.bsg_quantize_nvfp4(16, f32, 4, 32, 32, 0.0, 16, 16, 0, None) == 1
    assert lib.bsg_quantize_nvfp4(16, f32, 4, 32, 32, float("inf"), 16, 16, 0, None) == 1
    assert lib.bsg_quantize_nvfp4(16, f32, 4, 32, 32, 1.0, 18, 16, 0, None) == 3
    # bsg_gemm_nvfp4: K % 32, non-finite alpha, misaligned scales
    assert lib.bsg_gemm_nvfp4(4, 4, 48, 16, 16, 16, 16, 1.0, None, 16, f32, None) == 1
    assert lib.bsg_gemm_nvfp4(4, 4, 64, 16, 16, 16, 16, float("nan"), None, 16, f32, None) == 1
    assert lib.bsg_gemm_nvfp4(4, 4, 64, 16, 24, 16, 16, 1.0, None, 16, f32, None) == 3
    # bsg_gemm_nvfp4_ws validates the same way before it looks at the workspace
    assert lib.bsg_gemm_nvfp4_ws(4, 4, 48, 16, 16, 16, 16, 1.0, None, 16, f32, 16, 64, None) == 1
    assert lib.bsg_gemm_nvfp4_ws(4, 4, 64, 16, 16, 16, 16, float("inf"), None, 16, f32, 16, 64, None) == 1
    assert lib.bsg_gemm_nvfp4_ws(4, 4, 64, 16, 16, 24, 16, 1.0, None, 16, f32, 16, 64, None) == 3
    assert lib.bsg_gemm_nvfp4_ws(0, 4, 64, 16, 16, 16, 16, 1.0, None, 16, f32, None, 0, None) == 1
    # bsg_gemm: NVFP4 scales on one operand only
    assert lib.bsg_gemm(4, 4, 64, 16, e2m1, 16, nv, 16, e2m1, 16, mx, None, 16, f32, None, 0, None) == 2
    # scale sizes of the 1 x 16 E4M3 granularity
    assert bsg.bsg_scale_bytes(130, 96, "nv", "rowmajor") == 130 * 6
    assert bsg.bsg_scale_bytes(130, 96, "nv", "tcgen05") == 2 * 2 * 512
    assert bsg.bsg_scale_bytes(10, 40, "nv", "rowmajor") == 0

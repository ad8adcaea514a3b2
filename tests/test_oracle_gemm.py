"""Pins of the oracle GEMM: the Hopper page's vectors, closed forms and an
exact-rational brute force on tiny shapes (catches dropped terms, wrong scale
indices and transposed operands)."""
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden
from oracle import formats, gemm, quantize

VECTORS = read_golden("hopper_fp8_mma_vectors.txt")


def _e4m3_codes(vals):
    return formats.encode(np.array(vals, np.float32), "e4m3")


@pytest.mark.parametrize("row", VECTORS)
def test_exact_dot_of_hopper_vectors(row):
    a = [float(v) for v in row[0].split(",")]
    b = [float(v) for v in row[1].split(",")]
    exact = float(row[4])
    K = 32
    A = np.zeros((1, K), np.uint8)
    B = np.zeros((1, K), np.uint8)
    A[0, :len(a)] = _e4m3_codes(a)
    B[0, :len(b)] = _e4m3_codes(b)
    # the operands are exact E4M3 values
    assert list(formats.decode_array(A[0, :len(a)], "e4m3")) == a
    one = np.ones((1, 1), np.float32)
    D, Bnd = gemm.gemm_fp8(A, "e4m3", one, "tile", B, "e4m3", one, "tile")
    assert D[0, 0] == exact
    assert Bnd[0, 0] == sum(abs(x * y) for x, y in zip(a, b))


def test_all_ones_closed_form():
    M, N, K = 3, 5, 384                      # three K tiles
    A = np.full((M, K), 0x38, np.uint8)      # E4M3 1.0
    B = np.full((N, K), 0x38, np.uint8)
    sA = np.array([[0.5, 0.25, 3.0]], np.float32)
    sB = np.array([[2.0, 8.0, 0.125]], np.float32)
    D, _ = gemm.gemm_fp8(A, "e4m3", sA, "tile", B, "e4m3", sB, "tile")
    want = 128 * (0.5 * 2.0 + 0.25 * 8.0 + 3.0 * 0.125)
    assert np.all(D == want)


def test_single_nonzero_and_addend():
    M, N, K = 4, 3, 256
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    A[2, 200] = 0x44          # E4M3 3.0
    B[1, 200] = 0xC0          # E4M3 -2.0
    sA = np.array([[1.0, 0.75]], np.float32)
    sB = np.array([[1.0, 1.5]], np.float32)
    C = np.arange(M * N, dtype=np.float32).reshape(M, N)
    D, _ = gemm.gemm_fp8(A, "e4m3", sA, "tile", B, "e4m3", sB, "tile", C=C)
    want = C.astype(np.float64).copy()
    want[2, 1] += 0.75 * 3.0 * 1.5 * -2.0
    assert np.array_equal(D, want)


def _brute_fp8(A, fa, sA, ga, B, fb, sB, gb, C, rows):
    """sum_k (s_A a_k)(s_B b_k) + c in exact rationals, element by element."""
    dec = {"e4m3": formats.decode_e4m3, "e5m2": formats.decode_e5m2}
    K = A.shape[1]
    N = B.shape[0]
    out = np.zeros((len(rows), N))
    for r, i in enumerate(rows):
        for j in range(N):
            acc = Fraction(float(C[i, j]))
            for k in range(K):
                t = k // 128
                sa = sA[i // 128, t] if ga == "tile" else sA[t, i]
                sb = sB[j // 128, t] if gb == "tile" else sB[t, j]
                acc += (Fraction(float(sa)) * Fraction(dec[fa](int(A[i, k]))) *
                        Fraction(float(sb)) * Fraction(dec[fb](int(B[j, k]))))
            out[r, j] = float(acc)
    return out


@pytest.mark.parametrize("fa,ga,gb", [("e4m3", "tile", "tile"), ("e5m2", "row", "tile"),
                                      ("e4m3", "row", "row")])
def test_fp8_brute_force_tiny(fa, ga, gb):
    g = np.random.default_rng(42)
    M, N, K = 130, 3, 288            # two row tiles, three (ragged) K tiles
    rows = [0, 1, 127, 128, 129]
    xa = (g.standard_normal((M, K)) * np.exp2(g.uniform(-4, 4, (M, 1)))).astype(np.float32)
    xb = g.standard_normal((N, K)).astype(np.float32)
    A, sA = quantize.quantize_fp8(xa, fa, ga)
    B, sB = quantize.quantize_fp8(xb, "e4m3", gb)
    C = g.standard_normal((M, N)).astype(np.float32)
    D, _ = gemm.gemm_fp8(A, fa, sA, ga, B, "e4m3", sB, gb, C=C, rows=rows)
    want = _brute_fp8(A, fa, sA, ga, B, "e4m3", sB, gb, C, rows)
    assert np.allclose(D, want, rtol=1e-14, atol=0)


def test_fp8_transposed_b_is_detected():
    # B is stored N x K: using it as K x N must give a different answer
    g = np.random.default_rng(9)
    x = g.standard_normal((128, 128)).astype(np.float32)
    y = g.standard_normal((128, 128)).astype(np.float32)
    A, sA = quantize.quantize_fp8(x, "e4m3", "tile")
    B, sB = quantize.quantize_fp8(y, "e4m3", "tile")
    D, _ = gemm.gemm_fp8(A, "e4m3", sA, "tile", B, "e4m3", sB, "tile")
    Dt, _ = gemm.gemm_fp8(A, "e4m3", sA, "tile", np.ascontiguousarray(B.T), "e4m3", sB, "tile")
    a = formats.decode_array(A, "e4m3") * float(sA[0, 0])
    b = formats.decode_array(B, "e4m3") * float(sB[0, 0])
    assert np.allclose(D, a @ b.T, rtol=1e-12)
    assert not np.allclose(Dt, D)


def test_mxfp4_brute_force_tiny():
    g = np.random.default_rng(4)
    M, N, K = 3, 4, 96
    xa = (g.standard_normal((M, K)) * np.exp2(g.uniform(-8, 8, (M, 1)))).astype(np.float32)
    xb = (g.standard_normal((N, K)) * np.exp2(g.uniform(-8, 8, (N, 1)))).astype(np.float32)
    A, sfA = quantize.quantize_mxfp4(xa)
    B, sfB = quantize.quantize_mxfp4(xb)
    C = g.standard_normal((M, N)).astype(np.float32)
    D, Bnd = gemm.gemm_mxfp4(A, sfA, B, sfB, C=C)
    ca = formats.unpack_e2m1(A)
    cb = formats.unpack_e2m1(B)
    for i in range(M):
        for j in range(N):
            acc = Fraction(float(C[i, j]))
            bnd = Fraction(0)
            for k in range(K):
                ta = Fraction(formats.decode_e2m1(int(ca[i, k]))) * Fraction(2) ** (int(sfA[i, k // 32]) - 127)
                tb = Fraction(formats.decode_e2m1(int(cb[j, k]))) * Fraction(2) ** (int(sfB[j, k // 32]) - 127)
                acc += ta * tb
                bnd += abs(ta * tb)
            assert D[i, j] == float(acc)
            assert Bnd[i, j] == float(bnd)


def test_tolerance_helper():
    ref = np.array([[1.0, -2.0]])
    bnd = np.array([[10.0, 10.0]])
    ok, worst = gemm.within_tolerance(ref + 5e-4, ref, bnd)
    assert ok and worst < 1
    ok, _ = gemm.within_tolerance(ref + 2e-3, ref, bnd)
    assert not ok
    ok, _ = gemm.within_tolerance(ref * (1 + 7e-3), ref, bnd, bf16=True)
    assert ok


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_mxfp8_brute_force_tiny(fa, fb):
    g = np.random.default_rng(7)
    M, N, K = 3, 4, 96
    xa = (g.standard_normal((M, K)) * np.exp2(g.uniform(-8, 8, (M, 1)))).astype(np.float32)
    xb = (g.standard_normal((N, K)) * np.exp2(g.uniform(-8, 8, (N, 1)))).astype(np.float32)
    A, sfA = quantize.quantize_mxfp8(xa, fa)
    B, sfB = quantize.quantize_mxfp8(xb, fb)
    C = g.standard_normal((M, N)).astype(np.float32)
    D, Bnd = gemm.gemm_mxfp8(A, fa, sfA, B, fb, sfB, C=C)
    dec = {"e4m3": formats.decode_e4m3, "e5m2": formats.decode_e5m2}
    for i in range(M):
        for j in range(N):
            acc = Fraction(float(C[i, j]))
            bnd = Fraction(0)
            for k in range(K):
                ta = Fraction(dec[fa](int(A[i, k]))) * Fraction(2) ** (int(sfA[i, k // 32]) - 127)
                tb = Fraction(dec[fb](int(B[j, k]))) * Fraction(2) ** (int(sfB[j, k // 32]) - 127)
                acc += ta * tb
                bnd += abs(ta * tb)
            assert abs(D[i, j] - float(acc)) <= 1e-15 * float(bnd) + 1e-300
            assert Bnd[i, j] == pytest.approx(float(bnd), rel=1e-15)


def test_mxfp8_all_ones_closed_form_with_scales():
    # every element 1.0 (E4M3 0x38), A's scales 2^1 on its first K block and
    # 2^0 elsewhere, B's scales 2^-3: D = K/32 blocks * 32 * 2^(eA - 3)
    M, N, K = 2, 3, 128
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    sfA = np.full((M, K // 32), 127, np.uint8)
    sfA[:, 0] = 128
    sfB = np.full((N, K // 32), 124, np.uint8)
    D, Bnd = gemm.gemm_mxfp8(A, "e4m3", sfA, B, "e4m3", sfB)
    expect = (32 * 2.0 + 3 * 32 * 1.0) * 2.0 ** -3
    assert np.all(D == expect) and np.all(Bnd == expect)

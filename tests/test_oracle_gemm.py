"""Pins of the oracle GEMM: the Hopper page's vectors, closed forms and an
exact-rational brute force on tiny shapes (catches dropped terms, wrong scale
indices and transposed operands)."""
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden
from oracle import fda, formats, gemm, quantize

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


def test_f32_fma_single_rounding_at_a_midpoint():
    # (1 + 2^-23)(1 - 2^-24) + 2^-47 (1 + 2^-23) = 1 + 2^-24 + 2^-70: float64
    # rounds the sum onto the FP32 midpoint 1 + 2^-24, the exact value lies
    # above it, so one rounding gives 1 + 2^-23 (two roundings would give 1)
    a = np.array([1 + 2.0 ** -23])
    b = np.array([1 - 2.0 ** -24])
    assert gemm.f32_fma(a, b, np.array([2.0 ** -47 * (1 + 2.0 ** -23)]))[0] == 1 + 2.0 ** -23
    # an exact tie goes to the even neighbour
    assert gemm.f32_fma(a, b, np.array([2.0 ** -47]))[0] == 1.0


def test_f32_fma_random_against_exact_rationals():
    g = np.random.default_rng(12)
    a = (g.standard_normal(500) * np.exp2(g.integers(-20, 20, 500))).astype(np.float32).astype(np.float64)
    b = (g.standard_normal(500) * np.exp2(g.integers(-20, 20, 500))).astype(np.float32).astype(np.float64)
    c = (g.standard_normal(500) * np.exp2(g.integers(-40, 40, 500))).astype(np.float32).astype(np.float64)
    r = gemm.f32_fma(a, b, c)
    for i in range(500):
        x = Fraction(a[i]) * Fraction(b[i]) + Fraction(c[i])
        lo = np.float32(float(x))
        cands = [lo, np.nextafter(lo, np.float32(np.inf)), np.nextafter(lo, np.float32(-np.inf))]
        best = min(cands, key=lambda v: (abs(Fraction(float(v)) - x), int(np.array(v).view(np.uint32)) & 1))
        assert r[i] == float(best)


def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(13)
    x = (g.standard_normal(10000) * np.exp2(g.integers(-30, 30, 10000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(gemm.bf16_round(x.astype(np.float64)), ref)


def test_emulated_gemm_with_hopper_parameters_gives_the_page_bits():
    # one 32-wide K block holding the page's vectors, unit scales: with
    # Hopper's F = 13, G = 13 the emulation returns the bits the page prints
    for row in VECTORS:
        a = [float(v) for v in row[0].split(",")]
        b = [float(v) for v in row[1].split(",")]
        A = np.zeros((1, 32), np.uint8)
        B = np.zeros((1, 32), np.uint8)
        A[0, :len(a)] = _e4m3_codes(a)
        B[0, :len(b)] = _e4m3_codes(b)
        one = np.ones((1, 1), np.float32)
        d = gemm.gemm_fp8_bits(A, "e4m3", one, "tile", B, "e4m3", one, "tile", [0], [0], F=13, G=13)
        assert fda.f32_bits(d[0]) == int(row[2], 16)
        d = gemm.gemm_fp8_bits(A, "e4m3", one, "tile", B, "e4m3", one, "tile", [0], [0])
        assert d[0] == float(row[4])


def test_emulated_gemm_is_exact_where_the_gemm_is_exact():
    # small integers and power-of-two scales: nothing rounds anywhere
    g = np.random.default_rng(14)
    M, N, K = 5, 6, 320
    A = _e4m3_codes(g.integers(-3, 4, (M, K)).astype(np.float32)).reshape(M, K)
    B = _e4m3_codes(g.integers(-3, 4, (N, K)).astype(np.float32)).reshape(N, K)
    sA = np.exp2(g.integers(-4, 4, (1, 3))).astype(np.float32)
    sB = np.exp2(g.integers(-4, 4, (1, 3))).astype(np.float32)
    C = g.integers(-8, 8, (M, N)).astype(np.float32)
    D, _ = gemm.gemm_fp8(A, "e4m3", sA, "tile", B, "e4m3", sB, "tile", C=C)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    E = gemm.gemm_fp8_bits(A, "e4m3", sA, "tile", B, "e4m3", sB, "tile", rows.ravel(), cols.ravel(), C=C)
    assert np.array_equal(E.reshape(M, N), D)


def test_emulated_gemm_truncates_far_terms():
    # one K block: 16 * 16 = 256 and 2^-9 * 2^-9 = 2^-18, 26 bits below: the
    # MMA model drops it (exact GEMM keeps it); the FP32 promotion then adds
    # the partials of two K tiles exactly
    A = np.zeros((1, 256), np.uint8)
    B = np.zeros((1, 256), np.uint8)
    A[0, [0, 1, 128]] = _e4m3_codes([16.0, 2.0 ** -9, 1.0])
    B[0, [0, 1, 128]] = _e4m3_codes([16.0, 2.0 ** -9, 1.0])
    one = np.ones((1, 2), np.float32)
    d = gemm.gemm_fp8_bits(A, "e4m3", one, "tile", B, "e4m3", one, "tile", [0], [0])
    assert d[0] == 257.0
    D, _ = gemm.gemm_fp8(A, "e4m3", one, "tile", B, "e4m3", one, "tile")
    assert D[0, 0] == 257.0 + 2.0 ** -18


def test_nvfp4_brute_force_tiny():
    g = np.random.default_rng(9)
    M, N, K = 3, 5, 64
    xa = (g.standard_normal((M, K)) * np.exp2(g.uniform(-3, 3, (M, 1)))).astype(np.float32)
    xb = (g.standard_normal((N, K)) * 0.02).astype(np.float32)
    A, sfA = quantize.quantize_nvfp4(xa)
    B, sfB = quantize.quantize_nvfp4(xb, tensor_scale=2.0 ** -6)
    C = g.standard_normal((M, N)).astype(np.float32)
    alpha = 2.0 ** -6
    D, Bnd = gemm.gemm_nvfp4(A, sfA, B, sfB, alpha=alpha, C=C)
    ca, cb = formats.unpack_e2m1(A), formats.unpack_e2m1(B)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            bnd = Fraction(0)
            for k in range(K):
                ta = Fraction(formats.decode_e2m1(int(ca[i, k]))) * Fraction(formats.decode_e4m3(int(sfA[i, k // 16])))
                tb = Fraction(formats.decode_e2m1(int(cb[j, k]))) * Fraction(formats.decode_e4m3(int(sfB[j, k // 16])))
                acc += ta * tb
                bnd += abs(ta * tb)
            exact = Fraction(alpha) * acc + Fraction(float(C[i, j]))
            assert abs(D[i, j] - float(exact)) <= 1e-15 * float(bnd * Fraction(alpha)) + 1e-300
            assert Bnd[i, j] == pytest.approx(float(Fraction(alpha) * bnd), rel=1e-15)


def test_nvfp4_closed_form_with_mixed_block_scales():
    # every element 1.0 (E2M1 code 2), A's scales 2.0 (E4M3 0x40) on the
    # first 16-block and 0.5 (0x30) elsewhere, B's scales 1.0 (0x38), alpha 3
    M, N, K = 2, 3, 64
    A = formats.pack_e2m1(np.full((M, K), 2, np.uint8))
    B = formats.pack_e2m1(np.full((N, K), 2, np.uint8))
    sfA = np.full((M, K // 16), 0x30, np.uint8)
    sfA[:, 0] = 0x40
    sfB = np.full((N, K // 16), 0x38, np.uint8)
    D, _ = gemm.gemm_nvfp4(A, sfA, B, sfB, alpha=3.0)
    assert np.all(D == 3.0 * (16 * 2.0 + 48 * 0.5))


def _pow2_scales(rng, rows, blocks, lo, hi):
    return (127 + rng.integers(lo, hi + 1, (rows, blocks))).astype(np.uint8)


def test_mx_bits_emulation_equals_exact_gemm_when_nothing_rounds():
    # Operands whose partial sums all fit FP32's 24 bits and lie inside every
    # alignment window: the MMA chain must then return the exact GEMM of
    # gemm_mxfp8 / gemm_mxfp4 / gemm_nvfp4 (pinned above), so a wrong scale
    # index, block, operand or K order in the emulation shows up here.
    rng = np.random.default_rng(21)
    M, N = 6, 5
    i, j = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    i, j = i.ravel(), j.ravel()
    # MXFP8: E4M3 normals in [1, 8) (codes 0x38..0x4F, both signs), scales 2^0..2^1
    K = 96
    codes = np.r_[np.arange(0x38, 0x50), np.arange(0xB8, 0xD0)].astype(np.uint8)
    A, B = rng.choice(codes, (M, K)), rng.choice(codes, (N, K))
    sA, sB = _pow2_scales(rng, M, K // 32, 0, 1), _pow2_scales(rng, N, K // 32, 0, 1)
    C = rng.integers(-64, 64, (M, N)).astype(np.float32)
    Dx, _ = gemm.gemm_mxfp8(A, "e4m3", sA, B, "e4m3", sB, C=C)
    E = gemm.gemm_mx_bits("mxfp8", A, sA, B, sB, i, j, "e4m3", "e4m3", C=C)
    assert np.array_equal(E, Dx[i, j])
    # MXFP4: all E2M1 codes, scales 2^-2..2^2, K = 160 (a half-filled tail MMA)
    K = 160
    pa = formats.pack_e2m1(rng.integers(0, 16, (M, K)).astype(np.uint8))
    pb = formats.pack_e2m1(rng.integers(0, 16, (N, K)).astype(np.uint8))
    sA, sB = _pow2_scales(rng, M, K // 32, -2, 2), _pow2_scales(rng, N, K // 32, -2, 2)
    Dx, _ = gemm.gemm_mxfp4(pa, sA, pb, sB)
    E = gemm.gemm_mx_bits("mxfp4", pa, sA, pb, sB, i, j)
    assert np.array_equal(E, Dx[i, j])
    # NVFP4: E2M1 codes of magnitude <= 2, E4M3 scales 0.5..3.75, alpha = 2^-3
    K = 128
    small = np.r_[0:5, 8:13].astype(np.uint8)
    pa = formats.pack_e2m1(rng.choice(small, (M, K)))
    pb = formats.pack_e2m1(rng.choice(small, (N, K)))
    sA = rng.integers(0x30, 0x48, (M, K // 16)).astype(np.uint8)
    sB = rng.integers(0x30, 0x48, (N, K // 16)).astype(np.uint8)
    C = rng.integers(-64, 64, (M, N)).astype(np.float32)
    Dx, _ = gemm.gemm_nvfp4(pa, sA, pb, sB, alpha=0.125, C=C)
    E = gemm.gemm_mx_bits("nvfp4", pa, sA, pb, sB, i, j, C=C, alpha=0.125)
    assert np.array_equal(E, Dx[i, j])
    # BF16 output is the round-to-nearest-even of the FP32 result
    Eb = gemm.gemm_mx_bits("nvfp4", pa, sA, pb, sB, i, j, C=C, alpha=0.125, out="bf16")
    assert np.array_equal(Eb, gemm.bf16_round(Dx[i, j]))

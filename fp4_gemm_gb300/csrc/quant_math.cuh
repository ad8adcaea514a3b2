// Device arithmetic shared by the quantisers and by the GEMM epilogue that
// quantises its own output: FP8 and E2M1 conversions, the FP8 group scale,
// a correctly rounded division by a group's scale, and the E8M0 rounding.
// The rules are those of "FP8 GEMM on CDNA4" section 3.3 (s = max_abs /
// fmt_max, x / s stored as FP8) and "Rubin FP4 GEMM deep dive" section 4.2
// (nearest power of two of max_abs / 6, E2M1 elements).
#pragma once
#include <cstdint>

#include "common.cuh"

namespace bsg {

// Four FP32 values -> four FP8 codes, first value in the lowest byte.
__device__ __forceinline__ uint32_t cvt4_fp8(int fmt, float a, float b, float c, float d) {
  uint16_t lo, hi;
  if (fmt == 0) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  }
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float fp8_scale(float amax, float fmt_max) {
  float s = __fdiv_rn(amax, fmt_max);
  return s == 0.0f ? 1.0f : s;
}

// Correctly rounded x / s for a whole group that shares the divisor s.
//
// Markstein's division with a fused multiply-add (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with r = RN(1/s) and a faithful quotient q, the residual
// x - q s is exact and RN(q + (x - q s) r) = RN(x / s).  One correction step
// from RN(x r) (within 1.5 ulp) first makes q faithful.  The theorem needs
// every intermediate normal: for s in [2^-80, 2^80] that holds whenever
// |x / s| >= 2^-18, and smaller quotients become a signed zero in E4M3 and
// E5M2 whichever way they round, so only their sign is fixed up.  Groups
// with s outside that range (or not finite) divide with __fdiv_rn.
struct GroupDiv {
  float s, r;
  bool fast;
  __device__ __forceinline__ explicit GroupDiv(float s_) : s(s_) {
    fast = s_ >= 0x1p-80f && s_ <= 0x1p80f;
    r = __frcp_rn(s_);
  }
  // r_ must be RN(1 / s_), computed once for the group and shared
  __device__ __forceinline__ GroupDiv(float s_, float r_) : s(s_), r(r_) {
    fast = s_ >= 0x1p-80f && s_ <= 0x1p80f;
  }
  __device__ __forceinline__ float operator()(float x) const {
    if (!fast) return __fdiv_rn(x, s);
    const float q0 = x * r;
    const float q1 = fmaf(fmaf(-q0, s, x), r, q0);
    const float q2 = fmaf(fmaf(-q1, s, x), r, q1);
    return q2 == 0.0f ? x * 0.0f : q2;
  }
};

// Four FP8 codes of x / s (s = d.s), each quotient correctly rounded to FP32
// first: the codes of cvt4_fp8(fmt, RN(a/s), RN(b/s), RN(c/s), RN(e/s)).
// The range test is taken once for the four.  In range, Markstein's steps
// give RN(x/s) whenever |x/s| >= 2^-18; smaller quotients are an FP8 zero
// whichever way they round, so each code's sign bit is taken from its x
// (a quotient of x by a positive s has x's sign) and GroupDiv's per-element
// zero fix-up is not needed.
__device__ __forceinline__ uint32_t fp8_codes4(int fmt, const GroupDiv& d, float a, float b, float c,
                                               float e) {
  float q[4] = {a, b, c, e};
  if (d.fast) {
    // the same steps on pairs (fma.rn.f32x2 rounds each half like fmaf):
    // t = x r; t = (x - t s) r + t, twice; -t s + x is written t (-s) + x
    const uint64_t r2 = f32x2_pack(d.r, d.r), ns2 = f32x2_pack(-d.s, -d.s);
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      const uint64_t x2 = f32x2_pack(q[i], q[i + 1]);
      uint64_t t = fmul2(x2, r2);
      uint64_t rem = x2;
      ffma2(rem, t, ns2);
      ffma2(t, rem, r2);
      rem = x2;
      ffma2(rem, t, ns2);
      ffma2(t, rem, r2);
      f32x2_unpack(t, q[i], q[i + 1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = __fdiv_rn(q[i], d.s);
  }
  const uint32_t sg = __byte_perm(__byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0073),
                                  __byte_perm(__float_as_uint(c), __float_as_uint(e), 0x0073), 0x5410);
  return (cvt4_fp8(fmt, q[0], q[1], q[2], q[3]) & 0x7F7F7F7Fu) | (sg & 0x80808080u);
}

// E8M0 code of the power of two nearest to v >= 0 (ties up), from v's bits.
__device__ __forceinline__ uint32_t e8m0_nearest(float v) {
  const uint32_t b = __float_as_uint(v);
  const int ef = static_cast<int>((b >> 23) & 0xFFu);
  const uint32_t mf = b & 0x7FFFFFu;
  int e;
  if (ef != 0) {
    e = ef - 127 + (mf >= 0x400000u ? 1 : 0);
  } else if (mf == 0) {
    return 127u;  // v == 0
  } else {
    const int p = 31 - __clz(mf);  // leading one of the subnormal significand
    e = p - 149 + ((p >= 1 && ((mf >> (p - 1)) & 1u)) ? 1 : 0);
  }
  e += 127;
  return static_cast<uint32_t>(e < 0 ? 0 : (e > 254 ? 254 : e));
}

// Value of a non-negative E4M3 code (0x00..0x7E), exact in FP32.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e != 0u ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0x1p-9f;
}

__device__ __forceinline__ uint32_t cvt2_e2m1(float first, float second) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(r)
      : "f"(second), "f"(first));
  return r & 0xFFu;
}

__device__ __forceinline__ int64_t sf_tc_offset(int64_t row, int64_t b, int64_t kb_groups) {
  return ((row >> 7) * kb_groups + (b >> 2)) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4 +
         (b & 3);
}

}  // namespace bsg

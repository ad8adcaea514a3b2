// Quantisers: FP32/BF16 -> FP8 (E4M3/E5M2) with FP32 per-tile scales, and
// FP32/BF16 -> MXFP4 (E2M1 + E8M0 per 32 along K).
//
// FP8 ("FP8 GEMM on CDNA4", sections 3.3 and 4.2): each scale group's largest
// magnitude comes from a warp-shuffle max reduction; s = max_abs / fmt_max in
// FP32; every element is divided by s (correctly rounded FP32 division, see
// GroupDiv) and converted with the hardware's round-to-nearest-even,
// saturating cvt.
//
// MXFP4 ("Rubin FP4 GEMM deep dive", section 4.2 steps 1-3): per 32-element
// block v = max_abs / 6 in FP32; the E8M0 scale is the power of two nearest to
// v (linear distance, ties to the larger), read off v's exponent field and its
// first mantissa bit; elements are multiplied by the exact inverse power of
// two and converted with cvt.rn.satfinite.e2m1x2; two codes per byte, the
// first element in the low nibble.  MXFP8 applies the same rule with the FP8
// format's largest value in place of 6 and E4M3 / E5M2 elements.
//
// All kernels are single-pass and HBM-bound: each element is read once and
// its code written once.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "quant_math.cuh"

namespace bsg {
namespace {

__device__ uint32_t g_quant_error = 0;

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Load 4 consecutive source elements starting at (row, col) as FP32; columns
// at or beyond `cols` read as 0.
template <bool kBF16>
__device__ __forceinline__ void load4(const void* x, int64_t row, int64_t col, int64_t cols,
                                      int64_t ld, bool vec_ok, float (&v)[4]) {
  if (kBF16) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + row * ld + col;
    if (vec_ok && col + 3 < cols) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
      v[0] = __uint_as_float(u.x << 16);
      v[1] = __uint_as_float(u.x & 0xFFFF0000u);
      v[2] = __uint_as_float(u.y << 16);
      v[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = (col + j < cols) ? bf16_to_f32(p[j]) : 0.0f;
    }
  } else {
    const float* p = static_cast<const float*>(x) + row * ld + col;
    if (vec_ok && col + 3 < cols) {
      const float4 u = __ldg(reinterpret_cast<const float4*>(p));
      v[0] = u.x;
      v[1] = u.y;
      v[2] = u.z;
      v[3] = u.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = (col + j < cols) ? p[j] : 0.0f;
    }
  }
}

__device__ __forceinline__ void store_codes4(uint8_t* q, int64_t off, int64_t col, int64_t cols,
                                             bool vec_ok, uint32_t codes) {
  if (vec_ok && col + 3 < cols) {
    *reinterpret_cast<uint32_t*>(q + off) = codes;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (col + j < cols) q[off + j] = static_cast<uint8_t>(codes >> (8 * j));
  }
}

// One CTA per 128 x 128 tile; 512 threads, thread t owns columns 4*(t%32)..+3
// of rows t/32 + 16i, i < 8 (32 values in registers, so several CTAs fit on
// an SM and keep enough loads in flight).
constexpr int kTileThreads = 512;
constexpr int kTileRowsPerThread = 128 / (kTileThreads / 32);

template <bool kBF16>
__global__ void __launch_bounds__(kTileThreads) quantize_fp8_tile_kernel(
    const void* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, int fmt, float fmt_max,
    bool vec_in, bool vec_out, uint8_t* __restrict__ q, float* __restrict__ scales) {
  grid_dep_launch();
  grid_dep_wait();
  constexpr int kWarps = kTileThreads / 32;
  __shared__ float warp_max[kWarps];
  __shared__ float tile_scale, tile_rcp;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int cg = threadIdx.x & 31;
  const int rr = threadIdx.x >> 5;
  const int64_t col = c0 + 4 * cg;
  float v[kTileRowsPerThread][4];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kTileRowsPerThread; ++i) {
    const int64_t row = r0 + rr + kWarps * i;
    if (row < rows && col < cols) {
      load4<kBF16>(x, row, col, cols, ld, vec_in, v[i]);
    } else {
      v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (cg == 0) warp_max[rr] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = warp_max[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, warp_max[w]);
    const float s = fp8_scale(m, fmt_max);
    tile_scale = s;
    tile_rcp = __frcp_rn(s);
    scales[static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x] = s;
  }
  __syncthreads();
  const GroupDiv div(tile_scale, tile_rcp);
#pragma unroll
  for (int i = 0; i < kTileRowsPerThread; ++i) {
    const int64_t row = r0 + rr + kWarps * i;
    if (row < rows && col < cols) {
      const uint32_t c = fp8_codes4(fmt, div, v[i][0], v[i][1], v[i][2], v[i][3]);
      store_codes4(q, row * cols + col, col, cols, vec_out, c);
    }
  }
}

// Row quantiser (1 x 128 groups along each row).  A warp takes 512-column
// chunks of rows, lane l the 16 consecutive values 16l..16l+15, so the eight
// lanes of a 128-wide group find its maximum in three shuffle levels, and
// every lane loads and stores whole 16-byte pieces.  The warps walk the
// chunks grid-stride, each loading its next chunk before it converts the
// current one, so two chunks' loads are in flight per warp.  Scales are
// stored K-tile major, scales[t * rows + row], as the GEMM reads them.
constexpr int kRowWarps = 8;

template <bool kBF16>
__device__ __forceinline__ void load16(const void* x, int64_t row, int64_t col, int64_t cols, int64_t ld,
                                       bool vec_ok, float (&v)[16]) {
  if (kBF16) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + row * ld + col;
    if (vec_ok && col + 15 < cols) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + h);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * h + 2 * j] = __uint_as_float(w[j] << 16);
          v[8 * h + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = (col + j < cols) ? bf16_to_f32(p[j]) : 0.0f;
    }
  } else {
    const float* p = static_cast<const float*>(x) + row * ld + col;
    if (vec_ok && col + 15 < cols) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p) + h);
        v[4 * h] = u.x; v[4 * h + 1] = u.y; v[4 * h + 2] = u.z; v[4 * h + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = (col + j < cols) ? p[j] : 0.0f;
    }
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kRowWarps * 32) quantize_fp8_row_kernel(
    const void* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, int fmt, float fmt_max,
    bool vec_in, bool vec_out, uint8_t* __restrict__ q, float* __restrict__ scales) {
  grid_dep_launch();
  grid_dep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t chunks = (cols + 511) / 512;    // 512-column chunks per row
  const int64_t total = rows * chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRowWarps;
  // chunk w's row and this lane's first column in it
  auto where = [&](int64_t w, int64_t& row, int64_t& col) {
    row = w / chunks;
    col = (w - row * chunks) * 512 + 16 * lane;
  };
  auto load = [&](int64_t w, float (&v)[16]) {
    int64_t row, col;
    where(w, row, col);
    if (w < total && col < cols) {
      load16<kBF16>(x, row, col, cols, ld, vec_in, v);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.0f;   // past the row's end: no effect on the maximum
    }
  };
  auto convert = [&](int64_t w, const float (&v)[16]) {
    int64_t row, col;
    where(w, row, col);
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(v[j]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float sc = fp8_scale(a, fmt_max);
    const GroupDiv div(sc, __frcp_rn(sc));
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = fp8_codes4(fmt, div, v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    if (col < cols) {
      uint8_t* dst = q + row * cols + col;
      if (vec_out && col + 15 < cols) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (col + j < cols) dst[j] = static_cast<uint8_t>(c[j / 4] >> (8 * (j % 4)));
      }
      if ((lane & 7) == 0) scales[(col / 128) * rows + row] = sc;   // the group's first lane
    }
  };
  // w is uniform across the warp, so are the loop's branches
  int64_t w = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  float va[16], vb[16];
  load(w, va);
  for (; w < total; w += 2 * stride) {
    load(w + stride, vb);
    convert(w, va);
    if (w + stride >= total) break;
    load(w + 2 * stride, va);
    convert(w + stride, vb);
  }
}

// MX quantiser: one warp per (row, 256-column chunk); lane l owns 8
// elements, 4 lanes per 32-element block.  kFmt 2: E2M1 codes packed two per
// byte (MXFP4); kFmt 0 / 1: E4M3 / E5M2 codes, one per byte (MXFP8).  In the
// tcgen05 layout the grid also covers the padding rows / K-blocks of the last
// atoms and writes 127 there.
template <bool kBF16, bool kTC, int kFmt>
__global__ void __launch_bounds__(256) quantize_mx_kernel(
    const void* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, float fmt_max, bool vec_in,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  grid_dep_launch();
  grid_dep_wait();
  const int64_t kb = cols / 32;
  const int64_t kb_pad = kTC ? ((kb + 3) / 4) * 4 : kb;
  const int64_t chunks = (kb_pad + 7) / 8;
  const int64_t rows_pad = kTC ? ((rows + 127) / 128) * 128 : rows;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (w >= rows_pad * chunks) return;
  const int64_t row = w / chunks, chunk = w % chunks;
  const int lane = threadIdx.x & 31;
  const int64_t b = chunk * 8 + (lane >> 2);
  const int64_t col = b * 32 + (lane & 3) * 8;
  const bool data = row < rows && b < kb;
  float v[8];
  if (data) {
    load4<kBF16>(x, row, col, cols, ld, vec_in, *reinterpret_cast<float(*)[4]>(&v[0]));
    load4<kBF16>(x, row, col + 4, cols, ld, vec_in, *reinterpret_cast<float(*)[4]>(&v[4]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const uint32_t code = e8m0_nearest(__fdiv_rn(amax, fmt_max));
  if (data) {
    // 2^-(code-127) as an FP32 normal: code in [0,254] -> exponent field 254-code
    const float inv = __uint_as_float(static_cast<uint32_t>(254 - static_cast<int>(code)) << 23);
    if (kFmt == 2) {
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        packed |= cvt2_e2m1(v[2 * j] * inv, v[2 * j + 1] * inv) << (8 * j);
      *reinterpret_cast<uint32_t*>(q + row * (cols / 2) + col / 2) = packed;
    } else {
      uint2 c;
      c.x = cvt4_fp8(kFmt, v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
      c.y = cvt4_fp8(kFmt, v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
      *reinterpret_cast<uint2*>(q + row * cols + col) = c;
    }
  }
  if ((lane & 3) == 0 && b < kb_pad) {
    const uint8_t c = data ? static_cast<uint8_t>(code) : static_cast<uint8_t>(127);
    if (kTC) {
      sf[sf_tc_offset(row, b, kb_pad / 4)] = c;
    } else if (data) {
      sf[row * kb + b] = c;
    }
  }
}

// NVFP4 quantiser: one warp per (row, 256-column chunk = 16 blocks of 16);
// lane l owns 8 elements, 2 lanes per block.  Per block: v = max / 6,
// u = v / g (FP32 divisions, round to nearest), scale code = E4M3(u)
// (RNE, saturating), s = E4M3(code) * g, elements E2M1(x / s) with a
// correctly rounded quotient; s = 0 stores zero codes.  In the tcgen05
// layout the padding bytes get 0.
template <bool kBF16, bool kTC>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(
    const void* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, float g, bool vec_in,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  grid_dep_launch();
  grid_dep_wait();
  const int64_t kb = cols / 16;
  const int64_t kb_pad = kTC ? ((kb + 3) / 4) * 4 : kb;
  const int64_t chunks = (kb_pad + 15) / 16;
  const int64_t rows_pad = kTC ? ((rows + 127) / 128) * 128 : rows;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (w >= rows_pad * chunks) return;
  const int64_t row = w / chunks, chunk = w % chunks;
  const int lane = threadIdx.x & 31;
  const int64_t b = chunk * 16 + (lane >> 1);
  const int64_t col = b * 16 + (lane & 1) * 8;
  const bool data = row < rows && b < kb;
  float v[8];
  if (data) {
    load4<kBF16>(x, row, col, cols, ld, vec_in, *reinterpret_cast<float(*)[4]>(&v[0]));
    load4<kBF16>(x, row, col + 4, cols, ld, vec_in, *reinterpret_cast<float(*)[4]>(&v[4]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float u = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
  const uint32_t code = cvt4_fp8(0, u, 0.0f, 0.0f, 0.0f) & 0xFFu;
  if (data) {
    const float sc = __fmul_rn(e4m3_value(code), g);
    uint32_t packed = 0;
    if (sc != 0.0f) {
      const GroupDiv div(sc);
#pragma unroll
      for (int j = 0; j < 4; ++j) packed |= cvt2_e2m1(div(v[2 * j]), div(v[2 * j + 1])) << (8 * j);
    }
    *reinterpret_cast<uint32_t*>(q + row * (cols / 2) + col / 2) = packed;
  }
  if ((lane & 1) == 0 && b < kb_pad) {
    const uint8_t c = data ? static_cast<uint8_t>(code) : static_cast<uint8_t>(0);
    if (kTC) {
      sf[sf_tc_offset(row, b, kb_pad / 4)] = c;
    } else if (data) {
      sf[row * kb + b] = c;
    }
  }
}

// FP4 with 16-bit block scales ("Rubin FP4 GEMM deep dive", section 3.2):
// one warp per (row, 256-column chunk = 8 blocks of 32); lane l owns 8
// elements, 4 lanes per block.  Per block: v = max / 6 (FP32 division, round
// to nearest), scale code = v rounded to nearest even in BF16 or FP16 (FP16
// saturates at 65504 instead of becoming Inf), s = the code's value (exact),
// elements E2M1(x / s) with a correctly rounded quotient; s = 0 stores zero
// codes.  Scales are written [K/32][rows].
template <bool kBF16, bool kF16Scale>
__global__ void __launch_bounds__(256) quantize_fp4_bs16_kernel(
    const void* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, bool vec_in,
    uint8_t* __restrict__ q, uint16_t* __restrict__ sf) {
  grid_dep_launch();
  grid_dep_wait();
  const int64_t kb = cols / 32;
  const int64_t chunks = (kb + 7) / 8;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (w >= rows * chunks) return;
  const int64_t row = w / chunks, chunk = w % chunks;
  const int lane = threadIdx.x & 31;
  const int64_t b = chunk * 8 + (lane >> 2);
  const int64_t col = b * 32 + (lane & 3) * 8;
  const bool data = b < kb;
  float v[8];
  if (data) {
    load4<kBF16>(x, row, col, cols, ld, vec_in, *reinterpret_cast<float(*)[4]>(&v[0]));
    load4<kBF16>(x, row, col + 4, cols, ld, vec_in, *reinterpret_cast<float(*)[4]>(&v[4]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float u = __fdiv_rn(amax, 6.0f);
  uint16_t code;
  float sc;
  if (kF16Scale) {
    code = __half_as_ushort(__float2half_rn(u));
    if (code == 0x7C00u) code = 0x7BFFu;          // satfinite: 65504, not Inf
    sc = __half2float(__ushort_as_half(code));
  } else {
    code = __bfloat16_as_ushort(__float2bfloat16_rn(u));
    sc = __uint_as_float(static_cast<uint32_t>(code) << 16);
  }
  if (!data) return;
  uint32_t packed = 0;
  if (sc != 0.0f) {
    const GroupDiv div(sc);
#pragma unroll
    for (int j = 0; j < 4; ++j) packed |= cvt2_e2m1(div(v[2 * j]), div(v[2 * j + 1])) << (8 * j);
  }
  *reinterpret_cast<uint32_t*>(q + row * (cols / 2) + col / 2) = packed;
  if ((lane & 3) == 0) sf[b * rows + row] = code;
}

__global__ void sf_to_tcgen05_kernel(const uint8_t* __restrict__ sf, int64_t rows, int64_t kb,
                                     int64_t total, uint8_t* __restrict__ out) {
  grid_dep_launch();
  grid_dep_wait();
  const int64_t off = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (off >= total) return;
  const int64_t groups = (kb + 3) / 4;
  const int64_t atom = off / 512, within = off % 512;
  const int64_t rb = atom / groups, cb = atom % groups;
  const int64_t r = rb * 128 + ((within % 16) / 4) * 32 + within / 16;
  const int64_t c = cb * 4 + within % 4;
  out[off] = (r < rows && c < kb) ? sf[r * kb + c] : static_cast<uint8_t>(127);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

cudaError_t quantize_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_quant_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_quant_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t launch_quantize_fp8_tile(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                     int64_t ld, int fmt, float fmt_max, uint8_t* q,
                                     float* scales, cudaStream_t s) {
  const bool vec_in = src_bf16 ? (aligned(x, 8) && ld % 4 == 0) : (aligned(x, 16) && ld % 4 == 0);
  const bool vec_out = aligned(q, 4) && cols % 4 == 0;
  dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>((rows + 127) / 128));
  auto kern = src_bf16 ? quantize_fp8_tile_kernel<true> : quantize_fp8_tile_kernel<false>;
  return launch_pdl(kern, grid, dim3(kTileThreads), 0, s, x, rows, cols, ld, fmt, fmt_max, vec_in,
                    vec_out, q, scales);
}

cudaError_t launch_quantize_fp8_row(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                    int64_t ld, int fmt, float fmt_max, uint8_t* q, float* scales,
                                    cudaStream_t s) {
  // 16-byte loads of a lane's 16 values (FP32: four, BF16: two) and one
  // 16-byte store of its codes, where alignment allows
  const bool vec_in = aligned(x, 16) && ld % (src_bf16 ? 8 : 4) == 0;
  const bool vec_out = aligned(q, 16) && cols % 16 == 0;
  // enough warps to fill the GPU once; each walks several chunks
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 1;
  const int64_t warps = rows * ((cols + 511) / 512);
  int64_t blocks = (warps + kRowWarps - 1) / kRowWarps;
  if (blocks > static_cast<int64_t>(sms) * 4) blocks = static_cast<int64_t>(sms) * 4;
  const dim3 grid(static_cast<unsigned>(blocks));
  auto kern = src_bf16 ? quantize_fp8_row_kernel<true> : quantize_fp8_row_kernel<false>;
  return launch_pdl(kern, grid, dim3(kRowWarps * 32), 0, s, x, rows, cols, ld, fmt, fmt_max,
                    vec_in, vec_out, q, scales);
}

cudaError_t launch_quantize_mx(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                               int64_t ld, int fmt, float fmt_max, uint8_t* q, uint8_t* sf,
                               bool tc_layout, cudaStream_t s) {
  const bool vec_in = src_bf16 ? (aligned(x, 8) && ld % 4 == 0) : (aligned(x, 16) && ld % 4 == 0);
  const int64_t kb = cols / 32;
  const int64_t kb_pad = tc_layout ? ((kb + 3) / 4) * 4 : kb;
  const int64_t rows_pad = tc_layout ? ((rows + 127) / 128) * 128 : rows;
  const int64_t warps = rows_pad * ((kb_pad + 7) / 8);
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  using K = void (*)(const void*, int64_t, int64_t, int64_t, float, bool, uint8_t*, uint8_t*);
  // [fmt][bf16][tc]
  static const K table[3][2][2] = {
      {{quantize_mx_kernel<false, false, 0>, quantize_mx_kernel<false, true, 0>},
       {quantize_mx_kernel<true, false, 0>, quantize_mx_kernel<true, true, 0>}},
      {{quantize_mx_kernel<false, false, 1>, quantize_mx_kernel<false, true, 1>},
       {quantize_mx_kernel<true, false, 1>, quantize_mx_kernel<true, true, 1>}},
      {{quantize_mx_kernel<false, false, 2>, quantize_mx_kernel<false, true, 2>},
       {quantize_mx_kernel<true, false, 2>, quantize_mx_kernel<true, true, 2>}}};
  if (fmt < 0 || fmt > 2) return cudaErrorInvalidValue;
  const K kern = table[fmt][src_bf16 ? 1 : 0][tc_layout ? 1 : 0];
  return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, x, rows, cols, ld, fmt_max, vec_in, q, sf);
}

cudaError_t launch_quantize_nvfp4(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                  int64_t ld, float tensor_scale, uint8_t* q, uint8_t* sf,
                                  bool tc_layout, cudaStream_t s) {
  const bool vec_in = src_bf16 ? (aligned(x, 8) && ld % 4 == 0) : (aligned(x, 16) && ld % 4 == 0);
  const int64_t kb = cols / 16;
  const int64_t kb_pad = tc_layout ? ((kb + 3) / 4) * 4 : kb;
  const int64_t rows_pad = tc_layout ? ((rows + 127) / 128) * 128 : rows;
  const int64_t warps = rows_pad * ((kb_pad + 15) / 16);
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  using K = void (*)(const void*, int64_t, int64_t, int64_t, float, bool, uint8_t*, uint8_t*);
  static const K table[2][2] = {{quantize_nvfp4_kernel<false, false>, quantize_nvfp4_kernel<false, true>},
                                {quantize_nvfp4_kernel<true, false>, quantize_nvfp4_kernel<true, true>}};
  const K kern = table[src_bf16 ? 1 : 0][tc_layout ? 1 : 0];
  return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, x, rows, cols, ld, tensor_scale, vec_in, q,
                    sf);
}

cudaError_t launch_quantize_fp4_bs16(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                     int64_t ld, bool f16_scales, uint8_t* q, uint16_t* sf,
                                     cudaStream_t s) {
  const bool vec_in = src_bf16 ? (aligned(x, 8) && ld % 4 == 0) : (aligned(x, 16) && ld % 4 == 0);
  const int64_t warps = rows * ((cols / 32 + 7) / 8);
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  using K = void (*)(const void*, int64_t, int64_t, int64_t, bool, uint8_t*, uint16_t*);
  static const K table[2][2] = {{quantize_fp4_bs16_kernel<false, false>, quantize_fp4_bs16_kernel<false, true>},
                                {quantize_fp4_bs16_kernel<true, false>, quantize_fp4_bs16_kernel<true, true>}};
  const K kern = table[src_bf16 ? 1 : 0][f16_scales ? 1 : 0];
  return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, x, rows, cols, ld, vec_in, q, sf);
}

cudaError_t launch_sf_to_tcgen05(const uint8_t* sf, int64_t rows, int64_t kblocks, uint8_t* out,
                                 cudaStream_t s) {
  const int64_t total = ((rows + 127) / 128) * ((kblocks + 3) / 4) * 512;
  return launch_pdl(sf_to_tcgen05_kernel, dim3(static_cast<unsigned>((total + 255) / 256)),
                    dim3(256), 0, s, sf, rows, kblocks, total, out);
}

}  // namespace bsg

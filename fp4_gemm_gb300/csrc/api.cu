// The C ABI of libbsg.so (declared in include/bsg.h): host-side validation,
// TMA descriptor encoding and dispatch to the kernels.  Nothing here
// allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bsg.h"
#include "kernels.h"

namespace {

using bsg::Fp8GemmArgs;
using bsg::Mxfp4GemmArgs;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bsg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA; }

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

bool is_fp8(bsg_format f) { return f == BSG_E4M3 || f == BSG_E5M2; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rows of the activation operand up to which E2M1 GEMMs take the
// decode-shaped path (weights streamed once, swap-AB, split-K).
constexpr int64_t kDecodeMaxM = 32;

// Longest bsg_mma_peak launch: 2^20 iterations of four MMAs run well under
// the kernels' 2 s wait limit at any clock above 1 GHz.
constexpr int64_t kMaxPeakIters = int64_t{1} << 20;

}  // namespace

namespace bsg {

bool make_kmajor_map(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                     uint64_t pitch, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_out_map(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols, int elem_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4)) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (cols * elem_bytes) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), 128};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return fn(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_kmajor_map_chunked(CUtensorMap* map, const void* base, uint64_t inner_bytes,
                             uint64_t rows, uint64_t pitch, uint32_t box_rows,
                             uint32_t box_chunks) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || inner_bytes % 128 != 0) return false;
  cuuint64_t dims[3] = {128, rows, inner_bytes / 128};
  cuuint64_t strides[2] = {pitch, 128};
  cuuint32_t box[3] = {128, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_fp4_unpack_map(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows,
                         uint64_t pitch, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || K % 128 != 0 || pitch % 32 != 0 ||
      reinterpret_cast<uintptr_t>(base) % 32 != 0)
    return false;
  cuuint64_t dims[2] = {K, rows};               // in 4-bit values
  cuuint64_t strides[1] = {pitch};              // bytes
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace bsg

using bsg::make_kmajor_map;

namespace {

void fill_fp8_args(Fp8GemmArgs* a, int64_t M, int64_t N, int64_t K, bsg_format fa, const void* sA,
                   bsg_scale_gran ga, bsg_format fb, const void* sB, bsg_scale_gran gb,
                   const float* C) {
  a->M = static_cast<int>(M);
  a->N = static_cast<int>(N);
  a->K = static_cast<int>(K);
  a->afmt = fa == BSG_E4M3 ? 0 : 1;
  a->bfmt = fb == BSG_E4M3 ? 0 : 1;
  a->sA = static_cast<const float*>(sA);
  a->a_row = ga == BSG_SCALE_ROW1x128;
  a->sB = static_cast<const float*>(sB);
  a->b_row = gb == BSG_SCALE_ROW1x128;
  a->C = C;
}

// Shape choice, tensor maps and launch of the promoted FP8 GEMM; D (a->D)
// is written by TMA stores when its base and row pitch allow.
bsg_status run_fp8(Fp8GemmArgs* a, const void* A, const void* B, int out_elem_bytes, int sms,
                   cudaStream_t s) {
  a->pair = bsg::gemm_fp8_use_pair(a->M, a->N, sms);
  a->tma_out = bsg::make_out_map(&a->tmD, a->D, static_cast<uint64_t>(a->M),
                                 static_cast<uint64_t>(a->N), out_elem_bytes);
  if (!make_kmajor_map(&a->tmA, A, a->K, a->M, a->K, 128) ||
      !make_kmajor_map(&a->tmB, B, a->K, a->N, a->K,
                       static_cast<uint32_t>(bsg::gemm_fp8_b_box_rows(a->pair))))
    return BSG_ERR_CUDA;
  return from_cuda(bsg::launch_gemm_fp8(*a, sms, s));
}

// The 128 x 256 block-scaled kernel for large FP4 problems (kind 1 MXFP4,
// 2 NVFP4); operands packed, K/2 bytes per row.
bsg_status run_fp4_large(int kind, float alpha, int64_t M, int64_t N, int64_t K, const void* A,
                         const void* sA, const void* B, const void* sB, const float* C, void* D,
                         bool out_bf16, int sms, cudaStream_t s) {
  bsg::MxGemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.kind = kind;
  a.alpha = alpha;
  a.sfA = static_cast<const uint8_t*>(sA);
  a.sfB = static_cast<const uint8_t*>(sB);
  a.C = C;
  a.D = D;
  a.out_bf16 = out_bf16;
  a.pair = bsg::gemm_mx_use_pair(a.M, a.N, sms);
  if (!make_kmajor_map(&a.tmA, A, K / 2, M, K / 2, 128) ||
      !make_kmajor_map(&a.tmB, B, K / 2, N, K / 2, static_cast<uint32_t>(bsg::gemm_mx_b_box_rows(a.pair))))
    return BSG_ERR_CUDA;
  return from_cuda(bsg::launch_gemm_mx(a, sms, s));
}

}  // namespace

extern "C" {

const char* bsg_status_string(bsg_status s) {
  switch (s) {
    case BSG_OK: return "BSG_OK";
    case BSG_ERR_INVALID_ARG: return "BSG_ERR_INVALID_ARG";
    case BSG_ERR_UNSUPPORTED: return "BSG_ERR_UNSUPPORTED";
    case BSG_ERR_ALIGNMENT: return "BSG_ERR_ALIGNMENT";
    case BSG_ERR_CUDA: return "BSG_ERR_CUDA";
    case BSG_ERR_TIMEOUT: return "BSG_ERR_TIMEOUT";
    case BSG_ERR_WORKSPACE: return "BSG_ERR_WORKSPACE";
  }
  return "BSG_ERR_UNKNOWN";
}

int bsg_num_sms(void) { return num_sms_current(); }

size_t bsg_scale_bytes(int64_t rows, int64_t cols, bsg_scale_gran gran, bsg_sf_layout layout) {
  if (rows <= 0 || cols <= 0) return 0;
  switch (gran) {
    case BSG_SCALE_TILE128x128:
      return static_cast<size_t>(cdiv(rows, 128) * cdiv(cols, 128)) * sizeof(float);
    case BSG_SCALE_ROW1x128:
      return static_cast<size_t>(rows * cdiv(cols, 128)) * sizeof(float);
    case BSG_SCALE_BLOCK1x32_E8M0:
      if (cols % 32) return 0;
      if (layout == BSG_SF_TCGEN05)
        return static_cast<size_t>(cdiv(rows, 128) * cdiv(cols / 32, 4) * 512);
      return static_cast<size_t>(rows * (cols / 32));
    case BSG_SCALE_BLOCK1x16_E4M3:
      if (cols % 16) return 0;
      if (layout == BSG_SF_TCGEN05)
        return static_cast<size_t>(cdiv(rows, 128) * cdiv(cols / 16, 4) * 512);
      return static_cast<size_t>(rows * (cols / 16));
    case BSG_SCALE_BLOCK1x32_BF16:
    case BSG_SCALE_BLOCK1x32_F16:
      if (cols % 32) return 0;
      return static_cast<size_t>((cols / 32) * rows) * sizeof(uint16_t);
  }
  return 0;
}

bsg_status bsg_quantize_fp8(const void* x, bsg_dtype src, int64_t rows, int64_t cols, int64_t ld,
                            bsg_format fmt, bsg_scale_gran gran, float fmt_max, uint8_t* q,
                            float* scales, void* stream) {
  if (x == nullptr || q == nullptr || scales == nullptr) return BSG_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols || rows > kMaxDim || cols > kMaxDim)
    return BSG_ERR_INVALID_ARG;
  if (src != BSG_F32 && src != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (!(fmt_max >= 0.0f) || !std::isfinite(fmt_max)) return BSG_ERR_INVALID_ARG;
  if (!is_fp8(fmt)) return BSG_ERR_UNSUPPORTED;
  if (gran != BSG_SCALE_TILE128x128 && gran != BSG_SCALE_ROW1x128) return BSG_ERR_UNSUPPORTED;
  if (!aligned(x, src == BSG_F32 ? 4 : 2) || !aligned(scales, 4)) return BSG_ERR_ALIGNMENT;
  if (gran == BSG_SCALE_TILE128x128 && cdiv(rows, 128) > 65535) return BSG_ERR_INVALID_ARG;
  if (gran == BSG_SCALE_ROW1x128 && cdiv(cdiv(cols, 128), 4) > 65535) return BSG_ERR_INVALID_ARG;
  const float fm = fmt_max == 0.0f ? (fmt == BSG_E4M3 ? 448.0f : 57344.0f) : fmt_max;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int f = fmt == BSG_E4M3 ? 0 : 1;
  if (gran == BSG_SCALE_TILE128x128)
    return from_cuda(bsg::launch_quantize_fp8_tile(x, src == BSG_BF16, rows, cols, ld, f, fm, q,
                                                   scales, s));
  return from_cuda(
      bsg::launch_quantize_fp8_row(x, src == BSG_BF16, rows, cols, ld, f, fm, q, scales, s));
}

bsg_status bsg_quantize_mx(const void* x, bsg_dtype src, int64_t rows, int64_t cols, int64_t ld,
                           bsg_format fmt, float fmt_max, uint8_t* q, uint8_t* sf,
                           bsg_sf_layout layout, void* stream) {
  if (x == nullptr || q == nullptr || sf == nullptr) return BSG_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols || rows > kMaxDim || cols > kMaxDim || cols % 32)
    return BSG_ERR_INVALID_ARG;
  if (src != BSG_F32 && src != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (layout != BSG_SF_ROWMAJOR && layout != BSG_SF_TCGEN05) return BSG_ERR_INVALID_ARG;
  if (!(fmt_max >= 0.0f) || !std::isfinite(fmt_max)) return BSG_ERR_INVALID_ARG;
  if (fmt != BSG_E4M3 && fmt != BSG_E5M2 && fmt != BSG_E2M1) return BSG_ERR_INVALID_ARG;
  if (!aligned(x, src == BSG_F32 ? 4 : 2) || !aligned(q, fmt == BSG_E2M1 ? 4 : 8))
    return BSG_ERR_ALIGNMENT;
  const float fm = fmt_max != 0.0f ? fmt_max
                                   : (fmt == BSG_E2M1 ? 6.0f : (fmt == BSG_E4M3 ? 448.0f : 57344.0f));
  const int f = fmt == BSG_E4M3 ? 0 : (fmt == BSG_E5M2 ? 1 : 2);
  return from_cuda(bsg::launch_quantize_mx(x, src == BSG_BF16, rows, cols, ld, f, fm, q, sf,
                                           layout == BSG_SF_TCGEN05,
                                           static_cast<cudaStream_t>(stream)));
}

bsg_status bsg_quantize_mxfp4(const void* x, bsg_dtype src, int64_t rows, int64_t cols,
                              int64_t ld, uint8_t* q_packed, uint8_t* sf, bsg_sf_layout layout,
                              void* stream) {
  return bsg_quantize_mx(x, src, rows, cols, ld, BSG_E2M1, 0.0f, q_packed, sf, layout, stream);
}

bsg_status bsg_sf_to_tcgen05(const uint8_t* sf_rowmajor, int64_t rows, int64_t kblocks,
                             uint8_t* sf_tc, void* stream) {
  if (sf_rowmajor == nullptr || sf_tc == nullptr || rows <= 0 || kblocks <= 0 ||
      rows > kMaxDim || kblocks > kMaxDim)
    return BSG_ERR_INVALID_ARG;
  return from_cuda(
      bsg::launch_sf_to_tcgen05(sf_rowmajor, rows, kblocks, sf_tc, static_cast<cudaStream_t>(stream)));
}

size_t bsg_gemm_workspace_size(int64_t M, int64_t N, int64_t K, bsg_format fa, bsg_format fb) {
  // sizes bsg_gemm would reject need no workspace (and must not reach the
  // int arithmetic of the plan)
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
  if (fa == BSG_E2M1 && fb == BSG_E2M1 && M <= kDecodeMaxM) {
    const int sms = num_sms_current();
    return bsg::gemm_mxfp4_decode_workspace(static_cast<int>(M), static_cast<int>(N),
                                            static_cast<int>(K), sms > 0 ? sms : 1);
  }
  return 0;
}


size_t bsg_gemm_mxfp4_act_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || K % 32) return 0;
  const int sms = num_sms_current();
  return bsg::gemm_mxfp4_act_workspace(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                       sms > 0 ? sms : 1, nullptr);
}

bsg_status bsg_gemm_mxfp4_act(int64_t M, int64_t N, int64_t K, const void* x, bsg_dtype src,
                              int64_t ldx, const void* B, const void* sB, const float* C, void* D,
                              bsg_dtype out, void* workspace, size_t workspace_bytes, void* stream) {
  if (x == nullptr || B == nullptr || sB == nullptr || D == nullptr) return BSG_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || K % 32 || ldx < K)
    return BSG_ERR_INVALID_ARG;
  if (src != BSG_F32 && src != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (out != BSG_F32 && out != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (!aligned(x, src == BSG_F32 ? 4 : 2) || !aligned(B, 16) || !aligned(sB, 16) ||
      !aligned(D, out == BSG_F32 ? 4 : 2) || (C != nullptr && !aligned(C, 4)))
    return BSG_ERR_ALIGNMENT;
  const int sms = num_sms_current();
  if (sms <= 0) return BSG_ERR_CUDA;
  size_t off[3];
  const size_t need = bsg::gemm_mxfp4_act_workspace(static_cast<int>(M), static_cast<int>(N),
                                                    static_cast<int>(K), sms, off);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16)))
    return BSG_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M > bsg::kActFusedMaxM) {
    // the stand-alone quantiser into the workspace, then the GEMM (with the
    // decode kernel's split-K area at the front of the workspace)
    uint8_t* xq = ws + off[1];
    uint8_t* xsf = ws + off[2];
    const bsg_status st = bsg_quantize_mxfp4(x, src, M, K, ldx, xq, xsf, BSG_SF_TCGEN05, stream);
    if (st != BSG_OK) return st;
    return bsg_gemm(M, N, K, xq, BSG_E2M1, xsf, BSG_SCALE_BLOCK1x32_E8M0, B, BSG_E2M1, sB,
                    BSG_SCALE_BLOCK1x32_E8M0, C, D, out, off[1] > 0 ? workspace : nullptr, off[1], stream);
  }
  Mxfp4GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.sfB = static_cast<const uint8_t*>(sB);
  a.C = C;
  a.D = D;
  a.out_bf16 = out == BSG_BF16;
  a.workspace = need > 0 ? workspace : nullptr;   // the split-K area, when the plan has one
  a.workspace_bytes = need;
  a.B = B;
  a.xsrc = x;
  a.ldx = ldx;
  a.xsrc_bf16 = src == BSG_BF16;
  return from_cuda(bsg::launch_gemm_mxfp4_decode(a, sms, s));
}

bsg_status bsg_gemm_quantized(int64_t M, int64_t N, int64_t K, const void* A, bsg_format fa,
                              const void* sA, bsg_scale_gran ga, const void* B, bsg_format fb,
                              const void* sB, bsg_scale_gran gb, const float* C, bsg_format qfmt,
                              float fmt_max, uint8_t* Dq, float* sD, void* stream) {
  if (A == nullptr || B == nullptr || sA == nullptr || sB == nullptr || Dq == nullptr ||
      sD == nullptr)
    return BSG_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return BSG_ERR_INVALID_ARG;
  if (!(fmt_max >= 0.0f) || !(fmt_max <= 0x1p64f)) return BSG_ERR_INVALID_ARG;
  if (fa < BSG_E4M3 || fa > BSG_E2M1 || fb < BSG_E4M3 || fb > BSG_E2M1) return BSG_ERR_INVALID_ARG;
  if (qfmt < BSG_E4M3 || qfmt > BSG_E2M1) return BSG_ERR_INVALID_ARG;
  if (!is_fp8(fa) || !is_fp8(fb) || !is_fp8(qfmt)) return BSG_ERR_UNSUPPORTED;
  if (ga != BSG_SCALE_TILE128x128 && ga != BSG_SCALE_ROW1x128) return BSG_ERR_UNSUPPORTED;
  if (gb != BSG_SCALE_TILE128x128 && gb != BSG_SCALE_ROW1x128) return BSG_ERR_UNSUPPORTED;
  if (K % 16) return BSG_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 4) || !aligned(sB, 4) || !aligned(sD, 4) ||
      (C != nullptr && !aligned(C, 4)))
    return BSG_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = num_sms_current();
  if (sms <= 0) return BSG_ERR_CUDA;
  Fp8GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  fill_fp8_args(&a, M, N, K, fa, sA, ga, fb, sB, gb, C);
  a.D = Dq;
  a.out_fp8 = true;
  a.qfmt = qfmt == BSG_E4M3 ? 0 : 1;
  a.qmax = fmt_max != 0.0f ? fmt_max : (qfmt == BSG_E4M3 ? 448.0f : 57344.0f);
  a.sD = sD;
  return run_fp8(&a, A, B, 1, sms, s);
}

bsg_status bsg_gemm(int64_t M, int64_t N, int64_t K, const void* A, bsg_format fa, const void* sA,
                    bsg_scale_gran ga, const void* B, bsg_format fb, const void* sB,
                    bsg_scale_gran gb, const float* C, void* D, bsg_dtype out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (A == nullptr || B == nullptr || sA == nullptr || sB == nullptr || D == nullptr)
    return BSG_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return BSG_ERR_INVALID_ARG;
  if (out != BSG_F32 && out != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (fa < BSG_E4M3 || fa > BSG_E2M1 || fb < BSG_E4M3 || fb > BSG_E2M1) return BSG_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16)) return BSG_ERR_ALIGNMENT;
  if (!aligned(D, out == BSG_F32 ? 4 : 2) || (C != nullptr && !aligned(C, 4)))
    return BSG_ERR_ALIGNMENT;
  const bool fp8 = is_fp8(fa) && is_fp8(fb);
  const bool fp4 = fa == BSG_E2M1 && fb == BSG_E2M1;
  if (!fp8 && !fp4) return BSG_ERR_UNSUPPORTED;
  // FP8 operands take FP32 per-tile scales (promoted FP8 GEMM) or, both of
  // them, E8M0 scales per 32 along K (MXFP8)
  const bool mx8 = fp8 && ga == BSG_SCALE_BLOCK1x32_E8M0 && gb == BSG_SCALE_BLOCK1x32_E8M0;
  if (mx8) {
    if (K % 32) return BSG_ERR_INVALID_ARG;
    if (!aligned(sA, 16) || !aligned(sB, 16)) return BSG_ERR_ALIGNMENT;
  } else if (fp8) {
    if (ga != BSG_SCALE_TILE128x128 && ga != BSG_SCALE_ROW1x128) return BSG_ERR_UNSUPPORTED;
    if (gb != BSG_SCALE_TILE128x128 && gb != BSG_SCALE_ROW1x128) return BSG_ERR_UNSUPPORTED;
    if (K % 16) return BSG_ERR_INVALID_ARG;
    if (!aligned(sA, 4) || !aligned(sB, 4)) return BSG_ERR_ALIGNMENT;
  } else {
    const bool mx = ga == BSG_SCALE_BLOCK1x32_E8M0 && gb == BSG_SCALE_BLOCK1x32_E8M0;
    const bool nv = ga == BSG_SCALE_BLOCK1x16_E4M3 && gb == BSG_SCALE_BLOCK1x16_E4M3;
    const bool bs16 = (ga == BSG_SCALE_BLOCK1x32_BF16 || ga == BSG_SCALE_BLOCK1x32_F16) && gb == ga;
    if (!mx && !nv && !bs16) return BSG_ERR_UNSUPPORTED;
    if (bs16) {
      // the unpacking tensor maps need K % 128 == 0 and 32-byte aligned rows
      if (K % 128) return BSG_ERR_INVALID_ARG;
      if (!aligned(A, 32) || !aligned(B, 32) || !aligned(sA, 2) || !aligned(sB, 2))
        return BSG_ERR_ALIGNMENT;
    } else {
      if (K % 32) return BSG_ERR_INVALID_ARG;
      if (!aligned(sA, 16) || !aligned(sB, 16)) return BSG_ERR_ALIGNMENT;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = num_sms_current();
  if (sms <= 0) return BSG_ERR_CUDA;

  if (mx8) {
    bsg::MxGemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.afmt = fa == BSG_E4M3 ? 0 : 1;
    a.bfmt = fb == BSG_E4M3 ? 0 : 1;
    a.sfA = static_cast<const uint8_t*>(sA);
    a.sfB = static_cast<const uint8_t*>(sB);
    a.C = C;
    a.D = D;
    a.out_bf16 = out == BSG_BF16;
    a.pair = bsg::gemm_mx_use_pair(a.M, a.N, sms);
    if (!make_kmajor_map(&a.tmA, A, K, M, K, 128) ||
        !make_kmajor_map(&a.tmB, B, K, N, K, static_cast<uint32_t>(bsg::gemm_mx_b_box_rows(a.pair))))
      return BSG_ERR_CUDA;
    return from_cuda(bsg::launch_gemm_mx(a, sms, s));
  }
  if (fp8) {
    Fp8GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_fp8_args(&a, M, N, K, fa, sA, ga, fb, sB, gb, C);
    a.D = D;
    a.out_bf16 = out == BSG_BF16;
    return run_fp8(&a, A, B, out == BSG_BF16 ? 2 : 4, sms, s);
  }
  if (ga == BSG_SCALE_BLOCK1x32_BF16 || ga == BSG_SCALE_BLOCK1x32_F16) {
    bsg::Bs16GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.f16_scales = ga == BSG_SCALE_BLOCK1x32_F16;
    a.sfA = static_cast<const uint16_t*>(sA);
    a.sfB = static_cast<const uint16_t*>(sB);
    a.C = C;
    a.D = D;
    a.out_bf16 = out == BSG_BF16;
    a.vec_out = aligned(D, 16) && N % (out == BSG_BF16 ? 8 : 4) == 0;
    if (!bsg::make_fp4_unpack_map(&a.tmA, A, K, M, K / 2, 128) ||
        !bsg::make_fp4_unpack_map(&a.tmB, B, K, N, K / 2,
                                  static_cast<uint32_t>(bsg::gemm_bs16_b_box_rows())))
      return BSG_ERR_CUDA;
    return from_cuda(bsg::launch_gemm_bs16(a, sms, s));
  }
  {
    Mxfp4GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.sfA = static_cast<const uint8_t*>(sA);
    a.sfB = static_cast<const uint8_t*>(sB);
    a.C = C;
    a.D = D;
    a.out_bf16 = out == BSG_BF16;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.A = A;
    a.B = B;
    // NVFP4 through this entry point: tensor scales are folded into alpha by
    // bsg_gemm_nvfp4, so alpha is 1 here
    const bool nv = ga == BSG_SCALE_BLOCK1x16_E4M3;
    a.nvfp4 = nv;
    a.alpha = 1.0f;
    if (M <= kDecodeMaxM) {
      const size_t need = bsg::gemm_mxfp4_decode_workspace(a.M, a.N, a.K, sms);
      if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16)))
        return BSG_ERR_WORKSPACE;
      // swap-AB: the weights (B, N rows) are the MMA's 128-row operand; the
      // launcher encodes its own tensor maps
      return from_cuda(bsg::launch_gemm_mxfp4_decode(a, sms, s));
    }
    if (bsg::gemm_mx_fp4_large(a.M, a.N, sms))
      return run_fp4_large(nv ? 2 : 1, 1.0f, M, N, K, A, sA, B, sB, C, D, out == BSG_BF16, sms, s);
    if (!make_kmajor_map(&a.tmA, A, K / 2, M, K / 2, 128) ||
        !make_kmajor_map(&a.tmB, B, K / 2, N, K / 2, 128))
      return BSG_ERR_CUDA;
    return from_cuda(bsg::launch_gemm_mxfp4(a, sms, s));
  }
}

bsg_status bsg_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const void* A, const void* sA,
                          const void* B, const void* sB, float alpha, const float* C, void* D,
                          bsg_dtype out, void* stream) {
  return bsg_gemm_nvfp4_ws(M, N, K, A, sA, B, sB, alpha, C, D, out, nullptr, 0, stream);
}

bsg_status bsg_gemm_nvfp4_ws(int64_t M, int64_t N, int64_t K, const void* A, const void* sA,
                             const void* B, const void* sB, float alpha, const float* C, void* D,
                             bsg_dtype out, void* workspace, size_t workspace_bytes, void* stream) {
  if (A == nullptr || B == nullptr || sA == nullptr || sB == nullptr || D == nullptr)
    return BSG_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || K % 32)
    return BSG_ERR_INVALID_ARG;
  if (out != BSG_F32 && out != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return BSG_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 16) || !aligned(sB, 16))
    return BSG_ERR_ALIGNMENT;
  if (!aligned(D, out == BSG_F32 ? 4 : 2) || (C != nullptr && !aligned(C, 4)))
    return BSG_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = num_sms_current();
  if (sms <= 0) return BSG_ERR_CUDA;
  Mxfp4GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.nvfp4 = true;
  a.alpha = alpha;
  a.sfA = static_cast<const uint8_t*>(sA);
  a.sfB = static_cast<const uint8_t*>(sB);
  a.C = C;
  a.D = D;
  a.out_bf16 = out == BSG_BF16;
  a.A = A;
  a.B = B;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  if (M <= kDecodeMaxM) {
    // the decode-shaped kernel (weights streamed once, split over all SMs)
    // when its split-K workspace is given or not needed; without a
    // workspace the general kernel below serves the call
    const size_t need = bsg::gemm_mxfp4_decode_workspace(a.M, a.N, a.K, sms);
    const bool have = workspace != nullptr && workspace_bytes >= need && aligned(workspace, 16);
    if (need == 0 || have) return from_cuda(bsg::launch_gemm_mxfp4_decode(a, sms, s));
    if (workspace != nullptr) return BSG_ERR_WORKSPACE;
  }
  if (bsg::gemm_mx_fp4_large(static_cast<int>(M), static_cast<int>(N), sms))
    return run_fp4_large(2, alpha, M, N, K, A, sA, B, sB, C, D, out == BSG_BF16, sms, s);
  if (!make_kmajor_map(&a.tmA, A, K / 2, M, K / 2, 128) ||
      !make_kmajor_map(&a.tmB, B, K / 2, N, K / 2, 128))
    return BSG_ERR_CUDA;
  return from_cuda(bsg::launch_gemm_mxfp4(a, sms, s));
}

bsg_status bsg_quantize_nvfp4(const void* x, bsg_dtype src, int64_t rows, int64_t cols, int64_t ld,
                              float tensor_scale, uint8_t* q_packed, uint8_t* sf,
                              bsg_sf_layout layout, void* stream) {
  if (x == nullptr || q_packed == nullptr || sf == nullptr) return BSG_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols || rows > kMaxDim || cols > kMaxDim || cols % 16)
    return BSG_ERR_INVALID_ARG;
  if (src != BSG_F32 && src != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (layout != BSG_SF_ROWMAJOR && layout != BSG_SF_TCGEN05) return BSG_ERR_INVALID_ARG;
  if (!(tensor_scale >= 0x1p-126f) || !std::isfinite(tensor_scale)) return BSG_ERR_INVALID_ARG;
  if (!aligned(x, src == BSG_F32 ? 4 : 2) || !aligned(q_packed, 4)) return BSG_ERR_ALIGNMENT;
  return from_cuda(bsg::launch_quantize_nvfp4(x, src == BSG_BF16, rows, cols, ld, tensor_scale,
                                              q_packed, sf, layout == BSG_SF_TCGEN05,
                                              static_cast<cudaStream_t>(stream)));
}

bsg_status bsg_check_wait_timeout(void* stream) {
  return from_cuda(bsg::launch_wait_timeout_check(static_cast<cudaStream_t>(stream)));
}

bsg_status bsg_mma_probe_mx(int kind, const uint8_t* A, const uint8_t* sfA, const uint8_t* B,
                           const uint8_t* sfB, const float* C, float* D, bsg_format fa,
                           bsg_format fb, void* stream) {
  if (A == nullptr || sfA == nullptr || B == nullptr || sfB == nullptr || C == nullptr ||
      D == nullptr || kind < 0 || kind > 2)
    return BSG_ERR_INVALID_ARG;
  if (kind == 0 && (!is_fp8(fa) || !is_fp8(fb))) return BSG_ERR_UNSUPPORTED;
  if (!aligned(sfA, 4) || !aligned(sfB, 4) || !aligned(C, 4) || !aligned(D, 4))
    return BSG_ERR_ALIGNMENT;
  return from_cuda(bsg::launch_mma_probe_mx(kind, A, sfA, B, sfB, C, D, fa == BSG_E5M2 ? 1 : 0,
                                            fb == BSG_E5M2 ? 1 : 0, static_cast<cudaStream_t>(stream)));
}

bsg_status bsg_quantize_fp4_bs16(const void* x, bsg_dtype src, int64_t rows, int64_t cols,
                                 int64_t ld, bsg_scale_gran gran, uint8_t* q_packed, uint16_t* sf,
                                 void* stream) {
  if (x == nullptr || q_packed == nullptr || sf == nullptr) return BSG_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols || rows > kMaxDim || cols > kMaxDim || cols % 32)
    return BSG_ERR_INVALID_ARG;
  if (src != BSG_F32 && src != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (gran != BSG_SCALE_BLOCK1x32_BF16 && gran != BSG_SCALE_BLOCK1x32_F16) return BSG_ERR_UNSUPPORTED;
  if (!aligned(x, src == BSG_F32 ? 4 : 2) || !aligned(q_packed, 4) || !aligned(sf, 2))
    return BSG_ERR_ALIGNMENT;
  return from_cuda(bsg::launch_quantize_fp4_bs16(x, src == BSG_BF16, rows, cols, ld,
                                                 gran == BSG_SCALE_BLOCK1x32_F16, q_packed, sf,
                                                 static_cast<cudaStream_t>(stream)));
}

bsg_status bsg_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSG_ERR_CUDA;
  uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0, w4 = 0, w5 = 0, w6 = 0, w7 = 0;
  if (bsg::quantize_error_read_and_clear(s, &w0) != cudaSuccess ||
      bsg::gemm_fp8_error_read_and_clear(s, &w1) != cudaSuccess ||
      bsg::gemm_mxfp4_error_read_and_clear(s, &w2) != cudaSuccess ||
      bsg::mma_peak_error_read_and_clear(s, &w3) != cudaSuccess ||
      bsg::gemm_mx_error_read_and_clear(s, &w4) != cudaSuccess ||
      bsg::mma_probe_error_read_and_clear(s, &w5) != cudaSuccess ||
      bsg::watchdog_error_read_and_clear(s, &w6) != cudaSuccess ||
      bsg::gemm_bs16_error_read_and_clear(s, &w7) != cudaSuccess)
    return BSG_ERR_CUDA;
  const uint32_t w = w0 | w1 | w2 | w3 | w4 | w5 | w6 | w7;
  if (w & 1u) return BSG_ERR_TIMEOUT;
  if (w & 2u) return BSG_ERR_WORKSPACE;
  return BSG_OK;
}

bsg_status bsg_mma_peak(bsg_format fmt, int block_scaled, int pair, int64_t iters, int64_t* flops,
                        void* stream) {
  if (flops == nullptr || iters <= 0 || iters > kMaxPeakIters) return BSG_ERR_INVALID_ARG;
  int kind;
  if (fmt == BSG_E4M3)
    kind = block_scaled ? 1 : 0;
  else if (fmt == BSG_E2M1 && block_scaled)
    kind = 2;
  else
    return BSG_ERR_UNSUPPORTED;
  if (kind == 1 && pair) return BSG_ERR_UNSUPPORTED;
  const int sms = num_sms_current();
  if (sms <= 0 || (pair && sms < 2)) return BSG_ERR_CUDA;
  return from_cuda(bsg::launch_mma_peak(kind, pair != 0, iters, sms,
                                        static_cast<cudaStream_t>(stream), flops));
}

bsg_status bsg_mma_probe(const uint8_t* A, bsg_format fa, const uint8_t* B, bsg_format fb,
                         const float* C, float* D, void* stream) {
  if (A == nullptr || B == nullptr || C == nullptr || D == nullptr) return BSG_ERR_INVALID_ARG;
  if (!is_fp8(fa) || !is_fp8(fb)) return BSG_ERR_UNSUPPORTED;
  if (!aligned(C, 4) || !aligned(D, 4)) return BSG_ERR_ALIGNMENT;
  return from_cuda(bsg::launch_mma_probe(A, fa == BSG_E4M3 ? 0 : 1, B, fb == BSG_E4M3 ? 0 : 1, C, D,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

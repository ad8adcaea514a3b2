// Tensor-core throughput microbenchmark: the dense FP8, block-scaled FP8 and
// block-scaled FP4 rates of tcgen05.mma on this GPU, at whatever clock it
// runs at.
//
// The GEMM kernels of this library are reported against a peak.  The FP8 and
// FP4 peaks of GB300 are not given by any measured copy or library GEMM on
// the box, so this kernel measures them: every CTA (one per SM, or one per
// SM of a CTA pair) keeps its tensor core busy with back-to-back MMAs whose
// operands already sit in shared memory - no global traffic, no epilogue.
//   FP8:  tcgen05.mma kind::f8f6f4, E4M3 x E4M3, M128 N256 K32 per
//         instruction (M256 for a CTA pair, cta_group::2).
//   MXFP8: tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X, E4M3 x E4M3
//         with UE8M0 scales, M128 N256 K32 per instruction.
//   FP4:  tcgen05.mma kind::mxf4.block_scale.scale_vec::2X, E2M1 x E2M1 with
//         UE8M0 scales, M128 N256 K64 per instruction (M256 for a pair).
// The operand tiles are zero-filled; scales are whatever tensor memory holds.
// Results are discarded: only the time matters.
#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_peak_error = 0;

constexpr int kPeakThreads = 128;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;           // N = 256 FP32 accumulator columns
constexpr int kSfaCol = 256;            // scale columns (block-scaled kinds)
constexpr int kSfbCol = 288;
// Dynamic shared memory requested per CTA: large enough that only one CTA
// fits on an SM, so each SM's tensor memory has a single owner.
constexpr size_t kPeakSmem = 150 * 1024;

// kKind: 0 dense FP8, 1 block-scaled FP8 (MXFP8), 2 block-scaled FP4 (MXFP4)
template <bool kPair, int kKind>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int64_t iters) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kBRows = kPair ? 128 : 256;     // a pair splits N = 256 across its CTAs
  uint8_t* a = base;                            // 128 rows x 128 B
  uint8_t* b = base + 128 * 128;                // kBRows x 128 B
  uint64_t* bar = reinterpret_cast<uint64_t*>(b + kBRows * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;

  // zero the operand tiles (generic proxy) and make them visible to the
  // tensor core (async proxy)
  for (int i = threadIdx.x; i < (128 + kBRows) * 128 / 16; i += kPeakThreads)
    reinterpret_cast<uint4*>(a)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_barrier_init();
  }
  if (warp_id() == 0) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0 && rank == 0) {
    const uint64_t ad = sdesc_kmajor_sw128(smem_u32(a));
    const uint64_t bd = sdesc_kmajor_sw128(smem_u32(b));
    constexpr uint32_t M = kPair ? 256 : 128;
    const uint32_t id = kKind == 2   ? idesc_mxf4(M, kAccCols, 0, 0)
                        : kKind == 1 ? idesc_mxf8(0, 0, M, kAccCols, 0, 0)
                                     : idesc_f8f6f4(0, 0, M, kAccCols);
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        if (kKind == 2) {
          if (kPair)
            mma_mxf4_pair(tmem, ad + 2 * kk, bd + 2 * kk, id, tmem + kSfaCol, tmem + kSfbCol, acc);
          else
            mma_mxf4(tmem, ad + 2 * kk, bd + 2 * kk, id, tmem + kSfaCol, tmem + kSfbCol, acc);
        } else if (kKind == 1) {
          mma_mxf8(tmem, ad + 2 * kk, bd + 2 * kk, id, tmem + kSfaCol, tmem + kSfbCol, acc);
        } else {
          if (kPair)
            mma_f8f6f4_pair(tmem, ad + 2 * kk, bd + 2 * kk, id, acc);
          else
            mma_f8f6f4(tmem, ad + 2 * kk, bd + 2 * kk, id, acc);
        }
      }
    }
    if (kPair)
      tc_commit_pair(smem_u32(bar));
    else
      tc_commit(smem_u32(bar));
    if (!mbar_wait(smem_u32(bar), 0)) atomicOr(&g_peak_error, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();    // the peer's operands and tensor memory stay until the MMAs end
  if (warp_id() == 0) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
  if (kPair) cluster_sync();
}

template <bool kPair, int kKind>
cudaError_t launch_peak(int64_t iters, int num_sms, cudaStream_t s, int64_t* flops) {
  constexpr bool kFp4 = kKind == 2;
  auto kern = mma_peak_kernel<kPair, kKind>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kPeakSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPeakThreads);
  cfg.dynamicSmemBytes = kPeakSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int units = num_sms / (kPair ? 2 : 1);
  if (kPair) {
    cfg.gridDim = dim3(static_cast<unsigned>(2 * units));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0 && n < units)
      units = n;
  }
  cfg.gridDim = dim3(static_cast<unsigned>((kPair ? 2 : 1) * units));
  const int64_t m = kPair ? 256 : 128;
  const int64_t k = kFp4 ? 64 : 32;
  *flops = static_cast<int64_t>(units) * iters * 4 * 2 * m * kAccCols * k;
  return cudaLaunchKernelEx(&cfg, kern, iters);
}

}  // namespace

cudaError_t mma_peak_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_peak_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_peak_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t launch_mma_peak(int kind, bool pair, int64_t iters, int num_sms, cudaStream_t s,
                            int64_t* flops) {
  switch (kind) {
    case 0: return pair ? launch_peak<true, 0>(iters, num_sms, s, flops)
                        : launch_peak<false, 0>(iters, num_sms, s, flops);
    case 1: return launch_peak<false, 1>(iters, num_sms, s, flops);
    default: return pair ? launch_peak<true, 2>(iters, num_sms, s, flops)
                         : launch_peak<false, 2>(iters, num_sms, s, flops);
  }
}

}  // namespace bsg

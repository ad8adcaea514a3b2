// One tcgen05.mma on given operands, for characterising the tensor core's
// arithmetic bit by bit.
//
// "FP8 MMA internals on Hopper" shows that one FP8 MMA instruction on H100
// does not return the exact dot product: it aligns the products and the
// accumulator to the largest exponent, truncates what falls more than 13
// bits below it and rounds the sum toward zero with 13 fraction bits, and the
// page gives two test vectors with the bits H100 returns.  "Exact models of
// AMD matrix cores" (section 3) builds such models from test vectors plus
// large random campaigns.  This kernel is the measuring instrument for the
// same question on GB300: it runs exactly one
//   D[128][16] = A[128][32] . B[16][32]^T + C[128][16]
// tcgen05.mma kind::f8f6f4 (M128 N16 K32, FP32 accumulate) and returns D.
// One CTA of 128 threads; the operands go to shared memory in the K-major,
// 128-byte-swizzled layout the MMA descriptor describes (plain stores, no
// TMA), the accumulator C to tensor memory with tcgen05.st.
#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_probe_error = 0;

constexpr int PM = 128;
constexpr int PN = 16;
constexpr int PK = 32;

// Byte offset of element (r, k) of a K-major tile with 128-byte rows in the
// 128-byte swizzle: 8-row atoms of 1024 bytes, the 16-byte chunk index of a
// row XORed with the row's index inside its atom.
__device__ __forceinline__ int swz128(int r, int k) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 4) ^ (r & 7)) & 7) << 4) + (k & 15);
}

__global__ void __launch_bounds__(128, 1)
    mma_probe_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                     const float* __restrict__ C, float* __restrict__ D, uint32_t idesc) {
  __shared__ __align__(1024) uint8_t sa[PM * 128];
  __shared__ __align__(1024) uint8_t sb[PN * 128];
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  for (int i = threadIdx.x; i < PM * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sa)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < PN * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sb)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  for (int i = threadIdx.x; i < PM * PK; i += blockDim.x) sa[swz128(i / PK, i % PK)] = A[i];
  for (int i = threadIdx.x; i < PN * PK; i += blockDim.x) sb[swz128(i / PK, i % PK)] = B[i];
  fence_proxy_async_smem();   // the operands are read by the tensor core (async proxy)
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const int row = warp * 32 + lane;               // TMEM lane = row of D
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  uint32_t c[16];
#pragma unroll
  for (int j = 0; j < PN; ++j) c[j] = __float_as_uint(C[row * PN + j]);
  tmem_st_16(taddr, c);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    mma_f8f6f4(tmem, sdesc_kmajor_sw128(smem_u32(sa)), sdesc_kmajor_sw128(smem_u32(sb)), idesc, 1u);
    tc_commit(smem_u32(&bar));
  }
  if (!mbar_wait(smem_u32(&bar), 0)) atomicOr(&g_probe_error, kErrTimeout);
  tc_fence_after();
  uint32_t d[16];
  tmem_ld_16(taddr, d);
  tc_wait_ld_16(d);
#pragma unroll
  for (int j = 0; j < PN; ++j) D[row * PN + j] = __uint_as_float(d[j]);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

// The block-scaled kinds, one MMA of the GEMMs' own shape (M128 N256) and
// scale layout: D[128][256] = sum over the instruction's K of
// (sA a)(sB b) + C, with the scale bytes given per row as the four bytes of
// the row's tensor-memory scale cell (kind 0: kind::mxf8f6f4 scale_vec::1X,
// K = 32, byte 0; kind 1: kind::mxf4 scale_vec::2X, K = 64, bytes 0-1;
// kind 2: kind::mxf4nvf4 scale_vec::4X, K = 64, UE4M3 bytes 0-3).  A row's
// 32 operand bytes (32 FP8 values or 64 packed E2M1) are given as they sit in
// shared memory.
constexpr int XN = 256;
constexpr uint32_t kXScaleA = 256;       // scale columns after the accumulator
constexpr uint32_t kXScaleB = 264;       // B's two 128-row blocks: +0..3 and +4..7

__global__ void __launch_bounds__(128, 1)
    mma_probe_mx_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ sfA,
                        const uint8_t* __restrict__ B, const uint8_t* __restrict__ sfB,
                        const float* __restrict__ C, float* __restrict__ D, int kind, uint32_t idesc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sb = sa + PM * 128;
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  for (int i = threadIdx.x; i < (PM + XN) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sa)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  for (int i = threadIdx.x; i < PM * 32; i += blockDim.x) sa[swz128(i / 32, i % 32)] = A[i];
  for (int i = threadIdx.x; i < XN * 32; i += blockDim.x) sb[swz128(i / 32, i % 32)] = B[i];
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  // the accumulator: this warp's 32 rows x 256 columns of C
  const int row = warp * 32 + lane;
  for (int c0 = 0; c0 < XN; c0 += 16) {
    uint32_t c[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = __float_as_uint(C[row * XN + c0 + j]);
    tmem_st_16(tmem + lane_off + c0, c);
  }
  // scale cells in the atom layout the GEMMs use: lane 32q + i, column k
  // holds the four bytes of row i + 32 k (the same in every lane quarter)
  uint4 wa, wb0, wb1;
  const uint32_t* fa = reinterpret_cast<const uint32_t*>(sfA);
  const uint32_t* fb = reinterpret_cast<const uint32_t*>(sfB);
  wa = make_uint4(fa[lane], fa[lane + 32], fa[lane + 64], fa[lane + 96]);
  wb0 = make_uint4(fb[lane], fb[lane + 32], fb[lane + 64], fb[lane + 96]);
  wb1 = make_uint4(fb[128 + lane], fb[128 + lane + 32], fb[128 + lane + 64], fb[128 + lane + 96]);
  tmem_st_4(tmem + lane_off + kXScaleA, wa);
  tmem_st_4(tmem + lane_off + kXScaleB, wb0);
  tmem_st_4(tmem + lane_off + kXScaleB + 4, wb1);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sa)), bd = sdesc_kmajor_sw128(smem_u32(sb));
    if (kind == 0)
      mma_mxf8(tmem, ad, bd, idesc, tmem + kXScaleA, tmem + kXScaleB, 1u);
    else if (kind == 1)
      mma_mxf4(tmem, ad, bd, idesc, tmem + kXScaleA, tmem + kXScaleB, 1u);
    else
      mma_nvf4(tmem, ad, bd, idesc, tmem + kXScaleA, tmem + kXScaleB, 1u);
    tc_commit(smem_u32(&bar));
  }
  if (!mbar_wait(smem_u32(&bar), 0)) atomicOr(&g_probe_error, kErrTimeout);
  tc_fence_after();
  for (int c0 = 0; c0 < XN; c0 += 16) {
    uint32_t d[16];
    tmem_ld_16(tmem + lane_off + c0, d);
    tc_wait_ld_16(d);
#pragma unroll
    for (int j = 0; j < 16; ++j) D[row * XN + c0 + j] = __uint_as_float(d[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_mma_probe_mx(int kind, const uint8_t* A, const uint8_t* sfA, const uint8_t* B,
                                const uint8_t* sfB, const float* C, float* D, int afmt, int bfmt,
                                cudaStream_t s) {
  uint32_t idesc;
  if (kind == 0)
    idesc = idesc_mxf8(static_cast<uint32_t>(afmt), static_cast<uint32_t>(bfmt), PM, XN, 0u, 0u);
  else if (kind == 1)
    idesc = idesc_mxf4(PM, XN, 0u, 0u);
  else
    idesc = idesc_nvf4(PM, XN);
  const size_t smem = (PM + XN) * 128 + 1024;
  cudaError_t e = cudaFuncSetAttribute(mma_probe_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  mma_probe_mx_kernel<<<1, 128, smem, s>>>(A, sfA, B, sfB, C, D, kind, idesc);
  return cudaGetLastError();
}

cudaError_t mma_probe_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_probe_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_probe_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t launch_mma_probe(const uint8_t* A, int afmt, const uint8_t* B, int bfmt, const float* C,
                             float* D, cudaStream_t s) {
  const uint32_t idesc = idesc_f8f6f4(static_cast<uint32_t>(afmt), static_cast<uint32_t>(bfmt), PM, PN);
  mma_probe_kernel<<<1, 128, 0, s>>>(A, B, C, D, idesc);
  return cudaGetLastError();
}

}  // namespace bsg

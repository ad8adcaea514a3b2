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

}  // namespace

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

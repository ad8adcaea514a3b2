// Self-check of the kernels' failure detection.
//
// Every mbarrier wait in the library is bounded (kWaitLimitNs of
// %globaltimer): a wait that runs out sets its translation unit's error word,
// which the host reads with bsg_device_error, and the kernel unwinds instead
// of hanging or trapping.  This kernel waits, with the same bounded wait, on
// a barrier that nothing ever arrives on, so a caller (a test, or a health
// check at start-up) can see the limit end the wait and the status come back
// while the context stays usable.
#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_watchdog_error = 0;

__global__ void wait_timeout_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // no thread ever arrives: phase 0 never completes, the wait runs out
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0)) atomicOr(&g_watchdog_error, kErrTimeout);
}

}  // namespace

cudaError_t watchdog_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_watchdog_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_watchdog_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t launch_wait_timeout_check(cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

}  // namespace bsg

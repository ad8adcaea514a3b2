// bsg_gemm_decode_noalloc: the decode-shaped MXFP4 GEMM for callers that
// cannot allocate device memory.
//
// The decode path splits K across CTAs and needs scratch memory for its
// partial sums and per-tile counters.  bsg_gemm takes that scratch from the
// caller.  Some callers have no way to provide it: a plug-in that a serving
// runtime hands only its input and output buffers, or a loop that has to keep
// cudaMalloc (which can synchronise the device and can fail under memory
// pressure) out of its steady state.  This entry point uses a fixed scratch
// array that lives in the library's own device image instead, so a call
// allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoallocScratchBytes of it until the process exits.  Host
// code cannot use the variable's name as a device address, so the address is
// fetched with cudaGetSymbolAddress, once per device, with that device
// current, on the first call made on it.  The address is kept for the life
// of the process: a cudaDeviceReset (or any teardown of the device's primary
// context) after that first call is not supported, since the kept address
// would then point into a context that no longer exists.
#include <mutex>

#include "bsg.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t{8} << 20;  // 8 MiB
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (nullptr on
// failure).  The first call on a device does the lookup.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" bsg_status bsg_gemm_decode_noalloc(int64_t M, int64_t N, int64_t K, const void* A,
                                              const void* sA, const void* B, const void* sB,
                                              const float* C, void* D, bsg_dtype out,
                                              void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return BSG_ERR_INVALID_ARG;
  if (M > 32) return BSG_ERR_UNSUPPORTED;
  const size_t need = bsg_gemm_workspace_size(M, N, K, BSG_E2M1, BSG_E2M1);
  if (need > kNoallocScratchBytes) return BSG_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (scratch == nullptr) return BSG_ERR_CUDA;
    // The split-K scratch is the partial-sum slots followed by one 32-bit
    // counter per 128-row weight tile.  Only the counters must start at zero:
    // a tile's partials are summed once its counter shows that every
    // contributor of this call has written its slot, so a slot is never read
    // before this call wrote it, whatever an earlier call (even one that
    // stopped early) left there.
    const size_t counter_bytes = static_cast<size_t>((N + 127) / 128) * sizeof(uint32_t);
    if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - counter_bytes), 0,
                        counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return BSG_ERR_CUDA;
  }
  return bsg_gemm(M, N, K, A, BSG_E2M1, sA, BSG_SCALE_BLOCK1x32_E8M0, B, BSG_E2M1, sB,
                  BSG_SCALE_BLOCK1x32_E8M0, C, D, out, scratch, need, stream);
}

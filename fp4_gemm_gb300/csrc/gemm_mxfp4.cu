// MXFP4 block-scaled GEMMs for sm_103a.
//
//   D[i][j] = sum_k (2^eA(i,k/32) a[i][k]) (2^eB(j,k/32) b[j][k]) + C[i][j]
//
// "Rubin FP4 GEMM deep dive", sections 2.2 and 3.1: 32 consecutive K elements
// share one E8M0 scale, so every K block's partial sum is scaled by
// 2^(eA+eB) before it is accumulated.  The tensor core does exactly that:
// tcgen05.mma kind::mxf4.block_scale reads E2M1 operands (packed, two per
// byte) from shared memory and one UE8M0 scale per 32 K per row from tensor
// memory, and accumulates in FP32 tensor memory across all of K.  No
// promotion step is needed because the scales are powers of two.
//
// Scale factors arrive in the BSG_SF_TCGEN05 atom layout (512 bytes per
// 128 rows x 4 K-blocks), are bulk-copied to shared memory with the operands
// and moved to tensor memory with tcgen05.cp.32x128b.warpx4 right before the
// MMAs that use them (copy and MMA issued by one thread execute in order).
// Each pipeline stage owns its own tensor-memory scale columns, so a copy
// never overwrites scales an in-flight MMA still reads.
//
// Two kernels:
//  * gemm_mxfp4_kernel: 128 x 128 output tiles, persistent, warp-specialised
//    (TMA producer warp, MMA warp, 8 epilogue warps draining a double-
//    buffered accumulator).
//  * gemm_mxfp4_decode_kernel: decode shapes (M <= 32 activation rows).  The
//    weights are the MMA's 128-row operand and the activations its N = 16/32
//    operand ("swap AB"), so the weight matrix streams from HBM exactly once.
//    Work is split evenly over all SMs in units of (128 weight rows, 256 K);
//    a CTA whose range covers only part of a tile's K writes an FP32 partial
//    to the workspace, and the last contributor (per-tile counter) adds the
//    partials in a fixed order, so results are deterministic.
#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_mxfp4_error = 0;

constexpr int kRowBytes = 128;          // packed bytes per row per stage = 256 FP4 values
constexpr int kSfAtom = 512;            // 128 rows x 4 K-blocks of E8M0
constexpr int kThreads = 320;

__device__ __forceinline__ void raise_abort(volatile uint32_t* flag) {
  atomicOr(&g_mxfp4_error, kErrTimeout);
  *flag = 1u;
}

// ------------------------------------------------------------ general GEMM
namespace general {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kStages = 5;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr int kSfColsPerStage = 16;     // SFA: 2 atoms x 4 cols, SFB: 2 atoms x 4 cols
constexpr int kSfBase = 2 * BN;         // after the two accumulators
constexpr int kGroupM = 8;

struct __align__(1024) Smem {
  uint8_t a[kStages][BM * kRowBytes];
  uint8_t b[kStages][BN * kRowBytes];
  uint8_t sfa[kStages][2 * kSfAtom];
  uint8_t sfb[kStages][2 * kSfAtom];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
};

__device__ __forceinline__ void tile_coord(int t, int num_m, int num_n, int& m, int& n) {
  const int group_size = kGroupM * num_n;
  const int group = t / group_size;
  const int first_m = group * kGroupM;
  const int gsz = min(num_m - first_m, kGroupM);
  const int local = t % group_size;
  m = first_m + local % gsz;
  n = local / gsz;
}

template <bool kBF16Out>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxfp4_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const uint8_t* __restrict__ sfA,
                      const uint8_t* __restrict__ sfB, const float* __restrict__ Cin,
                      void* __restrict__ Dout, int M, int N, int K, bool vec_out) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int kbytes = K / 2;
  const int KS = (kbytes + kRowBytes - 1) / kRowBytes;   // stages of 256 K
  const int KA = (K / 32 + 3) / 4;                       // scale atoms along K

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.tfull[b]), 1);
      mbar_init(smem_u32(&sm.tempty[b]), 8);
    }
    mbar_init(smem_u32(&sm.final_bar), 1);
    sm.abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        int m, n;
        tile_coord(t, num_m, num_n, m, n);
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = static_cast<int>(it % kStages);
          const uint32_t ph = (it / kStages) & 1u;
          if (sm.abort_flag) { ok = false; break; }
          if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1u)) {
            raise_abort(&sm.abort_flag);
            ok = false;
            break;
          }
          const int ka0 = 2 * ks;
          const int na = min(2, KA - ka0);
          const uint32_t fb = smem_u32(&sm.full[s]);
          mbar_arrive_expect_tx(fb, (BM + BN) * kRowBytes + 2 * na * kSfAtom);
          tma_load_2d(smem_u32(sm.a[s]), &tmA, fb, ks * kRowBytes, m * BM);
          tma_load_2d(smem_u32(sm.b[s]), &tmB, fb, ks * kRowBytes, n * BN);
          bulk_load(smem_u32(sm.sfa[s]), sfA + (static_cast<int64_t>(m) * KA + ka0) * kSfAtom,
                    na * kSfAtom, fb);
          bulk_load(smem_u32(sm.sfb[s]), sfB + (static_cast<int64_t>(n) * KA + ka0) * kSfAtom,
                    na * kSfAtom, fb);
        }
      }
      drain_fills(sm.full, kStages, it);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tl) {
        const uint32_t buf = tl & 1u;
        if (!mbar_wait(smem_u32(&sm.tempty[buf]), ((tl >> 1) & 1u) ^ 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = static_cast<int>(it % kStages);
          const uint32_t ph = (it / kStages) & 1u;
          if (sm.abort_flag) { ok = false; break; }
          if (!mbar_wait(smem_u32(&sm.full[s]), ph)) {
            raise_abort(&sm.abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const int ka0 = 2 * ks;
          const int na = min(2, KA - ka0);
          const uint32_t sfc = tmem + kSfBase + s * kSfColsPerStage;
          for (int a = 0; a < na; ++a) {
            tc_cp_32x128b_warpx4(sfc + 4 * a, sdesc_sf_32x16(smem_u32(sm.sfa[s] + a * kSfAtom)));
            tc_cp_32x128b_warpx4(sfc + 8 + 4 * a, sdesc_sf_32x16(smem_u32(sm.sfb[s] + a * kSfAtom)));
          }
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm.a[s]));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sm.b[s]));
          const int rem = kbytes - ks * kRowBytes;
          const int nk = min(4, (rem + 31) / 32);
          for (int kk = 0; kk < nk; ++kk) {
            const uint32_t id = idesc_mxf4(BM, BN, (kk & 1) * 2, (kk & 1) * 2);
            mma_mxf4(d, ad + 2 * kk, bd + 2 * kk, id, sfc + 4 * (kk >> 1), sfc + 8 + 4 * (kk >> 1),
                     (ks > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&sm.empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.tfull[buf]));
      }
      tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(&sm.abort_flag);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int g = warp >> 2;             // 64-column half of the 128-wide tile
    const int row = q * 32 + lane;
    uint32_t tl = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
      int m, n;
      tile_coord(t, num_m, num_n, m, n);
      const uint32_t buf = tl & 1u;
      if (sm.abort_flag || !mbar_wait(smem_u32(&sm.tfull[buf]), (tl >> 1) & 1u)) {
        if (!sm.abort_flag) raise_abort(&sm.abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + g * 64;
      const int64_t grow = static_cast<int64_t>(m) * BM + row;
      const int gcol0 = n * BN + g * 64;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[16];
        tmem_ld_16(taddr + c * 16, r);
        tc_wait_ld_16(r);
        if (grow < M) {
          const int col = gcol0 + c * 16;
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          if (Cin != nullptr) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (col + j < N) v[j] += __ldg(Cin + grow * N + col + j);
          }
          if (kBF16Out) {
            __nv_bfloat16* D = static_cast<__nv_bfloat16*>(Dout) + grow * N;
#pragma unroll
            for (int h = 0; h < 16; h += 8) {
              if (vec_out && col + h + 7 < N) {
                uint4 u;
                u.x = pack_bf16x2(v[h + 0], v[h + 1]);
                u.y = pack_bf16x2(v[h + 2], v[h + 3]);
                u.z = pack_bf16x2(v[h + 4], v[h + 5]);
                u.w = pack_bf16x2(v[h + 6], v[h + 7]);
                *reinterpret_cast<uint4*>(D + col + h) = u;
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (col + h + j < N) D[col + h + j] = __float2bfloat16_rn(v[h + j]);
              }
            }
          } else {
            float* D = static_cast<float*>(Dout) + grow * N;
#pragma unroll
            for (int h = 0; h < 16; h += 4) {
              if (vec_out && col + h + 3 < N) {
                *reinterpret_cast<float4*>(D + col + h) =
                    make_float4(v[h], v[h + 1], v[h + 2], v[h + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (col + h + j < N) D[col + h + j] = v[h + j];
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tempty[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace general

// ------------------------------------------------------------- decode path
namespace decode {

constexpr int kDecThreads = 192;   // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kTmemCols = 512;
constexpr int kSlab = 128 * kRowBytes;   // one 128-row x 128-byte weight slab
// Each MMA is tiny (M128 x N<=32 x K64); consecutive MMAs rotate over kAcc
// independent accumulators so they do not form one dependent chain.  The
// epilogue sums them.
constexpr int kAcc = 4;
// K chunks of 128 bytes (256 FP4 values) per pipeline stage when K allows the
// chunked 3-D tensor map (K % 256 == 0): each TMA call then reads CH * 128
// contiguous bytes of every weight row instead of 128.
constexpr int kChunksWide = 2;

template <int NX, int CH>
struct Cfg {
  static constexpr int kStageBytes = CH * (kSlab + NX * kRowBytes + 4 * kSfAtom);
  static constexpr int kStages0 = (200 * 1024) / kStageBytes;
  static constexpr int kStages = kStages0 > 10 ? 10 : kStages0;
  static constexpr int kSfColsPerStage = CH * 16;   // per chunk: SFW 2 atoms + SFX 2 atoms
  static constexpr int kAccCols = kAcc * NX;         // one buffer of accumulators
  static constexpr int kSfBase = 2 * kAccCols;       // after the two buffers
  static_assert(kSfBase + kStages * kSfColsPerStage <= kTmemCols, "TMEM columns");
};

template <int NX, int CH>
struct __align__(1024) Smem {
  static constexpr int S = Cfg<NX, CH>::kStages;
  uint8_t w[S][CH * kSlab];
  uint8_t x[S][CH * NX * kRowBytes];
  uint8_t sfw[S][CH * 2 * kSfAtom];
  uint8_t sfx[S][CH * 2 * kSfAtom];
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  uint32_t last_flag;
  volatile uint32_t abort_flag;
};

// CTA that owns unit u when U units are split evenly over G CTAs
// (CTA c owns [floor(c*U/G), floor((c+1)*U/G))).
__host__ __device__ __forceinline__ int64_t owner(int64_t u, int64_t U, int64_t G) {
  return ((u + 1) * G - 1) / U;
}

struct Plan {
  int64_t tiles, KS, U, G, smax;
  int ch;
};

int chunks_for(int K) { return (K % 256 == 0) ? kChunksWide : 1; }

Plan make_plan(int N, int K, int num_sms) {
  Plan p;
  p.ch = chunks_for(K);
  p.tiles = (N + 127) / 128;
  p.KS = (static_cast<int64_t>(K) / 2 + kRowBytes * p.ch - 1) / (kRowBytes * p.ch);
  p.U = p.tiles * p.KS;
  p.G = p.U < num_sms ? p.U : num_sms;
  p.smax = 1;
  for (int64_t t = 0; t < p.tiles; ++t) {
    const int64_t ns = owner((t + 1) * p.KS - 1, p.U, p.G) - owner(t * p.KS, p.U, p.G) + 1;
    if (ns > p.smax) p.smax = ns;
  }
  return p;
}

template <int NX, int CH, bool kBF16Out>
__global__ void __launch_bounds__(kDecThreads, 1)
    gemm_mxfp4_decode_kernel(const __grid_constant__ CUtensorMap tmX,
                             const __grid_constant__ CUtensorMap tmW,
                             const uint8_t* __restrict__ sfX, const uint8_t* __restrict__ sfW,
                             const float* __restrict__ Cin, void* __restrict__ Dout, int M, int N,
                             int K, int64_t KS, int64_t U, int64_t smax,
                             float* __restrict__ ws, uint32_t* __restrict__ counters) {
  constexpr int kStages = Cfg<NX, CH>::kStages;
  constexpr int kSfCols = Cfg<NX, CH>::kSfColsPerStage;
  constexpr int kAccCols = Cfg<NX, CH>::kAccCols;
  constexpr int kSfBase = Cfg<NX, CH>::kSfBase;
  extern __shared__ uint8_t smem_raw[];
  Smem<NX, CH>& sm = *reinterpret_cast<Smem<NX, CH>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int64_t G = gridDim.x;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * U / G;
  const int64_t u1 = (static_cast<int64_t>(blockIdx.x) + 1) * U / G;
  const int kbytes = K / 2;
  const int KC = (kbytes + kRowBytes - 1) / kRowBytes;   // 128-byte chunks along K
  const int KA = (K / 32 + 3) / 4;                       // scale atoms along K

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.tfull[b]), 1);
      mbar_init(smem_u32(&sm.tempty[b]), 4);
    }
    mbar_init(smem_u32(&sm.final_bar), 1);
    sm.abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();    // activations: re-read by every CTA
      const uint64_t stream = l2_policy_evict_first(); // weights: read exactly once
      uint32_t it = 0;
      for (int64_t u = u0; u < u1; ++u, ++it) {
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        if (sm.abort_flag) break;
        if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        const int64_t tile = u / KS;
        const int c0 = static_cast<int>(u % KS) * CH;    // first 128-byte chunk
        const int ka0 = 2 * c0;
        const int na = min(2 * CH, KA - ka0);
        const uint32_t fb = smem_u32(&sm.full[s]);
        mbar_arrive_expect_tx(fb, CH * (128 + NX) * kRowBytes + 2 * na * kSfAtom);
        if (CH == 1) {
          tma_load_2d_hint(smem_u32(sm.w[s]), &tmW, fb, c0 * kRowBytes, static_cast<int32_t>(tile * 128), stream);
          tma_load_2d_hint(smem_u32(sm.x[s]), &tmX, fb, c0 * kRowBytes, 0, keep);
        } else {
          tma_load_3d_hint(smem_u32(sm.w[s]), &tmW, fb, 0, static_cast<int32_t>(tile * 128), c0, stream);
          tma_load_3d_hint(smem_u32(sm.x[s]), &tmX, fb, 0, 0, c0, keep);
        }
        bulk_load(smem_u32(sm.sfw[s]), sfW + (tile * KA + ka0) * kSfAtom, na * kSfAtom, fb);
        bulk_load(smem_u32(sm.sfx[s]), sfX + static_cast<int64_t>(ka0) * kSfAtom, na * kSfAtom, fb);
      }
      drain_fills(sm.full, kStages, it);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      uint32_t it = 0, seg = 0;
      for (int64_t u = u0; u < u1; ++u, ++it) {
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        const int ks = static_cast<int>(u % KS);
        const bool first = (u == u0) || ks == 0;
        const bool last = (u == u1 - 1) || ks == KS - 1;
        const uint32_t buf = seg & 1u;
        if (sm.abort_flag) break;
        // completion k of tempty[buf] = the k-th time the epilogue handed the
        // (zeroed) buffer back; completion 0 is the initial zeroing
        if (first && !mbar_wait(smem_u32(&sm.tempty[buf]), (seg >> 1) & 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        if (!mbar_wait(smem_u32(&sm.full[s]), ph)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        tc_fence_after();
        const int c0 = ks * CH;
        const int ka0 = 2 * c0;
        const int na = min(2 * CH, KA - ka0);
        const uint32_t sfc = tmem + kSfBase + s * kSfCols;
        const uint32_t d = tmem + buf * kAccCols;
        for (int a = 0; a < na; ++a) {
          tc_cp_32x128b_warpx4(sfc + 16 * (a >> 1) + 4 * (a & 1),
                               sdesc_sf_32x16(smem_u32(sm.sfw[s] + a * kSfAtom)));
          tc_cp_32x128b_warpx4(sfc + 16 * (a >> 1) + 8 + 4 * (a & 1),
                               sdesc_sf_32x16(smem_u32(sm.sfx[s] + a * kSfAtom)));
        }
        const int nch = min(CH, KC - c0);
        for (int j = 0; j < nch; ++j) {
          const uint64_t wd = sdesc_kmajor_sw128(smem_u32(sm.w[s] + j * kSlab));
          const uint64_t xd = sdesc_kmajor_sw128(smem_u32(sm.x[s] + j * NX * kRowBytes));
          const int rem = kbytes - (c0 + j) * kRowBytes;
          const int nk = min(4, (rem + 31) / 32);
          const uint32_t sfj = sfc + 16 * j;
          for (int kk = 0; kk < nk; ++kk) {
            const uint32_t id = idesc_mxf4(128, NX, (kk & 1) * 2, (kk & 1) * 2);
            mma_mxf4(d + (kk % kAcc) * NX, wd + 2 * kk, xd + 2 * kk, id, sfj + 4 * (kk >> 1),
                     sfj + 8 + 4 * (kk >> 1), 1u);
          }
        }
        tc_commit(smem_u32(&sm.empty[s]));
        if (last) {
          tc_commit(smem_u32(&sm.tfull[buf]));
          ++seg;
        }
      }
      tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(&sm.abort_flag);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int row = warp * 32 + lane;               // weight row within the tile
    const uint32_t lane_taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    {
      // zero both accumulator buffers and hand them to the MMA thread
      uint32_t z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) z[j] = 0u;
      for (int c = 0; c < 2 * kAccCols; c += 16) tmem_st_16(lane_taddr + c, z);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.tempty[0]));
        mbar_arrive(smem_u32(&sm.tempty[1]));
      }
    }
    uint32_t seg = 0;
    int64_t u = u0;
    while (u < u1) {
      const int64_t tile = u / KS;
      const int64_t seg_end = min(u1, (tile + 1) * KS);
      const bool whole = (u == tile * KS) && (seg_end == (tile + 1) * KS);
      const uint32_t buf = seg & 1u;
      if (sm.abort_flag || !mbar_wait(smem_u32(&sm.tfull[buf]), (seg >> 1) & 1u)) {
        if (!sm.abort_flag) raise_abort(&sm.abort_flag);
        break;
      }
      tc_fence_after();
      float acc[NX];
      {
        const uint32_t taddr = lane_taddr + buf * kAccCols;
        uint32_t z[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) z[j] = 0u;
#pragma unroll
        for (int c = 0; c < NX / 16; ++c) {
#pragma unroll
          for (int a = 0; a < kAcc; ++a) {
            uint32_t r[16];
            tmem_ld_16(taddr + a * NX + c * 16, r);
            tc_wait_ld_16(r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc[c * 16 + j] = (a == 0 ? 0.0f : acc[c * 16 + j]) + __uint_as_float(r[j]);
            tmem_st_16(taddr + a * NX + c * 16, z);    // zero for the next segment
          }
        }
        tc_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tempty[buf]));
      const int64_t n = tile * 128 + row;
      if (whole) {
        if (n < N) {
#pragma unroll
          for (int mm = 0; mm < NX; ++mm) {
            if (mm < M) {
              float v = acc[mm];
              if (Cin != nullptr) v += __ldg(Cin + static_cast<int64_t>(mm) * N + n);
              if (kBF16Out)
                static_cast<__nv_bfloat16*>(Dout)[static_cast<int64_t>(mm) * N + n] = __float2bfloat16_rn(v);
              else
                static_cast<float*>(Dout)[static_cast<int64_t>(mm) * N + n] = v;
            }
          }
        }
      } else {
        const int64_t first_owner = owner(tile * KS, U, G);
        const int64_t nseg = owner((tile + 1) * KS - 1, U, G) - first_owner + 1;
        const int64_t sidx = static_cast<int64_t>(blockIdx.x) - first_owner;
        float* part = ws + (tile * smax + sidx) * NX * 128;
#pragma unroll
        for (int mm = 0; mm < NX; ++mm) part[mm * 128 + row] = acc[mm];
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (threadIdx.x == 0) {
          const uint32_t prev = atomicAdd(&counters[tile], 1u);
          sm.last_flag = (prev + 1 == static_cast<uint32_t>(nseg)) ? 1u : 0u;
          // a counter past its segment count means the workspace was not zero
          if (prev + 1 > static_cast<uint32_t>(nseg)) atomicOr(&g_mxfp4_error, kErrWorkspace);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (sm.last_flag) {
          __threadfence();
          // Sum the segments in order (deterministic), then zero every slot
          // of this row so the workspace is left zero-filled for any shape.
          float* base = ws + tile * smax * NX * 128 + row;
          float tot[NX];
#pragma unroll
          for (int mm = 0; mm < NX; ++mm) tot[mm] = 0.0f;
          for (int64_t sg = 0; sg < nseg; ++sg) {
#pragma unroll
            for (int mm = 0; mm < NX; ++mm) {
              float* slot = base + (sg * NX + mm) * 128;
              tot[mm] += __ldcg(slot);
              *slot = 0.0f;
            }
          }
          if (n < N) {
#pragma unroll
            for (int mm = 0; mm < NX; ++mm) {
              if (mm < M) {
                float v = tot[mm];
                if (Cin != nullptr) v += __ldg(Cin + static_cast<int64_t>(mm) * N + n);
                if (kBF16Out)
                  static_cast<__nv_bfloat16*>(Dout)[static_cast<int64_t>(mm) * N + n] = __float2bfloat16_rn(v);
                else
                  static_cast<float*>(Dout)[static_cast<int64_t>(mm) * N + n] = v;
              }
            }
          }
          if (threadIdx.x == 0) atomicExch(&counters[tile], 0u);
        }
      }
      u = seg_end;
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace decode

template <typename Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

}  // namespace

cudaError_t gemm_mxfp4_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_mxfp4_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_mxfp4_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t launch_gemm_mxfp4(const Mxfp4GemmArgs& a, int num_sms, cudaStream_t s) {
  using namespace general;
  const size_t smem = sizeof(Smem) + 1024;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) &&
                       (a.out_bf16 ? (a.N % 8 == 0) : (a.N % 4 == 0));
  cudaError_t e;
  if (a.out_bf16) {
    e = set_smem(gemm_mxfp4_kernel<true>, smem);
    if (e != cudaSuccess) return e;
    gemm_mxfp4_kernel<true><<<grid, kThreads, smem, s>>>(a.tmA, a.tmB, a.sfA, a.sfB, a.C, a.D,
                                                         a.M, a.N, a.K, vec_out);
  } else {
    e = set_smem(gemm_mxfp4_kernel<false>, smem);
    if (e != cudaSuccess) return e;
    gemm_mxfp4_kernel<false><<<grid, kThreads, smem, s>>>(a.tmA, a.tmB, a.sfA, a.sfB, a.C, a.D,
                                                          a.M, a.N, a.K, vec_out);
  }
  return cudaGetLastError();
}

size_t gemm_mxfp4_decode_workspace(int M, int N, int K, int num_sms) {
  const decode::Plan p = decode::make_plan(N, K, num_sms);
  if (p.smax <= 1) return 0;
  const int nx = M <= 16 ? 16 : 32;
  const size_t floats = static_cast<size_t>(p.tiles * p.smax * nx * 128);
  return floats * sizeof(float) + static_cast<size_t>(p.tiles) * sizeof(uint32_t);
}

namespace {
template <int NX, int CH, bool BF>
cudaError_t launch_decode_variant(const Mxfp4GemmArgs& a, const decode::Plan& p, float* ws,
                                  uint32_t* counters, cudaStream_t s) {
  using namespace decode;
  CUtensorMap tmX, tmW;
  const uint64_t kb = static_cast<uint64_t>(a.K) / 2;
  if (CH == 1) {
    if (!make_kmajor_map(&tmX, a.A, kb, a.M, kb, NX) || !make_kmajor_map(&tmW, a.B, kb, a.N, kb, 128))
      return cudaErrorInvalidValue;
  } else {
    if (!make_kmajor_map_chunked(&tmX, a.A, kb, a.M, kb, NX, CH) ||
        !make_kmajor_map_chunked(&tmW, a.B, kb, a.N, kb, 128, CH))
      return cudaErrorInvalidValue;
  }
  const size_t smem = sizeof(Smem<NX, CH>) + 1024;
  cudaError_t e = set_smem(gemm_mxfp4_decode_kernel<NX, CH, BF>, smem);
  if (e != cudaSuccess) return e;
  gemm_mxfp4_decode_kernel<NX, CH, BF><<<static_cast<int>(p.G), kDecThreads, smem, s>>>(
      tmX, tmW, a.sfA, a.sfB, a.C, a.D, a.M, a.N, a.K, p.KS, p.U, p.smax, ws, counters);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_mxfp4_decode(const Mxfp4GemmArgs& a, int num_sms, cudaStream_t s) {
  using namespace decode;
  const Plan p = make_plan(a.N, a.K, num_sms);
  const int nx = a.M <= 16 ? 16 : 32;
  float* ws = static_cast<float*>(a.workspace);
  uint32_t* counters =
      ws == nullptr ? nullptr : reinterpret_cast<uint32_t*>(ws + p.tiles * p.smax * nx * 128);
  const int key = (nx == 16 ? 0 : 4) | (p.ch == 1 ? 0 : 2) | (a.out_bf16 ? 1 : 0);
  switch (key) {
    case 0: return launch_decode_variant<16, 1, false>(a, p, ws, counters, s);
    case 1: return launch_decode_variant<16, 1, true>(a, p, ws, counters, s);
    case 2: return launch_decode_variant<16, kChunksWide, false>(a, p, ws, counters, s);
    case 3: return launch_decode_variant<16, kChunksWide, true>(a, p, ws, counters, s);
    case 4: return launch_decode_variant<32, 1, false>(a, p, ws, counters, s);
    case 5: return launch_decode_variant<32, 1, true>(a, p, ws, counters, s);
    case 6: return launch_decode_variant<32, kChunksWide, false>(a, p, ws, counters, s);
    default: return launch_decode_variant<32, kChunksWide, true>(a, p, ws, counters, s);
  }
}

}  // namespace bsg

// FP8 block-scaled GEMM with per-K-tile promotion, for sm_103a.
//
//   D[i][j] = sum_t (s_A(i,t) * s_B(j,t)) * P_t[i][j] + C[i][j]
//   P_t     = sum_{k in K tile t} a[i][k] * b[j][k]      (128-wide K tiles)
//
// The per-tile FP32 scales of "FP8 GEMM on CDNA4" (section 3.3, multiplied
// back after accumulation in section 4.4) are not powers of two, so they can
// not ride inside the tensor core.  Each 128-wide K tile's partial product
// P_t is formed by four tcgen05.mma (K = 32 each) into a tensor-memory
// buffer, then drained by CUDA-core warps that compute
//     acc = fmaf(s_A * s_B, P_t, acc)
// in an FP32 register accumulator.  This is the promotion that
// "FP8 MMA internals on Hopper" motivates (a chained tensor-core accumulator
// sets the alignment exponent and drops small terms); on GB300 the partial
// lives in tensor memory, double-buffered, so the MMA of tile t+1 overlaps
// the drain of tile t.
//
// Two shapes of the same kernel:
//   * single CTA: 128 x 256 output tiles; per K tile the SM loads A 16 KB +
//     B 32 KB into a 3-stage ring;
//   * CTA pair (a cluster of two on neighbouring SMs, tcgen05 cta_group::2):
//     256 x 256 tiles.  Each CTA loads its 128 rows of A and 128 of the 256
//     rows of B (32 KB per K tile, 4 stages); one thread of the even CTA
//     issues M = 256 MMAs that read both CTAs' shared memory and write each
//     CTA's 128 rows of the partial into its own tensor memory.  Per FLOP an
//     SM moves two thirds of the single-CTA bytes.
//
// Warp roles (384 threads = 3 warpgroups, one CTA per SM, persistent):
//   warp 0     producer: TMA loads of A and B.
//   warp 1     tensor-memory allocator; MMA issuer (one lane; in a pair only
//              the even CTA's).  One tcgen05.commit per K tile arrives on
//              the stage's `done` barrier: it both frees the shared-memory
//              stage for the producer and hands the partial to the drain.
//   warp 2     scale loader: cp.async of each K tile's scales into an 8-slot
//              ring, as far ahead as the ring allows.
//   warp 3     output store: writes the staged tile to D (TMA tensor stores,
//              or a bounds-checked copy when D's pitch does not allow TMA).
//   warps 4-11 promotion + epilogue: warpgroups 1 and 2.  Warp w reads TMEM
//              lanes 32*(w%4)..+31 (its rows) and column half (w-4)/4 of the
//              256-wide tile.
// The promotion warps hand each finished tile to the store warp through a
// 64 KB shared-memory staging buffer (128-byte swizzled, the TMA layout) and
// go straight on to the next tile's drain, so the output stores of all SMs
// (which finish their tiles at the same moments) overlap the next tile's
// MMAs instead of stalling them.
// Registers: the kernel launches at 168 per thread (384 x 168 = 64512);
// warpgroup 0 gives back down to 56 and the promotion warpgroups take 224
// each, 128 x 56 + 256 x 224 = 64512, which holds 128 FP32 accumulators plus
// two 16-column TMEM load buffers per thread without spilling.  The drain
// uses paired FP32 FMAs (fma.rn.f32x2), one instruction per two elements.
// Every wait is bounded; a wait that runs out sets the error word, raises a
// CTA-wide abort flag and all roles unwind to the final barrier.
#include "common.cuh"
#include "kernels.h"
#include "quant_math.cuh"

namespace bsg {
namespace {

__device__ uint32_t g_fp8_error = 0;

constexpr int BM = 128;            // output rows per CTA
constexpr int BN = 256;            // output columns per tile
constexpr int BK = 128;            // one scale tile along K = one promotion unit
constexpr int kScaleSlots = 8;
constexpr int kThreads = 384;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp = 2;
constexpr int kStoreWarp = 3;
constexpr int kFirstPromoWarp = 4;
constexpr int kRegsSmall = 56;     // warpgroup 0 after setmaxnreg.dec
constexpr int kRegsLarge = 224;    // promotion warpgroups after setmaxnreg.inc
static_assert(128 * kRegsSmall + 256 * kRegsLarge <= kThreads * 168,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;     // two 256-column FP32 partial buffers
constexpr int kGroup = 8;          // tile raster: groups of 8 tiles
constexpr int kDrainCols = 32;     // TMEM columns per tcgen05.ld in the drain

template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 32) tmem_ld_32(taddr, r); else tmem_ld_16(taddr, r);
}
template <int W>
__device__ __forceinline__ void tmem_wait_cols(uint32_t (&r)[W]) {
  if constexpr (W == 32) tc_wait_ld_32(r); else tc_wait_ld_16(r);
}

// What the epilogue writes: FP32, BF16 (round to nearest even), or the
// result quantised to E4M3 / E5M2 per 1 x 128 run of a row (codes + FP32
// scales)
enum OutKind : int { kOutF32 = 0, kOutBF16 = 1, kOutE4M3 = 2, kOutE5M2 = 3 };

constexpr uint32_t kOutBytes = 64 * 1024;   // output staging
constexpr uint32_t kOutBlock = 128 * 128;   // one 128-row x 128-byte swizzled box

template <bool kPair>
struct Cfg {
  static constexpr int kStages = kPair ? 4 : 3;
  static constexpr int kBRows = kPair ? BN / 2 : BN;        // B rows this CTA loads
  static constexpr int kTileM = kPair ? 2 * BM : BM;        // rows of a tile
  static constexpr int kPromoArrivals = kPair ? 16 : 8;     // drains per TMEM buffer
  static constexpr uint32_t kStageBytes = (BM + kBRows) * BK;
  static constexpr uint32_t kFullBytes = (kPair ? 2 : 1) * kStageBytes;
};

template <bool kPair>
struct __align__(1024) Smem {
  uint8_t a[Cfg<kPair>::kStages][BM * BK];
  uint8_t b[Cfg<kPair>::kStages][Cfg<kPair>::kBRows * BK];
  // finished tile on its way to D: BF16 / FP8 codes -> the two column
  // halves in two 32 KB slots; FP32 -> one half at a time in all 64 KB
  uint8_t out[kOutBytes];
  float sa[kScaleSlots][BM];
  float sb[kScaleSlots][BN];
  uint64_t full[Cfg<kPair>::kStages];
  uint64_t done[Cfg<kPair>::kStages];   // MMAs of the stage complete
  uint64_t tempty[2];
  uint64_t sfull[kScaleSlots];
  uint64_t sempty[kScaleSlots];
  uint64_t ofull[2];                     // column half h staged
  uint64_t ofree[2];                     // its staging read out
  uint64_t final_bar;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
};

struct TileCoord {
  int m, n;
};

// Raster of the persistent tile loop.  Tiles are visited in groups of kGroup
// rows of tiles along one dimension while the other is swept, so the operand
// panel of the group stays in L2 and the swept operand is re-read from L2.
// along_n = true groups along N (sweeps M): chosen when A is the smaller
// operand, so the whole of A is what gets re-read and stays resident.
__device__ __forceinline__ TileCoord tile_coord(int t, int num_m, int num_n, bool along_n) {
  const int outer = along_n ? num_n : num_m;
  const int inner = along_n ? num_m : num_n;
  const int group_size = kGroup * inner;
  const int group = t / group_size;
  const int first = group * kGroup;
  const int gsz = min(outer - first, kGroup);
  const int local = t % group_size;
  const int o = first + local % gsz, i = local / gsz;
  return along_n ? TileCoord{i, o} : TileCoord{o, i};
}

// ---- the fused output quantiser (one thread = one 1 x 128 run of a row) --
//
// Codes of the 128 values (64 pairs) of acc divided by s, correctly rounded
// to FP32 first (as the stand-alone quantiser and the 1 x 128 rule require),
// then RNE-satfinite to the FP8 format, staged as eight 16-byte pieces of
// the 128-byte-swizzled box.  The quotient is Markstein's division (see
// GroupDiv): q0 = x r, q1 = q0 + (x - q0 s) r, q2 = q1 + (x - q1 s) r, valid
// for s in [2^-80, 2^80] (the caller scales other groups into that range).
// Scalar FMAs: the paired form needs aligned register pairs, and with the
// 128 accumulators live that made the promotion warps spill.  A code's sign bit is
// taken from x: a non-zero quotient of x by a positive s has x's sign, and a
// quotient that rounds to zero is -0 exactly when x is negative.
template <int kFmt>
__device__ __forceinline__ void stage_codes(const uint64_t (&acc)[64], float s, float r,
                                                 uint32_t base, int row) {
  const uint64_t r2 = f32x2_pack(r, r);
  const uint64_t ns2 = f32x2_pack(-s, -s);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint64_t x01 = acc[8 * c + 2 * p], x23 = acc[8 * c + 2 * p + 1];
      float v[4], q[4];
      f32x2_unpack(x01, v[0], v[1]);
      f32x2_unpack(x23, v[2], v[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float t = v[i] * r;
        t = fmaf(fmaf(-t, s, v[i]), r, t);
        q[i] = fmaf(fmaf(-t, s, v[i]), r, t);
      }
      const float a = q[0], b = q[1], cc = q[2], d = q[3];
      const uint32_t sg = __byte_perm(
          __byte_perm(static_cast<uint32_t>(x01), static_cast<uint32_t>(x01 >> 32), 0x0073),
          __byte_perm(static_cast<uint32_t>(x23), static_cast<uint32_t>(x23 >> 32), 0x0073), 0x5410);
      w[p] = (cvt4_fp8(kFmt, a, b, cc, d) & 0x7F7F7F7Fu) | (sg & 0x80808080u);
    }
    st_shared_v4(base + row * 128 + ((c ^ (row & 7)) << 4), make_uint4(w[0], w[1], w[2], w[3]));
  }
}

__device__ __forceinline__ void raise_abort(volatile uint32_t* flag) {
  atomicOr(&g_fp8_error, kErrTimeout);
  *flag = 1u;
}

template <bool kPair, bool kARow, bool kBRow, int kOut>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const float* __restrict__ sA,
                    const float* __restrict__ sB, const float* __restrict__ Cin,
                    void* __restrict__ Dout, float* __restrict__ sD, int M, int N, int K,
                    uint32_t idesc, bool tma_out, bool raster_n, float qmax) {
  using C = Cfg<kPair>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  Smem<kPair>& sm = *reinterpret_cast<Smem<kPair>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;      // 0 = the pair's MMA issuer
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int num_m = (M + C::kTileM - 1) / C::kTileM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int KT = (K + BK - 1) / BK;
  const int num_nb = (N + 127) / 128;   // 128-wide scale blocks of B

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.done[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.tempty[b]), C::kPromoArrivals);
      mbar_init(smem_u32(&sm.ofull[b]), 4);
      mbar_init(smem_u32(&sm.ofree[b]), 1);
    }
    for (int s = 0; s < kScaleSlots; ++s) {
      mbar_init(smem_u32(&sm.sfull[s]), 32);
      mbar_init(smem_u32(&sm.sempty[s]), 8);
    }
    mbar_init(smem_u32(&sm.final_bar), 1);
    sm.abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(&sm.tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (tma_out) tma_prefetch_desc(&tmD);
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();    // barriers and tensor memory of both CTAs are ready
  tc_fence_after();
  grid_dep_launch();
  grid_dep_wait();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kRegsSmall>();
    const uint64_t keep = l2_policy_evict_last();   // operands are re-read by other tiles
    uint32_t it = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      const int m_cta = tc.m * C::kTileM + static_cast<int>(rank) * BM;   // this CTA's rows
      const int n_b = tc.n * BN + static_cast<int>(rank) * (BN - C::kBRows);   // its B rows
      for (int kt = 0; kt < KT; ++kt, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(smem_u32(&sm.done[s]), ph ^ 1u);
          if (good) {
            const uint32_t fb = smem_u32(&sm.full[s]);
            if (kPair) {
              // both CTAs' loads complete on the even CTA's barrier
              if (rank == 0) mbar_arrive_expect_tx(fb, C::kFullBytes);
              const uint32_t fb0 = mapa_shared(fb, 0);
              tma_load_2d_pair(smem_u32(sm.a[s]), &tmA, fb0, kt * BK, m_cta, keep);
              tma_load_2d_pair(smem_u32(sm.b[s]), &tmB, fb0, kt * BK, n_b, keep);
            } else {
              mbar_arrive_expect_tx(fb, C::kFullBytes);
              tma_load_2d_hint(smem_u32(sm.a[s]), &tmA, fb, kt * BK, m_cta, keep);
              tma_load_2d_hint(smem_u32(sm.b[s]), &tmB, fb, kt * BK, n_b, keep);
            }
          } else {
            raise_abort(&sm.abort_flag);
          }
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
      }
    }
    // the even CTA's full barriers also count the peer's bytes
    if (lane == 0 && rank == 0) drain_fills(sm.full, kStages, it);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0 && rank == 0) {
      // K tile it (counted across this CTA's output tiles) may start once
      // its stage holds the operands (full) and its partial buffer it & 1
      // has been drained (tempty).  The MMA queue holds little more than the
      // running MMA, so a non-blocking test of the next stage goes between
      // this K tile's MMAs, where it hides under a running one; the commit
      // follows the last MMA at once (it starts the drain); the waits that
      // may block (the drain, a stage that was not ready) come after it.
      // No shared-memory flag is read per K tile: a shared-memory access
      // right after a commit stalls this thread for a few hundred cycles,
      // and the bounded waits catch an abort anyway.
      const int my_tiles = unit < tiles ? (tiles - 1 - unit) / units + 1 : 0;
      const uint32_t total = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(KT);
      bool ok = total == 0 ||
                (mbar_wait(smem_u32(&sm.tempty[0]), 1u) && mbar_wait(smem_u32(&sm.full[0]), 0u));
      if (!ok) raise_abort(&sm.abort_flag);
      tc_fence_after();
      for (uint32_t it = 0; it < total && ok; ++it) {
        const uint32_t b = it & 1u;
        const int s = static_cast<int>(it % kStages);
        const bool more = it + 1 < total;
        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm.a[s]));
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sm.b[s]));
        const uint32_t d = tmem + b * BN;
        bool next_ready = false;
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk) {
          if (kPair)
            mma_f8f6f4_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          else
            mma_f8f6f4(d, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          if (kk == 1 && more)
            next_ready = mbar_test(smem_u32(&sm.full[(it + 1) % kStages]), ((it + 1) / kStages) & 1u);
        }
        if (kPair)
          tc_commit_pair_mc(smem_u32(&sm.done[s]), 3);
        else
          tc_commit(smem_u32(&sm.done[s]));
        if (more && ((!next_ready && !mbar_wait(smem_u32(&sm.full[(it + 1) % kStages]),
                                                ((it + 1) / kStages) & 1u)) ||
                     !mbar_wait(smem_u32(&sm.tempty[(it + 1) & 1u]), (((it + 1) >> 1) & 1u) ^ 1u))) {
          raise_abort(&sm.abort_flag);
          ok = false;
        }
        tc_fence_after();
      }
      // every MMA this thread issued has completed once final_bar flips
      if (kPair)
        tc_commit_pair(smem_u32(&sm.final_bar));
      else
        tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(&sm.abort_flag);
    }
    __syncwarp();
  } else if (warp == kScaleWarp) {
    // ------------------------------------------------------- scale loader
    // Each K tile's scales go to one slot of an 8-slot ring.  This warp is
    // gated only by the promotion warps releasing slots, so it runs up to
    // eight K tiles ahead of them and the loads' latency stays off the
    // MMA -> drain -> MMA chain.
    setmaxnreg_dec<kRegsSmall>();
    uint32_t it = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      const int m_cta = tc.m * C::kTileM + static_cast<int>(rank) * BM;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int ss = static_cast<int>(it % kScaleSlots);
        const uint32_t phs = (it / kScaleSlots) & 1u;
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(smem_u32(&sm.sempty[ss]), phs ^ 1u);
          if (!good) raise_abort(&sm.abort_flag);
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
        // this CTA's 128 rows of A, all 256 columns of the tile
        if (kARow) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = m_cta + 4 * lane + j;
            if (r < M) cp_async_4(smem_u32(&sm.sa[ss][4 * lane + j]), sA + static_cast<int64_t>(kt) * M + r);
          }
        } else if (lane == 0) {
          cp_async_4(smem_u32(&sm.sa[ss][0]), sA + static_cast<int64_t>(m_cta / BM) * KT + kt);
        }
        if (kBRow) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = tc.n * BN + 8 * lane + j;
            if (c < N) cp_async_4(smem_u32(&sm.sb[ss][8 * lane + j]), sB + static_cast<int64_t>(kt) * N + c);
          }
        } else if (lane < BN / 128) {
          const int nb = tc.n * (BN / 128) + lane;
          if (nb < num_nb)
            cp_async_4(smem_u32(&sm.sb[ss][128 * lane]), sB + static_cast<int64_t>(nb) * KT + kt);
        }
        cp_async_mbar_arrive_noinc(smem_u32(&sm.sfull[ss]));
      }
    }
    cp_async_wait_all();
    __syncwarp();
  } else if (warp == kStoreWarp) {
    // -------------------------------------------------------- output store
    setmaxnreg_dec<kRegsSmall>();
    constexpr bool kCodes = kOut == kOutE4M3 || kOut == kOutE5M2;
    constexpr int kElem = kOut == kOutF32 ? 4 : (kOut == kOutBF16 ? 2 : 1);
    constexpr int kBoxCols = 128 / kElem;              // columns of one swizzled box
    constexpr int kHalfBlocks = 128 / kBoxCols;        // boxes of a 128-column half
    const uint64_t stream_out = l2_policy_evict_first();   // D is not re-read here
    uint32_t tl = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units, ++tl) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      const int row0 = tc.m * C::kTileM + static_cast<int>(rank) * BM;   // this CTA's rows
      for (int h = 0; h < 2; ++h) {
        if (sm.abort_flag) { ok = false; break; }
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(smem_u32(&sm.ofull[h]), tl & 1u);
          if (!good) raise_abort(&sm.abort_flag);
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
        const uint32_t base = smem_u32(sm.out) + (kOut != kOutF32 ? h * (kOutBytes / 2) : 0u);
        const int col0 = tc.n * BN + h * 128;
        if (tma_out) {
          if (lane == 0) {
            for (int blk = 0; blk < kHalfBlocks; ++blk) {
              const int x = col0 + blk * kBoxCols;
              if (x < N && row0 < M) tma_store_2d_hint(&tmD, base + blk * kOutBlock, x, row0, stream_out);
            }
            bulk_commit_group();
            bulk_wait_group_read0();   // the staging may be overwritten from here on
          }
        } else {
          // 16-byte pieces of 128 rows x 128 columns, bounds-checked
          constexpr int kPieces = 128 * 128 * kElem / 16;
          constexpr int kPerPiece = 16 / kElem;
          for (int i = lane; i < kPieces; i += 32) {
            const int r = i / (kPieces / 128);
            const int c = i % (kPieces / 128);           // piece along the row
            const int blk = c / 8, cc = c % 8;
            const uint4 u = ld_shared_v4(base + blk * kOutBlock + r * 128 + ((cc ^ (r & 7)) << 4));
            const int64_t grow = static_cast<int64_t>(row0) + r;
            const int col = col0 + c * kPerPiece;
            if (grow >= M || col >= N) continue;
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < kPerPiece; ++j) {
              if (col + j >= N) break;
              if (kCodes)
                reinterpret_cast<uint8_t*>(Dout)[grow * N + col + j] =
                    static_cast<uint8_t>(w[j / 4] >> (8 * (j % 4)));
              else if (kOut == kOutBF16)
                reinterpret_cast<uint16_t*>(Dout)[grow * N + col + j] =
                    static_cast<uint16_t>(w[j / 2] >> (16 * (j % 2)));
              else
                reinterpret_cast<float*>(Dout)[grow * N + col + j] = __uint_as_float(w[j]);
            }
          }
          __syncwarp();
        }
        if (lane == 0) mbar_arrive(smem_u32(&sm.ofree[h]));
      }
    }
    if (tma_out && lane == 0) bulk_wait_group0();   // stores complete before the CTA exits
    __syncwarp();
  } else {
    // ------------------------------------------------- promotion + epilogue
    setmaxnreg_inc<kRegsLarge>();
    const int q = warp & 3;                        // TMEM lane quarter = rows 32q..32q+31
    const int g = (warp - kFirstPromoWarp) >> 2;   // column half of the 256-wide tile
    const int row = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + g * 128;
    // where this warp reports a drained buffer: the issuing CTA's barrier
    const uint32_t tempty0 = kPair ? mapa_shared(smem_u32(&sm.tempty[0]), 0) : smem_u32(&sm.tempty[0]);
    uint32_t it = 0, tl = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units, ++tl) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      uint64_t acc[64];                            // 128 FP32 accumulators, in pairs
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0ull;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const uint32_t b = it & 1u;
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        const int ss = static_cast<int>(it % kScaleSlots);
        const uint32_t phs = (it / kScaleSlots) & 1u;
        // the MMA can run at most two K tiles ahead of this drain (two TMEM
        // buffers), less than a round of the stage ring, so done[s] is never
        // more than one phase past the one waited for
        if (sm.abort_flag || !mbar_wait(smem_u32(&sm.sfull[ss]), phs) ||
            !mbar_wait(smem_u32(&sm.done[s]), ph)) {
          if (!sm.abort_flag) raise_abort(&sm.abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const float sa = kARow ? sm.sa[ss][row] : sm.sa[ss][0];
        const float sc = kBRow ? sa : sa * sm.sb[ss][g * 128];
        const uint64_t sc2 = f32x2_pack(sc, sc);
        const uint32_t taddr = lane_base + b * BN;
        // kDrainCols columns per tcgen05.ld, double-buffered; the buffer is
        // handed back to the MMA as soon as its last load has landed, before
        // the last chunk's FMAs
        constexpr int kChunks = 128 / kDrainCols;
        uint32_t r0[kDrainCols], r1[kDrainCols];
        tmem_ld_cols(taddr, r0);
        tmem_wait_cols(r0);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          uint32_t (&cur)[kDrainCols] = (c & 1) ? r1 : r0;
          uint32_t (&nxt)[kDrainCols] = (c & 1) ? r0 : r1;
          if (c + 1 < kChunks) tmem_ld_cols(taddr + (c + 1) * kDrainCols, nxt);
#pragma unroll
          for (int j = 0; j < kDrainCols / 2; ++j) {
            const uint64_t p = f32x2_pack(__uint_as_float(cur[2 * j]), __uint_as_float(cur[2 * j + 1]));
            const int pair_idx = (c * kDrainCols) / 2 + j;
            if (kBRow) {
              const float2 sbv = *reinterpret_cast<const float2*>(&sm.sb[ss][g * 128 + 2 * pair_idx]);
              ffma2(acc[pair_idx], fmul2(sc2, f32x2_pack(sbv.x, sbv.y)), p);
            } else {
              ffma2(acc[pair_idx], sc2, p);
            }
          }
          if (c + 1 < kChunks) tmem_wait_cols(nxt);
          if (c == kChunks - 2) {
            // every tcgen05.ld of this buffer has completed: nothing to
            // publish, so a relaxed arrive suffices
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(tempty0 + b * 8);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(smem_u32(&sm.sempty[ss]));   // scales used
      }
      if (!ok) break;
      // ---- epilogue: this thread's row x 128 columns go to the staging
      // buffer as 16-byte pieces in the 128-byte-swizzled box layout (piece
      // c of row r at r*128 + ((c ^ (r & 7)) << 4) inside its box), which
      // the TMA store reads and which spreads a warp's 32 rows over all
      // banks.  BF16 / FP8: half g owns slot g and waits for the store of its
      // own previous tile; FP32: a half fills the whole buffer, so half 0
      // waits for the previous tile's half 1 and half 1 for this tile's half 0.
      {
        constexpr bool kSlots = kOut != kOutF32;
        const uint32_t wb = kSlots ? static_cast<uint32_t>(g) : static_cast<uint32_t>(g ^ 1);
        const uint32_t wph = kSlots ? ((tl & 1u) ^ 1u) : (g == 0 ? ((tl & 1u) ^ 1u) : (tl & 1u));
        if (!mbar_wait(smem_u32(&sm.ofree[wb]), wph)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        const uint32_t base = smem_u32(sm.out) + (kSlots ? g * (kOutBytes / 2) : 0u);
        const int64_t grow = static_cast<int64_t>(tc.m) * C::kTileM + rank * BM + row;
        const int gcol0 = tc.n * BN + g * 128;
        if constexpr (kOut == kOutE4M3 || kOut == kOutE5M2) {
          // The fused quantiser: this thread's 128 columns are one 1 x 128
          // run of the output row, i.e. one scale group of the next GEMM's
          // activations, so the group maximum needs no exchange between
          // threads.  Same rule as the stand-alone quantiser: s = max|x| /
          // fmt_max (1 if 0), codes = RNE_satfinite(x / s) with a correctly
          // rounded division.  Columns at or beyond N are zeroed first.
          const int nvalid = N - gcol0;
          if (Cin != nullptr && grow < M) {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
              float x0, x1;
              f32x2_unpack(acc[j], x0, x1);
              if (2 * j < nvalid) x0 += __ldg(Cin + grow * N + gcol0 + 2 * j);
              if (2 * j + 1 < nvalid) x1 += __ldg(Cin + grow * N + gcol0 + 2 * j + 1);
              acc[j] = f32x2_pack(x0, x1);
            }
          }
          if (nvalid < 128) {    // the group crosses N: zero what lies beyond
#pragma unroll
            for (int j = 0; j < 64; ++j) {
              float x0, x1;
              f32x2_unpack(acc[j], x0, x1);
              acc[j] = f32x2_pack(2 * j < nvalid ? x0 : 0.0f, 2 * j + 1 < nvalid ? x1 : 0.0f);
            }
          }
          float m[8];            // eight independent max chains
#pragma unroll
          for (int j = 0; j < 8; ++j) m[j] = 0.0f;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            float x0, x1;
            f32x2_unpack(acc[j], x0, x1);
            m[j & 7] = fmaxf(m[j & 7], fmaxf(fabsf(x0), fabsf(x1)));
          }
          const float amax = fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])),
                                   fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
          const float sc = fp8_scale(amax, qmax);
          float sd = sc;         // the divisor the quotients are formed with
          if (!(sc >= 0x1p-80f && sc <= 0x1p80f)) {
            // Bring s into the division's range with a power of two P applied
            // to s and to every x: x / s is unchanged.  P = 2^100 (s < 2^-80)
            // is exact for all x (|x| <= s fmt_max < 2^-16 with fmt_max <=
            // 2^64).  P = 2^-100 (s > 2^80) rounds x only when |x| < 2^-26,
            // i.e. |x / s| < 2^-106, which is a signed zero in FP8 either way.
            const float P = sc < 0x1p-80f ? 0x1p100f : 0x1p-100f;
            const uint64_t P2 = f32x2_pack(P, P);
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = fmul2(acc[j], P2);
            sd = sc * P;
          }
          stage_codes<kOut == kOutE4M3 ? 0 : 1>(acc, sd, __frcp_rn(sd), base, row);
          // scales K-tile major for the next GEMM: [ceil(N/128)][M]
          if (grow < M && nvalid > 0) sD[static_cast<int64_t>(gcol0 / 128) * M + grow] = sc;
        } else {
          constexpr int kElem = kOut == kOutBF16 ? 2 : 4;
          constexpr int kPerPiece = 16 / kElem;
#pragma unroll
          for (int c = 0; c < 128 / kPerPiece; ++c) {
            float v[kPerPiece];
#pragma unroll
            for (int j = 0; j < kPerPiece / 2; ++j)
              f32x2_unpack(acc[(c * kPerPiece) / 2 + j], v[2 * j], v[2 * j + 1]);
            if (Cin != nullptr && grow < M) {
#pragma unroll
              for (int j = 0; j < kPerPiece; ++j) {
                const int col = gcol0 + c * kPerPiece + j;
                if (col < N) v[j] += __ldg(Cin + grow * N + col);
              }
            }
            uint4 u;
            if (kOut == kOutBF16) {
              u.x = pack_bf16x2(v[0], v[1]);
              u.y = pack_bf16x2(v[2], v[3]);
              u.z = pack_bf16x2(v[4 % kPerPiece], v[5 % kPerPiece]);
              u.w = pack_bf16x2(v[6 % kPerPiece], v[7 % kPerPiece]);
            } else {
              u = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                             __float_as_uint(v[2 % kPerPiece]), __float_as_uint(v[3 % kPerPiece]));
            }
            const int blk = c / 8, cc = c % 8;
            st_shared_v4(base + blk * kOutBlock + row * 128 + ((cc ^ (row & 7)) << 4), u);
          }
        }
        fence_proxy_async_smem();    // the staged bytes are read by the TMA (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.ofull[g]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();    // neither CTA leaves while the other may still signal it
  if (warp == kMmaWarp) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
  if (kPair) {
    __syncthreads();
    cluster_sync();
  }
}

template <bool kPair, bool kARow, bool kBRow, int kOut>
cudaError_t launch_variant(const Fp8GemmArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gemm_fp8_kernel<kPair, kARow, kBRow, kOut>;
  const size_t smem = sizeof(Smem<kPair>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tile_m = Cfg<kPair>::kTileM;
  const int tiles = ((a.M + tile_m - 1) / tile_m) * ((a.N + BN - 1) / BN);
  const int per = kPair ? 2 : 1;
  int max_units = num_sms / per;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = per;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;   // the occupancy query below sees the cluster shape only
  if (kPair) {
    // A pair needs two SMs of one GPC; not every SM may find a partner, so a
    // persistent grid is sized by how many pairs can be resident at once.
    static int resident_pairs = 0;
    if (resident_pairs == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(2 * max_units));
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) resident_pairs = n;
      else resident_pairs = max_units;
    }
    if (resident_pairs < max_units) max_units = resident_pairs;
  }
  const int grid = per * (tiles < max_units ? tiles : max_units);
  const uint32_t idesc = idesc_f8f6f4(static_cast<uint32_t>(a.afmt), static_cast<uint32_t>(a.bfmt),
                                      tile_m, BN);
  // TMA stores need a 16-byte aligned D whose row pitch is a multiple of 16
  // bytes; otherwise the store warp copies the staged tile out itself
  const bool tma_out = a.tma_out;
  // keep the smaller operand resident: sweep it inside groups of the larger
  const bool raster_n = static_cast<int64_t>(a.M) < static_cast<int64_t>(a.N);
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.tmD, a.sA, a.sB, a.C, a.D, a.sD, a.M, a.N,
                            a.K, idesc, tma_out, raster_n, a.qmax);
}

template <bool kPair, int kOut>
cudaError_t launch_grans(const Fp8GemmArgs& a, int num_sms, cudaStream_t s) {
  if (a.a_row)
    return a.b_row ? launch_variant<kPair, true, true, kOut>(a, num_sms, s)
                   : launch_variant<kPair, true, false, kOut>(a, num_sms, s);
  return a.b_row ? launch_variant<kPair, false, true, kOut>(a, num_sms, s)
                 : launch_variant<kPair, false, false, kOut>(a, num_sms, s);
}

template <bool kPair>
cudaError_t launch_shape(const Fp8GemmArgs& a, int num_sms, cudaStream_t s) {
  if (a.out_fp8)
    return a.qfmt == 0 ? launch_grans<kPair, kOutE4M3>(a, num_sms, s)
                       : launch_grans<kPair, kOutE5M2>(a, num_sms, s);
  return a.out_bf16 ? launch_grans<kPair, kOutBF16>(a, num_sms, s)
                    : launch_grans<kPair, kOutF32>(a, num_sms, s);
}

}  // namespace

cudaError_t gemm_fp8_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fp8_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_fp8_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

int gemm_fp8_b_box_rows(bool pair) { return pair ? Cfg<true>::kBRows : Cfg<false>::kBRows; }

bool gemm_fp8_use_pair(int M, int N, int num_sms) {
  // Pairs need an even SM count and enough 256 x 256 tiles to fill the GPU.
  // A pair moves two thirds of the single CTA's bytes per FLOP and keeps four
  // stages in flight instead of three; on both large FP8 workloads it is the
  // faster shape.
  const int64_t pair_tiles = (static_cast<int64_t>(M) + 255) / 256 * ((N + BN - 1) / BN);
  return num_sms >= 2 && pair_tiles >= num_sms / 2;
}

cudaError_t launch_gemm_fp8(const Fp8GemmArgs& a, int num_sms, cudaStream_t s) {
  return a.pair ? launch_shape<true>(a, num_sms, s) : launch_shape<false>(a, num_sms, s);
}

}  // namespace bsg

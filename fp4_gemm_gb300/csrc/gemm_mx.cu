// Block-scaled GEMMs for large shapes, for sm_103a: MXFP8, MXFP4, NVFP4.
//
//   D[i][j] = alpha * sum_k (sA(i,k) a[i][k]) (sB(j,k) b[j][k]) + C[i][j]
//
// Three operand kinds share this kernel (kKind):
//   MXFP8  FP8 E4M3/E5M2, UE8M0 per 32 along K, kind::mxf8f6f4 scale_vec::1X
//          (K = 32 per MMA, one scale byte per row); a stage is 128 K.
//   MXFP4  packed E2M1, UE8M0 per 32, kind::mxf4 scale_vec::2X (K = 64 per
//          MMA, two scale bytes); a stage is 256 K = 2 scale atoms per 128
//          rows.
//   NVFP4  packed E2M1, UE4M3 per 16, kind::mxf4nvf4 scale_vec::4X (K = 64,
//          four scale bytes = one atom per MMA); a stage is 256 K = 4 atoms;
//          the sum is multiplied by alpha (the product of the tensor scales).
// In every kind a stage is 128 bytes of each operand row, so the MMA time and
// the bytes moved per stage are the same; the text below describes MXFP8.
//
// The K-blocked scaling of "Rubin FP4 GEMM deep dive" (sections 2.2 and 3.1:
// 32 consecutive K elements share one E8M0 scale, each block's partial sum
// is scaled by 2^(eA+eB) before it is accumulated) with FP8 E4M3 / E5M2
// elements.  tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X applies the
// scales inside the tensor core (K = 32 per instruction = one scale byte per
// row) and accumulates in FP32 tensor memory across all of K, so - unlike the
// per-tile FP32 scales of the FP8 path - no CUDA-core promotion is needed and
// the kernel runs at the tensor core's block-scaled FP8 rate, as long as the
// operands arrive fast enough.
//
// Two shapes of the same kernel (kPair):
//   * single CTA: 128 x 256 output tiles; per stage the SM loads A 16 KB +
//     B 32 KB (4 stages, 3 for NVFP4).
//   * CTA pair (a cluster of two on neighbouring SMs, tcgen05 cta_group::2):
//     256 x 256 tiles.  Each CTA loads its 128 rows of A and 128 of the 256
//     rows of B (32 KB per stage, 6 stages for MXFP8, 5 for the FP4 kinds);
//     one thread of the even CTA issues M = 256 MMAs.  Per FLOP an SM moves
//     two thirds of the single-CTA bytes, which matters because a single
//     CTA needs about 96 bytes per clock from L2 at the MMA's rate, more than
//     the roughly 60 the L2 delivers to each SM.  Each CTA's tensor memory
//     holds the scale factors of its own 128 rows of A and those of all 256
//     rows of B, at the same columns in both CTAs.
// A stage's scale atoms (512 bytes = 128 rows x 4 K-blocks) arrive by bulk
// copies; four scale-writer warps per CTA move them from shared to tensor
// memory with tcgen05.st, into columns owned by that stage (so an in-flight
// MMA never sees them overwritten), and release the stage to the MMA thread.
// (A tcgen05.cp issued by the MMA thread itself would do the same copy, but a
// copy that follows the thread's barrier wait holds up the MMAs behind it by
// about a third of a stage.)  The accumulator takes 256 of the 512 tensor-memory
// columns (the scale columns need the rest), so a tile's accumulator is
// handed to the epilogue warps, which read it into registers at once and
// return it before they convert and store the output; the next tile's MMAs
// wait only for that read, and the stores overlap them.
//
// Warp roles (512 threads = 4 warpgroups, one CTA per SM):
//   warp 0     producer: TMA loads of A and B, bulk copies of the scale atoms.
//   warp 1     tensor-memory allocator; MMA issuer (one lane; in a pair only
//              the even CTA's).
//   warps 2-3  idle (they complete warpgroup 0).
//   warps 4-11 epilogue: warp w reads TMEM lanes 32*(w%4)..+31 and column
//              half (w-4)/4 of the tile, adds C, converts, stores.
//   warps 12-15 scale writers: warp w writes the scales of TMEM lanes
//              32*(w%4)..+31.
// Registers: 512 x 128 at launch; warpgroups 0 and 3 give back to 56, the
// epilogue warpgroups take 200 (128 x 56 + 256 x 200 + 128 x 56 = 65536).
// Every wait is bounded; a wait that runs out sets the error word, raises a
// CTA-wide abort flag and all roles unwind to the final barrier.
#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_mx_error = 0;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kRowBytes = 128;          // bytes of an operand row per stage (128 FP8 / 256 FP4 values)
constexpr int kThreads = 512;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstEpiWarp = 4;
constexpr int kFirstSfWarp = 12;
constexpr int kRegsSmall = 56;
constexpr int kRegsLarge = 200;
static_assert(128 * kRegsSmall * 2 + 256 * kRegsLarge <= kThreads * 128,
              "register split exceeds the launch allocation");
constexpr int kSfAtom = 512;            // 128 rows x 4 K-blocks of E8M0
constexpr int kTmemCols = 512;
constexpr int kAccCols = BN;            // FP32 accumulator columns
constexpr int kGroup = 8;

enum Kind : int { kMxfp8 = 0, kMxfp4 = 1, kNvfp4 = 2 };

// Per kind: scale atoms (512 bytes = 128 rows x 4 scale bytes) per 128 rows
// per stage, the scale block along K, and the tensor-memory columns of a
// stage's scales: A's atoms (4 columns each) from the stage's first column,
// B's from sfb_off; B's K-atom j puts its two 128-row blocks at sfb_off + 8j
// and + 4 (the 256 rows of one N = 256 MMA, 8-column aligned).
template <bool kPair, int kKind>
struct KindCfg {
  static constexpr int kAtoms = kKind == kMxfp8 ? 1 : (kKind == kMxfp4 ? 2 : 4);
  static constexpr int kBlock = kKind == kNvfp4 ? 16 : 32;
  static constexpr int kSfbOff = kAtoms * 4 > 8 ? kAtoms * 4 : 8;
  static constexpr int kSfColsPerStage = kSfbOff + 8 * kAtoms;
  static constexpr int kBRows = kPair ? BN / 2 : BN;      // B rows this CTA loads
  static constexpr int kTileM = kPair ? 2 * BM : BM;      // rows of a tile
  // single CTA: NVFP4's 6 KB of scales per stage leave room for three
  // stages; a pair CTA's 32 KB stages fit six (MXFP8) or five (FP4 kinds)
  static constexpr int kStages = kPair ? (kKind == kMxfp8 ? 6 : 5) : (kKind == kNvfp4 ? 3 : 4);
  static constexpr int kEpiArrivals = kPair ? 16 : 8;     // accumulator reads per tile
  static constexpr int kSfArrivals = kPair ? 8 : 4;       // scale writers per stage
  static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory columns");
};

template <bool kPair, int kKind>
struct __align__(1024) Smem {
  using KC = KindCfg<kPair, kKind>;
  static constexpr int S = KC::kStages;
  static constexpr int A = KC::kAtoms;
  uint8_t a[S][BM * kRowBytes];
  uint8_t b[S][KC::kBRows * kRowBytes];
  uint8_t epi[8][32 * 64];     // per epilogue warp: 32 rows x 64 B output staging
  uint8_t sfa[S][A * kSfAtom];
  uint8_t sfb[S][2][A * kSfAtom];   // B's two 128-row blocks
  uint64_t full[S];           // operands (pair: both CTAs', on the even CTA's barrier)
  uint64_t sfl[S];            // pair: this CTA's scale atoms landed
  uint64_t sready[S];         // the stage's scales are in tensor memory
  uint64_t done[S];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t final_bar;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
};

struct TileCoord {
  int m, n;
};

// Persistent raster: groups of kGroup tiles along the larger operand, the
// smaller operand swept inside a group (it stays resident in L2).
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

__device__ __forceinline__ void raise_abort(volatile uint32_t* flag) {
  atomicOr(&g_mx_error, kErrTimeout);
  *flag = 1u;
}

template <bool kPair, bool kBF16Out, int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ sfA, const uint8_t* __restrict__ sfB,
                   const float* __restrict__ Cin, void* __restrict__ Dout, int M, int N, int K,
                   uint32_t idesc_base, bool vec_out, bool raster_n, float alpha) {
  using KC = KindCfg<kPair, kKind>;
  constexpr int kStages = KC::kStages;
  constexpr int kAtoms = KC::kAtoms;
  constexpr int kSfColsPerStage = KC::kSfColsPerStage;
  extern __shared__ uint8_t smem_raw[];
  Smem<kPair, kKind>& sm = *reinterpret_cast<Smem<kPair, kKind>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;      // 0 = the pair's MMA issuer
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int num_m = (M + KC::kTileM - 1) / KC::kTileM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int kbytes = kKind == kMxfp8 ? K : K / 2;  // operand bytes per row
  const int KS = (kbytes + kRowBytes - 1) / kRowBytes;   // stages along K
  const int KA = (K / KC::kBlock + 3) / 4;          // scale atoms along K
  const int num_nb = (N + 127) / 128;               // 128-row blocks of B

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.sfl[s]), 1);
      mbar_init(smem_u32(&sm.sready[s]), KC::kSfArrivals);
      mbar_init(smem_u32(&sm.done[s]), 1);
    }
    mbar_init(smem_u32(&sm.tfull), 1);
    mbar_init(smem_u32(&sm.tempty), KC::kEpiArrivals);
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
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();    // barriers and tensor memory of both CTAs are ready
  tc_fence_after();
  grid_dep_launch();
  grid_dep_wait();
  const uint32_t tmem = sm.tmem_base;
  // where this CTA signals the issuing CTA: the even CTA's barriers
  const uint32_t sready0 = kPair ? mapa_shared(smem_u32(&sm.sready[0]), 0) : smem_u32(&sm.sready[0]);
  const uint32_t tempty0 = kPair ? mapa_shared(smem_u32(&sm.tempty), 0) : smem_u32(&sm.tempty);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();   // operands are re-read by other tiles
      uint32_t it = 0;
      bool ok = true;
      for (int t = unit; t < tiles && ok; t += units) {
        const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
        const int m_cta = tc.m * KC::kTileM + static_cast<int>(rank) * BM;   // this CTA's rows
        const int n_b = tc.n * BN + static_cast<int>(rank) * KC::kBRows;   // its B rows
        const int nbv = (2 * tc.n + 1 < num_nb) ? 2 : 1;   // scale atoms of B that exist
        for (int ks = 0; ks < KS; ++ks, ++it) {
          if (sm.abort_flag) { ok = false; break; }
          const int s = static_cast<int>(it % kStages);
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait(smem_u32(&sm.done[s]), ph ^ 1u)) {
            raise_abort(&sm.abort_flag);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&sm.full[s]);
          const int ka0 = ks * kAtoms;
          const int na = min(kAtoms, KA - ka0);               // atoms of this stage
          const uint32_t sf_bytes = static_cast<uint32_t>((1 + nbv) * na * kSfAtom);
          // the scale atoms complete on full (single CTA) or on this CTA's
          // own sfl barrier (pair: the operands complete on the even CTA's)
          const uint32_t sb = kPair ? smem_u32(&sm.sfl[s]) : fb;
          if (kPair) {
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (BM + KC::kBRows) * kRowBytes);
            const uint32_t fb0 = mapa_shared(fb, 0);
            tma_load_2d_pair(smem_u32(sm.a[s]), &tmA, fb0, ks * kRowBytes, m_cta, keep);
            tma_load_2d_pair(smem_u32(sm.b[s]), &tmB, fb0, ks * kRowBytes, n_b, keep);
            mbar_arrive_expect_tx(sb, sf_bytes);
          } else {
            mbar_arrive_expect_tx(fb, (BM + BN) * kRowBytes + sf_bytes);
            tma_load_2d_hint(smem_u32(sm.a[s]), &tmA, fb, ks * kRowBytes, m_cta, keep);
            tma_load_2d_hint(smem_u32(sm.b[s]), &tmB, fb, ks * kRowBytes, n_b, keep);
          }
          // a row block's atoms along K are contiguous: one copy per block
          bulk_load(smem_u32(sm.sfa[s]), sfA + (static_cast<int64_t>(m_cta / BM) * KA + ka0) * kSfAtom,
                    na * kSfAtom, sb);
          for (int j = 0; j < nbv; ++j)
            bulk_load(smem_u32(sm.sfb[s][j]),
                      sfB + (static_cast<int64_t>(2 * tc.n + j) * KA + ka0) * kSfAtom, na * kSfAtom, sb);
        }
      }
      // the even CTA's full barriers also count the peer's bytes
      if (rank == 0) drain_fills(sm.full, kStages, it);
      if (kPair) drain_fills(sm.sfl, kStages, it);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0 && rank == 0) {
      // The MMA queue holds little more than the running MMA, so the thread
      // must issue a stage's first MMA while the previous stage's last two
      // still run: everything that depends on the stage slot is a base plus
      // the slot times a constant stride, and the slot and its phase parity
      // advance by increments, so that little but the MMAs themselves lies
      // between two stages.
      const uint64_t ad0 = sdesc_kmajor_sw128(smem_u32(sm.a[0]));
      const uint64_t bd0 = sdesc_kmajor_sw128(smem_u32(sm.b[0]));
      constexpr uint32_t kADescStep = (BM * kRowBytes) >> 4;   // descriptor address units (16 B)
      constexpr uint32_t kBDescStep = (KC::kBRows * kRowBytes) >> 4;
      const uint32_t sf0 = tmem + kAccCols;
      const int rem_last = kbytes - (KS - 1) * kRowBytes;     // 32 bytes per MMA
      const int nk_last = rem_last >= kRowBytes ? 4 : (rem_last + 31) / 32;
      uint32_t s = 0, ph = 0, tl = 0;    // slot and phase parity of the next stage
      bool ok = true;
      bool next_ready = false;           // the next stage's scales are known to be in place
      for (int t = unit; t < tiles && ok; t += units, ++tl) {
        // A stage may start once its operands have landed (the scale writers
        // waited for the stage's TMA) and its scales are in tensor memory.
        // A non-blocking test of the next stage goes after this stage's
        // second MMA and, if it passed, the fence after its third, where they
        // hide under running MMAs; the commit that frees this stage follows
        // its last MMA at once (deferring it would delay the stage's refill);
        // a wait that may block comes only after it, when the test failed.
        // A tile's last stage tests the next tile's first, so that a new tile
        // waits only for the epilogue to have read the accumulator.
        if (!mbar_wait(smem_u32(&sm.tempty), (tl & 1u) ^ 1u) ||
            (!next_ready && (sm.abort_flag || !mbar_wait(smem_u32(&sm.sready[s]), ph)))) {
          raise_abort(&sm.abort_flag);
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < KS && ok; ++ks) {
          const uint32_t sfa_t = sf0 + s * kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + KC::kSfbOff;
          const uint64_t ad = ad0 + s * kADescStep;
          const uint64_t bd = bd0 + s * kBDescStep;
          const bool more = ks + 1 < KS;
          const int nk = more ? 4 : nk_last;
          const uint32_t s1 = s + 1 == static_cast<uint32_t>(kStages) ? 0u : s + 1;
          const uint32_t ph1 = s1 == 0 ? ph ^ 1u : ph;
          next_ready = false;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (kk < nk) {
              const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
              if (kKind == kMxfp8) {
                // K block kk of the atom: scale byte kk of each row's cell
                const uint32_t id = idesc_base | (static_cast<uint32_t>(kk) << 4) |
                                    (static_cast<uint32_t>(kk) << 29);
                if (kPair)
                  mma_mxf8_pair(tmem, ad + 2 * kk, bd + 2 * kk, id, sfa_t, sfb_t, acc);
                else
                  mma_mxf8(tmem, ad + 2 * kk, bd + 2 * kk, id, sfa_t, sfb_t, acc);
              } else if (kKind == kMxfp4) {
                // K = 64: half of atom kk / 2, bytes 0-1 or 2-3 of each cell
                const uint32_t sid = static_cast<uint32_t>((kk & 1) * 2);
                const uint32_t id = idesc_base | (sid << 4) | (sid << 29);
                if (kPair)
                  mma_mxf4_pair(tmem, ad + 2 * kk, bd + 2 * kk, id, sfa_t + 4 * (kk >> 1),
                                sfb_t + 8 * (kk >> 1), acc);
                else
                  mma_mxf4(tmem, ad + 2 * kk, bd + 2 * kk, id, sfa_t + 4 * (kk >> 1),
                           sfb_t + 8 * (kk >> 1), acc);
              } else {
                // K = 64: all four bytes of atom kk
                if (kPair)
                  mma_nvf4_pair(tmem, ad + 2 * kk, bd + 2 * kk, idesc_base, sfa_t + 4 * kk,
                                sfb_t + 8 * kk, acc);
                else
                  mma_nvf4(tmem, ad + 2 * kk, bd + 2 * kk, idesc_base, sfa_t + 4 * kk, sfb_t + 8 * kk,
                           acc);
              }
            }
            if (kk == 1) next_ready = mbar_test(smem_u32(&sm.sready[s1]), ph1);
            if (kk == 2 && next_ready) tc_fence_after();
          }
          if (kPair)
            tc_commit_pair_mc(smem_u32(&sm.done[s]), 3);
          else
            tc_commit(smem_u32(&sm.done[s]));
          if (more && !next_ready) {
            if (!mbar_wait(smem_u32(&sm.sready[s1]), ph1)) {
              raise_abort(&sm.abort_flag);
              ok = false;
            }
            tc_fence_after();
          }
          s = s1;
          ph = ph1;
        }
        if (!ok) break;
        if (kPair)
          tc_commit_pair_mc(smem_u32(&sm.tfull), 3);
        else
          tc_commit(smem_u32(&sm.tfull));
      }
      if (kPair)
        tc_commit_pair(smem_u32(&sm.final_bar));
      else
        tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(&sm.abort_flag);
    }
    __syncwarp();
  } else if (warp >= kFirstSfWarp) {
    // ------------------------------------------------------ scale writers
    // Tensor-memory lane 32q + i, columns c..c+3 of an atom hold the 16
    // bytes of row i of the 512-byte atom in shared memory (the 32-lane
    // pattern a 32x128b warpx4 copy replicates to all four lane quarters).
    // Pair: each CTA's writers wait for their own scale atoms (sfl); the
    // even CTA's also wait for both CTAs' operands (full), so the issuer's
    // sready barrier - all eight writer warps - means the stage is ready.
    setmaxnreg_dec<kRegsSmall>();
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units) {
      for (int ks = 0; ks < KS; ++ks, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        bool good = true;
        if (kPair) {
          good = mbar_wait(smem_u32(&sm.sfl[s]), ph) && (rank != 0 || mbar_wait(smem_u32(&sm.full[s]), ph));
        } else {
          good = mbar_wait(smem_u32(&sm.full[s]), ph);
        }
        if (!good) {
          raise_abort(&sm.abort_flag);
          ok = false;
          break;
        }
        const uint32_t sfa_t = tmem + lane_off + kAccCols + s * kSfColsPerStage;
        const uint32_t sfb_t = sfa_t + KC::kSfbOff;
        const int na = min(kAtoms, KA - ks * kAtoms);
#pragma unroll
        for (int a = 0; a < kAtoms; ++a) {
          if (a < na) {
            tmem_st_4(sfa_t + 4 * a, ld_shared_v4(smem_u32(sm.sfa[s]) + a * kSfAtom + lane * 16));
            tmem_st_4(sfb_t + 8 * a, ld_shared_v4(smem_u32(sm.sfb[s][0]) + a * kSfAtom + lane * 16));
            tmem_st_4(sfb_t + 8 * a + 4, ld_shared_v4(smem_u32(sm.sfb[s][1]) + a * kSfAtom + lane * 16));
          }
        }
        // tcgen05.wait::st returns once the stores are in tensor memory, so
        // the arrive has nothing left to publish: a relaxed arrive suffices.
        // (A release arrive at cluster scope would first wait until every
        // earlier memory operation is visible cluster-wide, which costs more
        // than a whole stage while the epilogue's output stores are in
        // flight.)
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(sready0 + s * 8);
      }
    }
  } else if (warp >= kFirstEpiWarp) {
    // ----------------------------------------------------------- epilogue
    setmaxnreg_inc<kRegsLarge>();
    const int q = warp & 3;
    const int g = (warp - kFirstEpiWarp) >> 2;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + g * 128;
    const uint64_t stream_out = l2_policy_evict_first();   // the result is not re-read
    uint32_t tl = 0;
    for (int t = unit; t < tiles; t += units, ++tl) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      if (sm.abort_flag || !mbar_wait(smem_u32(&sm.tfull), tl & 1u)) {
        if (!sm.abort_flag) raise_abort(&sm.abort_flag);
        break;
      }
      tc_fence_after();
      // the whole 128-column half of this warp's 32 rows into registers, then
      // the accumulator goes straight back to the MMA
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32(taddr + c * 32, r[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tc_wait_ld_32(r[c]);
      tc_fence_before();
      __syncwarp();
      // every tcgen05.ld of the accumulator has completed: nothing to
      // publish, so a relaxed arrive suffices
      if (lane == 0) mbar_arrive_relaxed(tempty0);
      // The accumulator is back with the MMA, so the stores below overlap
      // the next tile.  The warp passes its 32 rows through a 32 x 64-byte
      // staging buffer (16-byte pieces XOR-swizzled by row, so both phases
      // are bank-conflict free) and writes 8 rows x 64 contiguous bytes per
      // store instruction instead of 32 scattered 16-byte pieces.
      constexpr int kElem = kBF16Out ? 2 : 4;
      constexpr int kColsPerChunk = 64 / kElem;     // 32 (BF16) or 16 (FP32)
      constexpr int kPerPiece = 16 / kElem;
      const int64_t row0 = static_cast<int64_t>(tc.m) * KC::kTileM + rank * BM + q * 32;
      const int gcol0 = tc.n * BN + g * 128;
      const uint32_t stage = smem_u32(sm.epi[warp - kFirstEpiWarp]);
      const int64_t my_row = row0 + lane;
#pragma unroll
      for (int ch = 0; ch < 128 / kColsPerChunk; ++ch) {
        const int col0 = gcol0 + ch * kColsPerChunk;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          float v[kPerPiece];
#pragma unroll
          for (int j = 0; j < kPerPiece; ++j) {
            const int col = ch * kColsPerChunk + p * kPerPiece + j;
            v[j] = __uint_as_float(r[col / 32][col % 32]);
          }
          // alpha * acc + C with one rounding (NVFP4), acc + C otherwise:
          // written out so that the compiler's contraction choices do not
          // decide the result bits
          const bool add_c = Cin != nullptr && my_row < M;
#pragma unroll
          for (int j = 0; j < kPerPiece; ++j) {
            const int col = col0 + p * kPerPiece + j;
            const float c = (add_c && col < N) ? __ldg(Cin + my_row * N + col) : 0.0f;
            if (kKind == kNvfp4)
              v[j] = add_c ? __fmaf_rn(v[j], alpha, c) : __fmul_rn(v[j], alpha);
            else if (add_c)
              v[j] = __fadd_rn(v[j], c);
          }
          uint4 u;
          if (kBF16Out) {
            u.x = pack_bf16x2(v[0], v[1]);
            u.y = pack_bf16x2(v[2], v[3]);
            u.z = pack_bf16x2(v[4 % kPerPiece], v[5 % kPerPiece]);
            u.w = pack_bf16x2(v[6 % kPerPiece], v[7 % kPerPiece]);
          } else {
            u = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                           __float_as_uint(v[2 % kPerPiece]), __float_as_uint(v[3 % kPerPiece]));
          }
          st_shared_v4(stage + lane * 64 + ((p ^ ((lane >> 1) & 3)) << 4), u);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 8 * i + (lane >> 2);
          const int p = lane & 3;
          const uint4 u = ld_shared_v4(stage + rr * 64 + ((p ^ ((rr >> 1) & 3)) << 4));
          const int64_t grow = row0 + rr;
          const int col = col0 + p * kPerPiece;
          if (grow < M && col < N) {
            if (vec_out && col + kPerPiece <= N) {
              st_global_v4_hint(static_cast<uint8_t*>(Dout) + (grow * N + col) * kElem, u, stream_out);
            } else {
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int j = 0; j < kPerPiece; ++j) {
                if (col + j >= N) break;
                if (kBF16Out)
                  reinterpret_cast<uint16_t*>(Dout)[grow * N + col + j] =
                      static_cast<uint16_t>(w[j / 2] >> (16 * (j % 2)));
                else
                  reinterpret_cast<float*>(Dout)[grow * N + col + j] = __uint_as_float(w[j]);
              }
            }
          }
        }
        __syncwarp();
      }
    }
  } else {
    setmaxnreg_dec<kRegsSmall>();            // idle warp of warpgroup 0
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

template <bool kPair, bool kBF16Out, int kKind>
cudaError_t launch_variant(const MxGemmArgs& a, int num_sms, cudaStream_t s) {
  using KC = KindCfg<kPair, kKind>;
  auto kern = gemm_mx_kernel<kPair, kBF16Out, kKind>;
  static_assert(sizeof(Smem<kPair, kKind>) + 1024 <= 227 * 1024, "shared memory per CTA");
  const size_t smem = sizeof(Smem<kPair, kKind>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + KC::kTileM - 1) / KC::kTileM) * ((a.N + BN - 1) / BN);
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
  // keep the smaller operand resident: sweep it inside groups of the larger
  const bool raster_n = a.M < a.N;
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) &&
                       (a.out_bf16 ? (a.N % 8 == 0) : (a.N % 4 == 0));
  const uint32_t tile_m = static_cast<uint32_t>(KC::kTileM);
  const uint32_t idesc = kKind == kMxfp8   ? idesc_mxf8(static_cast<uint32_t>(a.afmt), static_cast<uint32_t>(a.bfmt),
                                                        tile_m, BN, 0u, 0u)
                         : kKind == kMxfp4 ? idesc_mxf4(tile_m, BN, 0u, 0u)
                                           : idesc_nvf4(tile_m, BN);
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.sfA, a.sfB, a.C, a.D, a.M, a.N, a.K, idesc,
                            vec_out, raster_n, a.alpha);
}

}  // namespace

cudaError_t gemm_mx_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_mx_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_mx_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

int gemm_mx_b_box_rows(bool pair) { return pair ? BN / 2 : BN; }

bool gemm_mx_fp4_large(int M, int N, int num_sms) {
  // the 128 x 256 kernel once there are at least half as many tiles as SMs;
  // smaller FP4 problems keep the 128 x 128 general kernel (more CTAs)
  const int64_t tiles = (static_cast<int64_t>(M) + BM - 1) / BM * ((N + BN - 1) / BN);
  return tiles >= num_sms / 2;
}

bool gemm_mx_use_pair(int M, int N, int num_sms) {
  // pairs need an even SM count and enough 256 x 256 tiles to fill the GPU
  const int64_t pair_tiles = (static_cast<int64_t>(M) + 2 * BM - 1) / (2 * BM) * ((N + BN - 1) / BN);
  return num_sms >= 2 && pair_tiles >= num_sms / 2;
}

namespace {
template <bool kPair>
cudaError_t launch_kind(const MxGemmArgs& a, int num_sms, cudaStream_t s) {
  switch (a.kind) {
    case kMxfp4:
      return a.out_bf16 ? launch_variant<kPair, true, kMxfp4>(a, num_sms, s)
                        : launch_variant<kPair, false, kMxfp4>(a, num_sms, s);
    case kNvfp4:
      return a.out_bf16 ? launch_variant<kPair, true, kNvfp4>(a, num_sms, s)
                        : launch_variant<kPair, false, kNvfp4>(a, num_sms, s);
    default:
      return a.out_bf16 ? launch_variant<kPair, true, kMxfp8>(a, num_sms, s)
                        : launch_variant<kPair, false, kMxfp8>(a, num_sms, s);
  }
}
}  // namespace

cudaError_t launch_gemm_mx(const MxGemmArgs& a, int num_sms, cudaStream_t s) {
  return a.pair ? launch_kind<true>(a, num_sms, s) : launch_kind<false>(a, num_sms, s);
}

}  // namespace bsg

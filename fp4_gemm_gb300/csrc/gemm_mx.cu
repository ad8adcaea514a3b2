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
// the kernel runs at the tensor core's block-scaled FP8 rate.
//
// One CTA per SM, persistent over 128 x 256 output tiles; per pipeline stage
// 128 K (A 16 KB + B 32 KB + one 512-byte E8M0 scale atom of A and two of B,
// all brought by TMA / bulk copies on one barrier; 4 stages).  Four
// scale-writer warps move the stage's scale atoms from shared to tensor
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
// Warp roles (512 threads = 4 warpgroups):
//   warp 0     producer: TMA loads of A and B, bulk copies of the scale atoms.
//   warp 1     tensor-memory allocator; MMA issuer (one lane).
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
template <int kKind>
struct KindCfg {
  static constexpr int kAtoms = kKind == kMxfp8 ? 1 : (kKind == kMxfp4 ? 2 : 4);
  static constexpr int kBlock = kKind == kNvfp4 ? 16 : 32;
  static constexpr int kSfbOff = kAtoms * 4 > 8 ? kAtoms * 4 : 8;
  static constexpr int kSfColsPerStage = kSfbOff + 8 * kAtoms;
  // NVFP4's 6 KB of scales per stage leave room for three stages
  static constexpr int kStages = kKind == kNvfp4 ? 3 : 4;
  static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory columns");
};

template <int kKind>
struct __align__(1024) Smem {
  static constexpr int S = KindCfg<kKind>::kStages;
  static constexpr int A = KindCfg<kKind>::kAtoms;
  uint8_t a[S][BM * kRowBytes];
  uint8_t b[S][BN * kRowBytes];
  uint8_t epi[8][32 * 64];     // per epilogue warp: 32 rows x 64 B output staging
  uint8_t sfa[S][A * kSfAtom];
  uint8_t sfb[S][2][A * kSfAtom];   // B's two 128-row blocks
  uint64_t full[S];
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

template <bool kBF16Out, int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ sfA, const uint8_t* __restrict__ sfB,
                   const float* __restrict__ Cin, void* __restrict__ Dout, int M, int N, int K,
                   uint32_t afmt, uint32_t bfmt, bool vec_out, bool raster_n, float alpha) {
  using KC = KindCfg<kKind>;
  constexpr int kStages = KC::kStages;
  constexpr int kAtoms = KC::kAtoms;
  constexpr int kSfColsPerStage = KC::kSfColsPerStage;
  extern __shared__ uint8_t smem_raw[];
  Smem<kKind>& sm = *reinterpret_cast<Smem<kKind>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int kbytes = kKind == kMxfp8 ? K : K / 2;  // operand bytes per row
  const int KS = (kbytes + kRowBytes - 1) / kRowBytes;   // stages along K
  const int KA = (K / KC::kBlock + 3) / 4;          // scale atoms along K
  const int num_nb = (N + 127) / 128;               // 128-row blocks of B

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.sready[s]), 4);
      mbar_init(smem_u32(&sm.done[s]), 1);
    }
    mbar_init(smem_u32(&sm.tfull), 1);
    mbar_init(smem_u32(&sm.tempty), 8);
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
  grid_dep_launch();
  grid_dep_wait();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();   // operands are re-read by other tiles
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
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
          mbar_arrive_expect_tx(fb, (BM + BN) * kRowBytes + (1 + nbv) * na * kSfAtom);
          tma_load_2d_hint(smem_u32(sm.a[s]), &tmA, fb, ks * kRowBytes, tc.m * BM, keep);
          tma_load_2d_hint(smem_u32(sm.b[s]), &tmB, fb, ks * kRowBytes, tc.n * BN, keep);
          // a row block's atoms along K are contiguous: one copy per block
          bulk_load(smem_u32(sm.sfa[s]), sfA + (static_cast<int64_t>(tc.m) * KA + ka0) * kSfAtom,
                    na * kSfAtom, fb);
          for (int j = 0; j < nbv; ++j)
            bulk_load(smem_u32(sm.sfb[s][j]),
                      sfB + (static_cast<int64_t>(2 * tc.n + j) * KA + ka0) * kSfAtom, na * kSfAtom, fb);
        }
      }
      drain_fills(sm.full, kStages, it);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0) {
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tl) {
        // the epilogue has read the previous tile's accumulator
        if (!mbar_wait(smem_u32(&sm.tempty), (tl & 1u) ^ 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        tc_fence_after();
        // A stage may start once its operands have landed (the scale writers
        // waited for the stage's TMA) and its scales are in tensor memory.
        // The MMA queue holds little more than the running MMA, so work
        // between two stages' MMAs can leave the tensor core idle: the wait
        // for stage it+1 is issued after stage it's second MMA and the fence
        // after its third, where they hide under running MMAs; the commit
        // that frees stage it follows its last MMA at once (deferring it
        // would delay the stage's refill, which the ring of four stages
        // cannot afford).
        if (sm.abort_flag || !mbar_wait(smem_u32(&sm.sready[it % kStages]), (it / kStages) & 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < KS && ok; ++ks, ++it) {
          const int s = static_cast<int>(it % kStages);
          const uint32_t sfa_t = tmem + kAccCols + s * kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + KC::kSfbOff;
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm.a[s]));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sm.b[s]));
          const int rem = kbytes - ks * kRowBytes;           // 32 bytes per MMA
          const int nk = rem >= kRowBytes ? 4 : (rem + 31) / 32;
          const bool more = ks + 1 < KS;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (kk < nk) {
              const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
              if (kKind == kMxfp8) {
                // K block kk of the atom: scale byte kk of each row's cell
                mma_mxf8(tmem, ad + 2 * kk, bd + 2 * kk,
                         idesc_mxf8(afmt, bfmt, BM, BN, static_cast<uint32_t>(kk), static_cast<uint32_t>(kk)),
                         sfa_t, sfb_t, acc);
              } else if (kKind == kMxfp4) {
                // K = 64: half of atom kk / 2, bytes 0-1 or 2-3 of each cell
                const uint32_t id = static_cast<uint32_t>((kk & 1) * 2);
                mma_mxf4(tmem, ad + 2 * kk, bd + 2 * kk, idesc_mxf4(BM, BN, id, id),
                         sfa_t + 4 * (kk >> 1), sfb_t + 8 * (kk >> 1), acc);
              } else {
                // K = 64: all four bytes of atom kk
                mma_nvf4(tmem, ad + 2 * kk, bd + 2 * kk, idesc_nvf4(BM, BN), sfa_t + 4 * kk,
                         sfb_t + 8 * kk, acc);
              }
            }
            if (kk == 1 && more &&
                !mbar_wait(smem_u32(&sm.sready[(it + 1) % kStages]), ((it + 1) / kStages) & 1u)) {
              raise_abort(&sm.abort_flag);
              ok = false;
            }
            if (kk == 2 && more) tc_fence_after();
          }
          tc_commit(smem_u32(&sm.done[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.tfull));
      }
      tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(&sm.abort_flag);
    }
    __syncwarp();
  } else if (warp >= kFirstSfWarp) {
    // ------------------------------------------------------ scale writers
    // Tensor-memory lane 32q + i, columns c..c+3 of an atom hold the 16
    // bytes of row i of the 512-byte atom in shared memory (the 32-lane
    // pattern a 32x128b warpx4 copy replicates to all four lane quarters).
    setmaxnreg_dec<kRegsSmall>();
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      for (int ks = 0; ks < KS; ++ks, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        if (!mbar_wait(smem_u32(&sm.full[s]), ph)) {
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
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.sready[s]));
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
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
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
      if (lane == 0) mbar_arrive(smem_u32(&sm.tempty));
      // The accumulator is back with the MMA, so the stores below overlap
      // the next tile.  The warp passes its 32 rows through a 32 x 64-byte
      // staging buffer (16-byte pieces XOR-swizzled by row, so both phases
      // are bank-conflict free) and writes 8 rows x 64 contiguous bytes per
      // store instruction instead of 32 scattered 16-byte pieces.
      constexpr int kElem = kBF16Out ? 2 : 4;
      constexpr int kColsPerChunk = 64 / kElem;     // 32 (BF16) or 16 (FP32)
      constexpr int kPerPiece = 16 / kElem;
      const int64_t row0 = static_cast<int64_t>(tc.m) * BM + q * 32;
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
            if (kKind == kNvfp4) v[j] *= alpha;
          }
          if (Cin != nullptr && my_row < M) {
#pragma unroll
            for (int j = 0; j < kPerPiece; ++j) {
              const int col = col0 + p * kPerPiece + j;
              if (col < N) v[j] += __ldg(Cin + my_row * N + col);
            }
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kBF16Out, int kKind>
cudaError_t launch_variant(const MxGemmArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gemm_mx_kernel<kBF16Out, kKind>;
  static_assert(sizeof(Smem<kKind>) + 1024 <= 227 * 1024, "shared memory per CTA");
  const size_t smem = sizeof(Smem<kKind>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  // keep the smaller operand resident: sweep it inside groups of the larger
  const bool raster_n = a.M < a.N;
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) &&
                       (a.out_bf16 ? (a.N % 8 == 0) : (a.N % 4 == 0));
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, s, a.tmA, a.tmB,
                    a.sfA, a.sfB, a.C, a.D, a.M, a.N, a.K, static_cast<uint32_t>(a.afmt),
                    static_cast<uint32_t>(a.bfmt), vec_out, raster_n, a.alpha);
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

int gemm_mx_b_box_rows() { return BN; }

bool gemm_mx_fp4_large(int M, int N, int num_sms) {
  // the 128 x 256 kernel once there are at least half as many tiles as SMs;
  // smaller FP4 problems keep the 128 x 128 general kernel (more CTAs)
  const int64_t tiles = (static_cast<int64_t>(M) + BM - 1) / BM * ((N + BN - 1) / BN);
  return tiles >= num_sms / 2;
}

cudaError_t launch_gemm_mx(const MxGemmArgs& a, int num_sms, cudaStream_t s) {
  switch (a.kind) {
    case kMxfp4:
      return a.out_bf16 ? launch_variant<true, kMxfp4>(a, num_sms, s)
                        : launch_variant<false, kMxfp4>(a, num_sms, s);
    case kNvfp4:
      return a.out_bf16 ? launch_variant<true, kNvfp4>(a, num_sms, s)
                        : launch_variant<false, kNvfp4>(a, num_sms, s);
    default:
      return a.out_bf16 ? launch_variant<true, kMxfp8>(a, num_sms, s)
                        : launch_variant<false, kMxfp8>(a, num_sms, s);
  }
}

}  // namespace bsg

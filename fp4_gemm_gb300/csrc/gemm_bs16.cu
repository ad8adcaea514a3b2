// FP4 GEMM with 16-bit block scales, promoted per 32-wide K block, for
// sm_103a.
//
//   D[i][j] = sum_kb fl32(s_A(i,kb) * s_B(j,kb)) * P_kb[i][j] + C[i][j]
//   P_kb    = sum_{k in block kb} a[i][k] * b[j][k]        (32-wide K blocks)
//
// "Rubin FP4 GEMM deep dive", section 3.2: where the power-of-two E8M0 block
// scale is too coarse, the scale of each block of 32 E2M1 values may be kept
// in BF16 or FP16.  The tensor core's block-scaled kinds take only UE8M0 /
// UE4M3 scales, so these scales are applied outside it, the way the FP8 path
// applies its FP32 tile scales ("FP8 GEMM on CDNA4", section 4.4, per K
// block): every 32-wide K block is one tcgen05.mma kind::f8f6f4 with E2M1
// operands (K = 32, no accumulation across blocks) into one of two tensor-
// memory buffers, and CUDA-core warps drain it and promote
//     acc = fma(s_A * s_B, P_kb, acc)
// into FP32 registers.  Both factors are exact: an E2M1 partial over 32
// elements is a multiple of 1/4 below 2^11, and s_A * s_B has at most 22
// significant bits; so the result depends only on the FMA order (blocks in
// K order), which makes it reproducible bit for bit.
//
// The operands stay packed in global memory (two E2M1 values per byte, first
// in the low nibble).  The tensor map's 16U4_ALIGN16B type unpacks them on
// the way into shared memory - each 16 values become 8 data bytes and an
// 8-byte gap - which is the layout kind::f8f6f4 reads E2M1 operands in, so a
// 128-element K stage occupies 128 bytes per row like an FP8 stage.
//
// Where the time goes: per output element and K block the drain needs one
// 4-byte tensor-memory read and two FP32 operations (the scale product and
// the FMA), against 64 tensor-core FLOPs.  The FP32 pipe (128 lanes per SM)
// therefore bounds the kernel near a quarter of the FP8 MMA rate; the
// tensor core idles most of the time.  What matters is keeping the FP32
// pipe fed: three drain warps per SM sub-partition, each with 64 columns
// (64 accumulators), so one warp's waits and load latencies overlap the
// others' arithmetic.
//
// Warp roles (512 threads, one CTA per SM, persistent over 128 x 192 tiles):
//   warp 0     producer: TMA loads of A (128 rows) and B (192 rows), one
//              128-element K stage at a time, into a 4-stage ring.
//   warp 1     tensor-memory allocator; MMA issuer (one lane): per K block
//              one M128 N192 K32 MMA into buffer (block & 1), a commit to
//              that buffer's pfull barrier, and after a stage's fourth block
//              a commit to the stage's done barrier.
//   warp 2     scale loader: each stage's A and B block scales (16-bit codes,
//              [K/32][rows] in global memory) into a 4-slot shared-memory
//              ring, by bulk copies when the rows are whole 16-byte pieces
//              (else by plain loads); the drain warps convert the codes as
//              they use them.
//   warps 4-15 drain + epilogue: warp w drains TMEM lanes 32 (w % 4) .. +31
//              (its rows) and column group (w - 4) / 4 (64 columns) of the
//              192-wide tile into 64 FP32 accumulators per thread; after the
//              last block the thread adds C and stores its 64 outputs.
// Every wait is bounded; a wait that runs out sets the error word, raises a
// CTA-wide abort flag and every role unwinds to the final barrier.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_bs16_error = 0;

constexpr int BM = 128;             // output rows per tile
constexpr int BN = 192;             // output columns per tile
constexpr int kGroupCols = 64;      // columns per drain warp
constexpr int BKS = 128;            // K elements per shared-memory stage
constexpr int KBLK = 32;            // K elements per scale block = per MMA
constexpr int kBlocksPerStage = BKS / KBLK;
constexpr int kStages = 4;
constexpr int kScaleSlots = 4;
constexpr int kThreads = 512;
constexpr int kDrainWarps = 12;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp = 2;
constexpr int kFirstDrainWarp = 4;
constexpr int kRegsSmall = 56;
constexpr int kRegsLarge = 152;
static_assert(128 * kRegsSmall + 32 * kDrainWarps * kRegsLarge <= kThreads * 128,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;      // two 192-column FP32 partial buffers
constexpr int kBufStride = 256;     // buffer b starts at column 256 b
constexpr int kGroup = 8;           // tile raster: groups of 8 tiles along M

// Bytes the TMA moves per stage: the packed operands (half a byte per
// element), not the unpacked shared-memory footprint.
constexpr uint32_t kStageTxBytes = (BM + BN) * BKS / 2;

struct __align__(1024) Smem {
  uint8_t a[kStages][BM * BKS];       // unpacked: 128 bytes per row per stage
  uint8_t b[kStages][BN * BKS];
  uint16_t sa[kScaleSlots][kBlocksPerStage][BM];     // scale codes as stored in global memory
  uint16_t sb[kScaleSlots][kBlocksPerStage][BN];
  uint64_t full[kStages];
  uint64_t done[kStages];             // the stage's MMAs completed: slot free
  uint64_t pfull[2];                  // partial of the block in buffer b ready
  uint64_t tempty[2];                 // buffer b drained
  uint64_t sfull[kScaleSlots];
  uint64_t sempty[kScaleSlots];
  uint64_t final_bar;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
};

struct TileCoord {
  int m, n;
};

// Tiles are visited in groups of kGroup rows of tiles while N is swept, so
// the A panel of a group stays in L2 while B streams past it.
__device__ __forceinline__ TileCoord tile_coord(int t, int num_m, int num_n) {
  const int group_size = kGroup * num_n;
  const int group = t / group_size;
  const int first = group * kGroup;
  const int gsz = min(num_m - first, kGroup);
  const int local = t % group_size;
  return TileCoord{first + local % gsz, local / gsz};
}

__device__ __forceinline__ void raise_abort(volatile uint32_t* flag) {
  atomicOr(&g_bs16_error, kErrTimeout);
  *flag = 1u;
}

// Scale codes to FP32, exactly.  A BF16 code is the top half of an FP32.
// An FP16 code (non-negative) moved into FP32's exponent/mantissa position
// reads as its value times 2^-112, subnormals included (the FP16 exponent
// field lines up with FP32's, and a zero exponent field gives an FP32
// subnormal with the same significand).  So for FP16 the row scale carries
// the factor 2^112 (at most 65504 * 2^112 < 2^128, no overflow) and the
// column scales carry 2^-112: their product is the exact s_A * s_B, rounded
// once by the multiply, as for BF16.
template <bool kF16>
__device__ __forceinline__ float row_scale(uint32_t c) {
  if constexpr (kF16)
    return __fmul_rn(__fmul_rn(__uint_as_float((c & 0x7FFFu) << 13), 0x1p112f), 0x1p112f);
  else
    return __uint_as_float(c << 16);
}
// Two column scales from one 32-bit word of codes (first column in the low
// half), as an FP32 pair (FP16: times 2^-112).
template <bool kF16>
__device__ __forceinline__ uint64_t col_scale_pair(uint32_t w) {
  if constexpr (kF16)
    return f32x2_pack(__uint_as_float((w & 0x7FFFu) << 13), __uint_as_float((w >> 3) & 0x0FFFE000u));
  else
    return f32x2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

template <bool kF16, bool kBF16Out>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bs16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const uint16_t* __restrict__ sfA, const uint16_t* __restrict__ sfB,
                     const float* __restrict__ Cin, void* __restrict__ Dout, int M, int N, int K,
                     uint32_t idesc, bool vec_out, bool bulk_scales) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int KT = K / BKS;                  // K % 128 == 0 (host check)
  const int KB = K / KBLK;
  const int unit = static_cast<int>(blockIdx.x), units = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.done[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.pfull[b]), 1);
      mbar_init(smem_u32(&sm.tempty[b]), kDrainWarps);
    }
    for (int s = 0; s < kScaleSlots; ++s) {
      mbar_init(smem_u32(&sm.sfull[s]), 1);
      mbar_init(smem_u32(&sm.sempty[s]), kDrainWarps);
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
      const TileCoord tc = tile_coord(t, num_m, num_n);
      for (int kt = 0; kt < KT; ++kt, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int s = static_cast<int>(it % kStages);
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(smem_u32(&sm.done[s]), ((it / kStages) & 1u) ^ 1u);
          if (good) {
            const uint32_t fb = smem_u32(&sm.full[s]);
            mbar_arrive_expect_tx(fb, kStageTxBytes);
            tma_load_2d_hint(smem_u32(sm.a[s]), &tmA, fb, kt * BKS, tc.m * BM, keep);
            tma_load_2d_hint(smem_u32(sm.b[s]), &tmB, fb, kt * BKS, tc.n * BN, keep);
          } else {
            raise_abort(&sm.abort_flag);
          }
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
      }
    }
    if (lane == 0) drain_fills(sm.full, kStages, it);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0) {
      // Block j (counted across this CTA's tiles) goes to buffer j & 1 once
      // the drain of block j - 2 has released it.  Each MMA starts a fresh
      // partial (no accumulation across blocks).
      const int my_tiles = unit < tiles ? (tiles - 1 - unit) / units + 1 : 0;
      const uint32_t total = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(KT);
      bool ok = true;
      for (uint32_t it = 0; it < total && ok; ++it) {
        const int s = static_cast<int>(it % kStages);
        if (!mbar_wait(smem_u32(&sm.full[s]), (it / kStages) & 1u)) {
          raise_abort(&sm.abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm.a[s]));
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sm.b[s]));
#pragma unroll
        for (int kk = 0; kk < kBlocksPerStage; ++kk) {
          const uint32_t j = it * kBlocksPerStage + static_cast<uint32_t>(kk);
          const uint32_t b = j & 1u;
          if (!mbar_wait(smem_u32(&sm.tempty[b]), ((j >> 1) & 1u) ^ 1u)) {
            raise_abort(&sm.abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          mma_f8f6f4(tmem + b * kBufStride, ad + 2 * kk, bd + 2 * kk, idesc, 0u);
          tc_commit(smem_u32(&sm.pfull[b]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.done[s]));
      }
      // every MMA this thread issued has completed once final_bar flips
      tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(&sm.abort_flag);
    }
    __syncwarp();
  } else if (warp == kScaleWarp) {
    // ------------------------------------------------------- scale loader
    // Stage it's scale codes: A's 4 blocks x 128 rows and B's 4 blocks x 192
    // rows, [kb][row] in global memory, into slot it % kScaleSlots once the
    // drains have released it.  With whole 16-byte rows (M, N multiples of
    // 8) one bulk copy per block and operand, completing on sfull; else plain
    // loads (codes past M / N become 0) and an arrive after them.
    setmaxnreg_dec<kRegsSmall>();
    for (int i = lane; i < kScaleSlots * kBlocksPerStage * (BM + BN) / 2; i += 32)
      reinterpret_cast<uint32_t*>(&sm.sa[0][0][0])[i] = 0u;     // sa and sb are contiguous
    fence_proxy_async_smem();   // before bulk copies overwrite them
    __syncwarp();
    uint32_t it = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units) {
      const TileCoord tc = tile_coord(t, num_m, num_n);
      const int m0 = tc.m * BM, n0 = tc.n * BN;
      const int na = min(BM, M - m0), nb = min(BN, N - n0);
      for (int kt = 0; kt < KT; ++kt, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int ss = static_cast<int>(it % kScaleSlots);
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(smem_u32(&sm.sempty[ss]), ((it / kScaleSlots) & 1u) ^ 1u);
          if (!good) raise_abort(&sm.abort_flag);
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
        if (bulk_scales) {
          if (lane == 0) {
            fence_proxy_async_smem();   // the drains' reads of the slot come first
            const uint32_t bar = smem_u32(&sm.sfull[ss]);
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kBlocksPerStage * (na + nb) * 2));
#pragma unroll
            for (int kk = 0; kk < kBlocksPerStage; ++kk) {
              const int64_t kb = static_cast<int64_t>(kt) * kBlocksPerStage + kk;
              bulk_load(smem_u32(sm.sa[ss][kk]), sfA + kb * M + m0, static_cast<uint32_t>(na * 2), bar);
              bulk_load(smem_u32(sm.sb[ss][kk]), sfB + kb * N + n0, static_cast<uint32_t>(nb * 2), bar);
            }
          }
        } else {
          for (int i = lane; i < kBlocksPerStage * BM; i += 32) {
            const int kk = i / BM, r = i % BM;
            const int64_t kb = static_cast<int64_t>(kt) * kBlocksPerStage + kk;
            sm.sa[ss][kk][r] = r < na ? __ldg(sfA + kb * M + m0 + r) : static_cast<uint16_t>(0);
          }
          for (int i = lane; i < kBlocksPerStage * BN; i += 32) {
            const int kk = i / BN, c = i % BN;
            const int64_t kb = static_cast<int64_t>(kt) * kBlocksPerStage + kk;
            sm.sb[ss][kk][c] = c < nb ? __ldg(sfB + kb * N + n0 + c) : static_cast<uint16_t>(0);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.sfull[ss]));
        }
      }
    }
    // no bulk copy may still be landing when the CTA exits
    if (bulk_scales && lane == 0)
      for (uint32_t j = it > kScaleSlots ? it - kScaleSlots : 0u; j < it; ++j)
        if (!mbar_wait(smem_u32(&sm.sfull[j % kScaleSlots]), (j / kScaleSlots) & 1u)) break;
    (void)KB;
    __syncwarp();
  } else if (warp < kFirstDrainWarp) {
    // warp 3 has no role; setmaxnreg is per warpgroup, so it gives its
    // registers back with the rest of warpgroup 0
    setmaxnreg_dec<kRegsSmall>();
  } else {
    // ---------------------------------------------------- drain + epilogue
    setmaxnreg_inc<kRegsLarge>();
    const int q = warp & 3;                        // TMEM lane quarter = rows 32q..32q+31
    const int g = (warp - kFirstDrainWarp) >> 2;   // 64-column group of the tile
    const int row = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + g * kGroupCols;
    uint32_t it = 0;
    bool ok = true;
    for (int t = unit; t < tiles && ok; t += units) {
      if (sm.abort_flag) break;
      const TileCoord tc = tile_coord(t, num_m, num_n);
      uint64_t acc[kGroupCols / 2];                // 64 FP32 accumulators, in pairs
#pragma unroll
      for (int i = 0; i < kGroupCols / 2; ++i) acc[i] = 0ull;
      for (int kt = 0; kt < KT && ok; ++kt, ++it) {
        const int ss = static_cast<int>(it % kScaleSlots);
        if (!mbar_wait(smem_u32(&sm.sfull[ss]), (it / kScaleSlots) & 1u)) {
          if (!sm.abort_flag) raise_abort(&sm.abort_flag);
          ok = false;
          break;
        }
        for (int kk = 0; kk < kBlocksPerStage; ++kk) {
          const uint32_t j = it * kBlocksPerStage + static_cast<uint32_t>(kk);
          const uint32_t b = j & 1u;
          if (!mbar_wait(smem_u32(&sm.pfull[b]), (j >> 1) & 1u)) {
            if (!sm.abort_flag) raise_abort(&sm.abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = lane_base + b * kBufStride;
          // both 32-column loads in flight at once; the buffer goes back to
          // the MMA as soon as they have landed
          uint32_t r0[32], r1[32];
          tmem_ld_32(taddr, r0);
          tmem_ld_32(taddr + 32, r1);
          const float sa = row_scale<kF16>(sm.sa[ss][kk][row]);
          const uint64_t sa2 = f32x2_pack(sa, sa);
          const uint16_t* sbp = &sm.sb[ss][kk][g * kGroupCols];
          tc_wait_ld_32(r0);
          tc_wait_ld_32(r1);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.tempty[b]));
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t (&cur)[32] = c ? r1 : r0;
#pragma unroll
            for (int v = 0; v < 4; ++v) {          // 8 columns: one 16-byte load of codes
              const uint4 w = *reinterpret_cast<const uint4*>(sbp + c * 32 + v * 8);
              const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int jj = v * 4 + e;          // pair within the chunk
                const uint64_t sc = fmul2(sa2, col_scale_pair<kF16>(wv[e]));
                ffma2(acc[c * 16 + jj], sc,
                      f32x2_pack(__uint_as_float(cur[2 * jj]), __uint_as_float(cur[2 * jj + 1])));
              }
            }
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.sempty[ss]));   // scales used
      }
      if (!ok) break;
      // ---- epilogue: this thread's row x 64 columns, + C, straight to D
      const int64_t grow = static_cast<int64_t>(tc.m) * BM + row;
      const int gcol0 = tc.n * BN + g * kGroupCols;
      if (grow < M) {
        constexpr int kPer = kBF16Out ? 8 : 4;     // values per 16-byte store
#pragma unroll
        for (int c = 0; c < kGroupCols / kPer; ++c) {
          float v[kPer];
#pragma unroll
          for (int e = 0; e < kPer / 2; ++e) f32x2_unpack(acc[c * (kPer / 2) + e], v[2 * e], v[2 * e + 1]);
          const int col = gcol0 + c * kPer;
          if (Cin != nullptr) {
#pragma unroll
            for (int e = 0; e < kPer; ++e)
              if (col + e < N) v[e] += __ldg(Cin + grow * N + col + e);
          }
          if (vec_out && col + kPer <= N) {
            uint4 u;
            if (kBF16Out) {
              u.x = pack_bf16x2(v[0], v[1]);
              u.y = pack_bf16x2(v[2], v[3]);
              u.z = pack_bf16x2(v[4 % kPer], v[5 % kPer]);
              u.w = pack_bf16x2(v[6 % kPer], v[7 % kPer]);
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(Dout) + grow * N + col) = u;
            } else {
              u = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2 % kPer]),
                             __float_as_uint(v[3 % kPer]));
              *reinterpret_cast<uint4*>(static_cast<float*>(Dout) + grow * N + col) = u;
            }
          } else {
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
              if (col + e >= N) break;
              if (kBF16Out)
                static_cast<__nv_bfloat16*>(Dout)[grow * N + col + e] = __float2bfloat16_rn(v[e]);
              else
                static_cast<float*>(Dout)[grow * N + col + e] = v[e];
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kF16, bool kBF16Out>
cudaError_t launch_variant(const Bs16GemmArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gemm_bs16_kernel<kF16, kBF16Out>;
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  const uint32_t idesc = idesc_f8f6f4(5u, 5u, BM, BN);   // E2M1 x E2M1, M128 N192
  // bulk copies of scale rows need 16-byte aligned rows: M, N multiples of 8
  const bool bulk = a.M % 8 == 0 && a.N % 8 == 0 && reinterpret_cast<uintptr_t>(a.sfA) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(a.sfB) % 16 == 0;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, s, a.tmA, a.tmB,
                    a.sfA, a.sfB, a.C, a.D, a.M, a.N, a.K, idesc, a.vec_out, bulk);
}

}  // namespace

cudaError_t gemm_bs16_error_read_and_clear(cudaStream_t s, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_bs16_error, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_bs16_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

int gemm_bs16_b_box_rows() { return BN; }

cudaError_t launch_gemm_bs16(const Bs16GemmArgs& a, int num_sms, cudaStream_t s) {
  if (a.f16_scales)
    return a.out_bf16 ? launch_variant<true, true>(a, num_sms, s) : launch_variant<true, false>(a, num_sms, s);
  return a.out_bf16 ? launch_variant<false, true>(a, num_sms, s) : launch_variant<false, false>(a, num_sms, s);
}

}  // namespace bsg

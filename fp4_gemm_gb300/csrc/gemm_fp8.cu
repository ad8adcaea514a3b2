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
// Warp roles (384 threads = 3 warpgroups, one CTA per SM, persistent over
// output tiles):
//   warp 0     producer: TMA loads of A (128 x 128 B) and B (256 x 128 B)
//              into a 4-stage ring; cp.async of the K tile's scales into an
//              8-slot scale ring.
//   warp 1     tensor-memory allocator and MMA issuer (one lane).
//   warps 2-3  idle (they complete warpgroup 0).
//   warps 4-11 promotion + epilogue: warpgroups 1 and 2.  Warp w reads TMEM
//              lanes 32*(w%4)..+31 (its rows) and column half (w-4)/4 of the
//              256-wide tile.
// Registers: the kernel launches at 168 per thread (384 x 168 = 64512);
// warpgroup 0 gives back down to 40 and the promotion warpgroups take 232
// each, 128 x 40 + 256 x 232 = 64512, which holds 128 FP32 accumulators plus
// two 32-column TMEM load buffers per thread without spilling.  The drain
// uses paired FP32 FMAs (fma.rn.f32x2), one instruction per two elements.
// Every wait is bounded; a wait that runs out sets the error word, raises a
// CTA-wide abort flag and all roles unwind to the final barrier.
#include "common.cuh"
#include "kernels.h"

namespace bsg {
namespace {

__device__ uint32_t g_fp8_error = 0;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;            // one scale tile along K = one promotion unit
constexpr int kStages = 4;
constexpr int kScaleSlots = 8;
constexpr int kThreads = 384;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstPromoWarp = 4;
constexpr int kRegsSmall = 56;     // warpgroup 0 after setmaxnreg.dec
constexpr int kRegsLarge = 224;    // promotion warpgroups after setmaxnreg.inc
static_assert(128 * kRegsSmall + 256 * kRegsLarge <= kThreads * 168,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;     // two 256-column FP32 partial buffers
constexpr int kGroupM = 8;         // tile raster: groups of 8 M tiles

struct __align__(1024) Smem {
  uint8_t a[kStages][BM * BK];
  uint8_t b[kStages][BN * BK];
  float sa[kScaleSlots][BM];
  float sb[kScaleSlots][BN];
  uint8_t epi[8][32 * 64];   // per promotion warp: 32 rows x 64 B output staging
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t sfull[kScaleSlots];
  uint64_t sempty[kScaleSlots];
  uint64_t final_bar;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
};

struct TileCoord {
  int m, n;
};

// Raster of the persistent tile loop.  Tiles are visited in groups of
// kGroupM rows of tiles along one dimension while the other is swept, so the
// operand panel of the group stays in L2 and the swept operand is re-read
// from L2.  along_n = true groups along N (sweeps M): chosen when A is the
// smaller operand, so the whole of A is what gets re-read and stays resident.
__device__ __forceinline__ TileCoord tile_coord(int t, int num_m, int num_n, bool along_n) {
  const int outer = along_n ? num_n : num_m;
  const int inner = along_n ? num_m : num_n;
  const int group_size = kGroupM * inner;
  const int group = t / group_size;
  const int first = group * kGroupM;
  const int gsz = min(outer - first, kGroupM);
  const int local = t % group_size;
  const int o = first + local % gsz, i = local / gsz;
  return along_n ? TileCoord{i, o} : TileCoord{o, i};
}

__device__ __forceinline__ void raise_abort(Smem& sm) {
  atomicOr(&g_fp8_error, kErrTimeout);
  sm.abort_flag = 1u;
}

template <bool kARow, bool kBRow, bool kBF16Out>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const float* __restrict__ sA, const float* __restrict__ sB,
                    const float* __restrict__ Cin, void* __restrict__ Dout, int M, int N, int K,
                    uint32_t idesc, bool vec_out, bool raster_n) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int KT = (K + BK - 1) / BK;
  const int num_nb = (N + 127) / 128;   // 128-wide scale blocks of B

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.tfull[b]), 1);
      mbar_init(smem_u32(&sm.tempty[b]), 8);
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
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kRegsSmall>();
    const uint64_t keep = l2_policy_evict_last();   // operands are re-read by other tiles
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      for (int kt = 0; kt < KT; ++kt, ++it) {
        if (sm.abort_flag) { ok = false; break; }
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        const int ss = static_cast<int>(it % kScaleSlots);
        const uint32_t phs = (it / kScaleSlots) & 1u;
        int good = 1;
        if (lane == 0) {
          good = mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1u) &&
                 mbar_wait(smem_u32(&sm.sempty[ss]), phs ^ 1u);
          if (good) {
            const uint32_t fb = smem_u32(&sm.full[s]);
            mbar_arrive_expect_tx(fb, (BM + BN) * BK);
            tma_load_2d_hint(smem_u32(sm.a[s]), &tmA, fb, kt * BK, tc.m * BM, keep);
            tma_load_2d_hint(smem_u32(sm.b[s]), &tmB, fb, kt * BK, tc.n * BN, keep);
          } else {
            raise_abort(sm);
          }
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) { ok = false; break; }
        // scales of this K tile -> scale slot ss
        if (kARow) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = tc.m * BM + 4 * lane + j;
            if (r < M) cp_async_4(smem_u32(&sm.sa[ss][4 * lane + j]), sA + static_cast<int64_t>(kt) * M + r);
          }
        } else if (lane == 0) {
          cp_async_4(smem_u32(&sm.sa[ss][0]), sA + static_cast<int64_t>(tc.m) * KT + kt);
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
    if (lane == 0) drain_fills(sm.full, kStages, it);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    setmaxnreg_dec<kRegsSmall>();
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int kt = 0; kt < KT; ++kt, ++it) {
          if (sm.abort_flag) { ok = false; break; }
          const uint32_t b = it & 1u;
          const uint32_t tph = (it >> 1) & 1u;
          const int s = static_cast<int>(it % kStages);
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait(smem_u32(&sm.tempty[b]), tph ^ 1u) ||
              !mbar_wait(smem_u32(&sm.full[s]), ph)) {
            raise_abort(sm);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm.a[s]));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sm.b[s]));
          const uint32_t d = tmem + b * BN;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            mma_f8f6f4(d, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          tc_commit(smem_u32(&sm.empty[s]));
          tc_commit(smem_u32(&sm.tfull[b]));
        }
      }
      // every MMA this thread issued has completed once final_bar flips
      tc_commit(smem_u32(&sm.final_bar));
      if (!mbar_wait(smem_u32(&sm.final_bar), 0)) raise_abort(sm);
    }
    __syncwarp();
  } else if (warp < kFirstPromoWarp) {
    setmaxnreg_dec<kRegsSmall>();            // idle warps of warpgroup 0
  } else {
    // ------------------------------------------------- promotion + epilogue
    setmaxnreg_inc<kRegsLarge>();
    const int q = warp & 3;                        // TMEM lane quarter = rows 32q..32q+31
    const int g = (warp - kFirstPromoWarp) >> 2;   // column half of the 256-wide tile
    const int row = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + g * 128;
    const uint64_t stream_out = l2_policy_evict_first();   // the result is not re-read
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, num_m, num_n, raster_n);
      uint64_t acc[64];                            // 128 FP32 accumulators, in pairs
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0ull;
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const uint32_t b = it & 1u;
        const uint32_t tph = (it >> 1) & 1u;
        const int ss = static_cast<int>(it % kScaleSlots);
        const uint32_t phs = (it / kScaleSlots) & 1u;
        if (sm.abort_flag || !mbar_wait(smem_u32(&sm.sfull[ss]), phs) ||
            !mbar_wait(smem_u32(&sm.tfull[b]), tph)) {
          if (!sm.abort_flag) raise_abort(sm);
          ok = false;
          break;
        }
        tc_fence_after();
        const float sa = kARow ? sm.sa[ss][row] : sm.sa[ss][0];
        const float sc = kBRow ? sa : sa * sm.sb[ss][g * 128];
        const uint64_t sc2 = f32x2_pack(sc, sc);
        const uint32_t taddr = lane_base + b * BN;
        uint32_t r0[16], r1[16];
        tmem_ld_16(taddr, r0);
        tc_wait_ld_16(r0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t (&cur)[16] = (c & 1) ? r1 : r0;
          uint32_t (&nxt)[16] = (c & 1) ? r0 : r1;
          if (c + 1 < 8) tmem_ld_16(taddr + (c + 1) * 16, nxt);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint64_t p = f32x2_pack(__uint_as_float(cur[2 * j]), __uint_as_float(cur[2 * j + 1]));
            if (kBRow) {
              const float2 sbv = *reinterpret_cast<const float2*>(&sm.sb[ss][g * 128 + c * 16 + 2 * j]);
              ffma2(acc[c * 8 + j], fmul2(sc2, f32x2_pack(sbv.x, sbv.y)), p);
            } else {
              ffma2(acc[c * 8 + j], sc2, p);
            }
          }
          if (c + 1 < 8) tc_wait_ld_16(nxt);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sm.tempty[b]));
          mbar_arrive(smem_u32(&sm.sempty[ss]));
        }
      }
      if (!ok) break;
      // ---- epilogue.  Each thread holds one row x 128 columns.  The warp
      // passes its 32 rows through a 32 x 64-byte staging buffer (16-byte
      // pieces XOR-swizzled by row, so both phases are bank-conflict free)
      // and writes back 8 rows x 64 contiguous bytes per store instruction
      // instead of 32 scattered 16-byte pieces.
      const int64_t row0 = static_cast<int64_t>(tc.m) * BM + q * 32;
      const int gcol0 = tc.n * BN + g * 128;
      const uint32_t stage = smem_u32(sm.epi[warp - kFirstPromoWarp]);
      constexpr int kElem = kBF16Out ? 2 : 4;
      constexpr int kColsPerChunk = 64 / kElem;     // 32 (BF16) or 16 (FP32)
      constexpr int kPerPiece = 16 / kElem;         // values per 16-byte piece
      const int64_t my_row = row0 + lane;
#pragma unroll
      for (int ch = 0; ch < 128 / kColsPerChunk; ++ch) {
        const int col0 = gcol0 + ch * kColsPerChunk;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          float v[kPerPiece];
#pragma unroll
          for (int j = 0; j < kPerPiece / 2; ++j)
            f32x2_unpack(acc[(ch * kColsPerChunk + p * kPerPiece) / 2 + j], v[2 * j], v[2 * j + 1]);
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
          const int r = 8 * i + (lane >> 2);
          const int p = lane & 3;
          const uint4 u = ld_shared_v4(stage + r * 64 + ((p ^ ((r >> 1) & 3)) << 4));
          const int64_t grow = row0 + r;
          const int col = col0 + p * kPerPiece;
          if (grow < M && col < N) {
            if (vec_out && col + kPerPiece <= N) {
              st_global_v4_hint(static_cast<uint8_t*>(Dout) + (grow * N + col) * kElem, u, stream_out);
            } else {
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int j = 0; j < kPerPiece; ++j) {
                if (col + j >= N) break;
                if (kBF16Out) {
                  const uint16_t h = static_cast<uint16_t>(w[j / 2] >> (16 * (j % 2)));
                  reinterpret_cast<uint16_t*>(Dout)[grow * N + col + j] = h;
                } else {
                  reinterpret_cast<float*>(Dout)[grow * N + col + j] = __uint_as_float(w[j]);
                }
              }
            }
          }
        }
        __syncwarp();
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

template <bool kARow, bool kBRow, bool kBF16Out>
cudaError_t launch_variant(const Fp8GemmArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gemm_fp8_kernel<kARow, kBRow, kBF16Out>;
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  const uint32_t idesc = idesc_f8f6f4(static_cast<uint32_t>(a.afmt), static_cast<uint32_t>(a.bfmt), BM, BN);
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) &&
                       (a.out_bf16 ? (a.N % 8 == 0) : (a.N % 4 == 0));
  // keep the smaller operand resident: sweep it inside groups of the larger
  const bool raster_n = static_cast<int64_t>(a.M) < static_cast<int64_t>(a.N);
  kern<<<grid, kThreads, smem, s>>>(a.tmA, a.tmB, a.sA, a.sB, a.C, a.D, a.M, a.N, a.K, idesc,
                                    vec_out, raster_n);
  return cudaGetLastError();
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

cudaError_t launch_gemm_fp8(const Fp8GemmArgs& a, int num_sms, cudaStream_t s) {
  const int key = (a.a_row ? 4 : 0) | (a.b_row ? 2 : 0) | (a.out_bf16 ? 1 : 0);
  switch (key) {
    case 0: return launch_variant<false, false, false>(a, num_sms, s);
    case 1: return launch_variant<false, false, true>(a, num_sms, s);
    case 2: return launch_variant<false, true, false>(a, num_sms, s);
    case 3: return launch_variant<false, true, true>(a, num_sms, s);
    case 4: return launch_variant<true, false, false>(a, num_sms, s);
    case 5: return launch_variant<true, false, true>(a, num_sms, s);
    case 6: return launch_variant<true, true, false>(a, num_sms, s);
    default: return launch_variant<true, true, true>(a, num_sms, s);
  }
}

}  // namespace bsg

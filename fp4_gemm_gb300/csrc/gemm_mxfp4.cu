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
// 128 rows x 4 K-blocks).  Each pipeline stage owns its own tensor-memory
// scale columns, so new scales never overwrite ones an in-flight MMA still
// reads.  The general kernel bulk-copies them to shared memory with the
// operands and moves them to tensor memory with tcgen05.cp.32x128b.warpx4
// right before the MMAs that use them (copy and MMA issued by one thread
// execute in order).  The decode kernel, whose MMAs are too small to hide a
// copy, has four warps store them with tcgen05.st instead.
//
// Two kernels:
//  * gemm_mxfp4_kernel: 128 x 128 output tiles, persistent, warp-specialised
//    (TMA producer warp, MMA warp, 8 epilogue warps draining a double-
//    buffered accumulator).  It also runs NVFP4 (kNv: UE4M3 scales per 16,
//    kind::mxf4nvf4 scale_vec::4X, the sum times alpha).  It serves problems
//    with few tiles; larger FP4 problems go to the 128 x 256 block-scaled
//    kernel of gemm_mx.cu.
//  * gemm_mxfp4_decode_kernel: decode shapes (M <= 32 activation rows), in
//    MXFP4 or NVFP4 form (kNv).  The weights are the MMA's 128-row operand
//    and the activations its N = 16/32 operand ("swap AB"), so the weight
//    matrix streams from HBM exactly once.
//    Work is split evenly over all SMs in units of (128 weight rows, 256 K);
//    a CTA whose range covers only part of a tile's K writes an FP32 partial
//    to the workspace, and the last contributor (per-tile counter) adds the
//    partials in a fixed order, so results are deterministic.
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "quant_math.cuh"

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
constexpr int kSfBase = 2 * BN;         // after the two accumulators
constexpr int kGroupM = 8;

// A stage covers 256 K: MXFP4 (blocks of 32) needs 2 scale atoms per operand,
// NVFP4 (blocks of 16) 4.  Each atom takes 4 tensor-memory columns; a stage's
// columns hold A's atoms, then B's: 16 (MXFP4) or 32 (NVFP4) per stage, so
// 5 stages fit beside the two accumulators in 512 columns.
template <bool kNv>
struct Fmt {
  static constexpr int kAtoms = kNv ? 4 : 2;
  static constexpr int kBlock = kNv ? 16 : 32;
  static constexpr int kSfColsPerStage = 8 * kAtoms;
};
static_assert(kSfBase + kStages * Fmt<true>::kSfColsPerStage <= kTmemCols, "TMEM columns");

template <bool kNv>
struct __align__(1024) Smem {
  uint8_t a[kStages][BM * kRowBytes];
  uint8_t b[kStages][BN * kRowBytes];
  uint8_t sfa[kStages][Fmt<kNv>::kAtoms * kSfAtom];
  uint8_t sfb[kStages][Fmt<kNv>::kAtoms * kSfAtom];
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

// kNv: NVFP4 (UE4M3 scales per 16, kind::mxf4nvf4 scale_vec::4X) instead of
// MXFP4 (UE8M0 per 32, kind::mxf4 scale_vec::2X); the sum is multiplied by
// alpha (the product of the two tensor scales) before the addend.
template <bool kBF16Out, bool kNv>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxfp4_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const uint8_t* __restrict__ sfA,
                      const uint8_t* __restrict__ sfB, const float* __restrict__ Cin,
                      void* __restrict__ Dout, int M, int N, int K, bool vec_out, float alpha) {
  using F = Fmt<kNv>;
  extern __shared__ uint8_t smem_raw[];
  Smem<kNv>& sm = *reinterpret_cast<Smem<kNv>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int kbytes = K / 2;
  const int KS = (kbytes + kRowBytes - 1) / kRowBytes;   // stages of 256 K
  const int KA = (K / F::kBlock + 3) / 4;                // scale atoms along K

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
  grid_dep_launch();
  grid_dep_wait();

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
          const int ka0 = F::kAtoms * ks;
          const int na = min(F::kAtoms, KA - ka0);
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
          const int ka0 = F::kAtoms * ks;
          const int na = min(F::kAtoms, KA - ka0);
          const uint32_t sfc = tmem + kSfBase + s * F::kSfColsPerStage;
          const uint32_t sfbc = sfc + 4 * F::kAtoms;    // B's atoms follow A's
          for (int a = 0; a < na; ++a) {
            tc_cp_32x128b_warpx4(sfc + 4 * a, sdesc_sf_32x16(smem_u32(sm.sfa[s] + a * kSfAtom)));
            tc_cp_32x128b_warpx4(sfbc + 4 * a, sdesc_sf_32x16(smem_u32(sm.sfb[s] + a * kSfAtom)));
          }
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm.a[s]));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sm.b[s]));
          const int rem = kbytes - ks * kRowBytes;
          const int nk = min(4, (rem + 31) / 32);
          for (int kk = 0; kk < nk; ++kk) {
            const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
            if (kNv) {
              // K = 64 = one atom (4 blocks of 16) per MMA
              mma_nvf4(d, ad + 2 * kk, bd + 2 * kk, idesc_nvf4(BM, BN), sfc + 4 * kk, sfbc + 4 * kk,
                       acc);
            } else {
              // K = 64 = half an atom: the scale id picks bytes 0-1 or 2-3
              const uint32_t id = idesc_mxf4(BM, BN, (kk & 1) * 2, (kk & 1) * 2);
              mma_mxf4(d, ad + 2 * kk, bd + 2 * kk, id, sfc + 4 * (kk >> 1), sfbc + 4 * (kk >> 1),
                       acc);
            }
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
          // alpha * acc + C with one rounding (NVFP4), acc + C otherwise:
          // written out so that the compiler's contraction choices do not
          // decide the result bits
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float c = (Cin != nullptr && col + j < N) ? __ldg(Cin + grow * N + col + j) : 0.0f;
            if (kNv)
              v[j] = Cin != nullptr ? __fmaf_rn(v[j], alpha, c) : __fmul_rn(v[j], alpha);
            else if (Cin != nullptr)
              v[j] = __fadd_rn(v[j], c);
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

// Warp roles: 0-3 epilogue (tensor-memory lane quarters 0-3), 4-7 scale
// writers (lane quarters 0-3), 8 TMA producer, 9 MMA issuer.
constexpr int kDecThreads = 320;
constexpr int kSfWarp0 = 4;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSlab = 128 * kRowBytes;   // one 128-row x 128-byte weight slab

// K chunks of 128 bytes (256 FP4 values) per pipeline stage.  With the
// chunked 3-D tensor map (K % 256 == 0) one TMA call reads CH * 128
// contiguous bytes of every weight row.  Big stages matter here: every stage
// costs the MMA thread one barrier wait, one fence and one commit (a few
// hundred ns), while each of its M128 x N16 x K64 MMAs takes ~30 ns.
__host__ __device__ constexpr int pow2_at_least(int v, int p) { return p >= v ? p : pow2_at_least(v, 2 * p); }

template <int NX, int CH, bool kNv = false>
struct Cfg {
  static constexpr int kStageBytes = CH * (kSlab + NX * kRowBytes);
  static constexpr int kStages0 = (216 * 1024) / kStageBytes;
  static constexpr int kStages = kStages0 > 12 ? 12 : kStages0;
  // scale atoms per 128-byte chunk and operand: MXFP4 two (E8M0 per 32),
  // NVFP4 four (UE4M3 per 16); per chunk the weights' atoms, then the
  // activations', four columns each
  static constexpr int kAtomsPerChunk = kNv ? 4 : 2;
  static constexpr int kSfColsPerStage = CH * 8 * kAtomsPerChunk;
  static constexpr int kSfBase = 2 * NX;            // after the two accumulator buffers
  static constexpr int kTmemCols = pow2_at_least(kSfBase + kStages * kSfColsPerStage, 32);
  static_assert(kStages >= 2, "at least two stages");
  static_assert(kTmemCols <= 512, "TMEM columns");
};

template <int NX, int CH>
struct __align__(1024) Smem {
  static constexpr int S = Cfg<NX, CH>::kStages;
  uint8_t w[S][CH * kSlab];
  uint8_t x[S][CH * NX * kRowBytes];
  // TMA bytes of the stage landed and the four scale-writer warps stored its
  // scales (so the MMA thread waits on one barrier per stage)
  uint64_t full[S];
  uint64_t empty[S];     // MMAs of the stage done: smem and scale columns free
  uint64_t tfull[2];     // accumulator buffer holds a finished segment
  uint64_t tempty[2];    // epilogue drained the buffer
  uint64_t final_bar;
  // on-the-fly activations: per stage (two in turn) and 4-block atom, each
  // activation row's four E8M0 codes, the first word of its scale cell
  uint32_t xsc[2][2 * CH][32];
  uint64_t xbar[2];      // all 128 scale-writer threads wrote stage buffer b's codes
  uint32_t tmem_base;
  uint32_t fast_flag;
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
  int nx, ch;
};

int chunks_for(int K, int nx) {
  if (K % 256 != 0) return 1;
  return nx == 16 ? 4 : 2;
}

Plan make_plan(int M, int N, int K, int num_sms) {
  Plan p;
  p.nx = M <= 16 ? 16 : 32;
  p.ch = chunks_for(K, p.nx);
  p.tiles = (static_cast<int64_t>(N) + 127) / 128;
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

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One 32-value block of activation row r quantised to MXFP4 with the rule of
// the stand-alone quantiser ("Rubin FP4 GEMM deep dive" section 4.2): the
// E8M0 code of the power of two nearest max|x| / 6, then E2M1(x * 2^-e),
// two codes per byte, first value in the low nibble.  Returns the code.
__device__ __forceinline__ uint32_t quantize_block_mxfp4(const void* x, bool bf16, bool vec, int64_t ldx,
                                                         int r, int64_t b, uint4& codes) {
  float v[32];
  if (bf16) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + r * ldx + b * 32;
    if (vec) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + h);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * h + 2 * j] = __uint_as_float(w[j] << 16);
          v[8 * h + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(static_cast<uint32_t>(p[j]) << 16);
    }
  } else {
    const float* p = static_cast<const float*>(x) + r * ldx + b * 32;
    if (vec) {
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p) + h);
        v[4 * h] = u.x; v[4 * h + 1] = u.y; v[4 * h + 2] = u.z; v[4 * h + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = p[j];
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  // The E8M0 code of the power of two nearest RN(amax / 6), without the
  // division: with amax = m 2^e (1 <= m < 2), amax / 6 = (m / 1.5) 2^(e-2),
  // which is 2^(e-2) after that rounding when m >= 1.125 and 2^(e-3) below.
  // RN to FP32 cannot move the quotient across the boundary: m / 0.75 is
  // 1.5 only at m = 1.125 exactly (a tie, rounded up like the rule does) and
  // never reaches 2.  Zero, tiny (quotient near the subnormals), infinite or
  // NaN maxima take the rule itself.
  const uint32_t ab = __float_as_uint(amax);
  const int ef = static_cast<int>(ab >> 23);          // amax >= 0: no sign bit
  const uint32_t code = (ef < 27 || ef == 255)
                            ? e8m0_nearest(__fdiv_rn(amax, 6.0f))
                            : static_cast<uint32_t>(ef - 2 - ((ab & 0x7FFFFFu) >= 0x100000u ? 0 : 1));
  // 2^-(code-127) as an FP32 normal: code in [0,254] -> exponent field 254-code
  const float inv = __uint_as_float(static_cast<uint32_t>(254 - static_cast<int>(code)) << 23);
  const uint64_t inv2 = f32x2_pack(inv, inv);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w[q] = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float lo, hi;
      f32x2_unpack(fmul2(f32x2_pack(v[8 * q + 2 * j], v[8 * q + 2 * j + 1]), inv2), lo, hi);
      w[q] |= cvt2_e2m1(lo, hi) << (8 * j);
    }
  }
  codes = make_uint4(w[0], w[1], w[2], w[3]);
  return code;
}

// Byte offset of the 16-byte piece p (0..7) of row r in a K-major tile with
// 128-byte rows in the 128-byte swizzle (the layout a SWIZZLE_128B TMA box
// writes): 8-row atoms of 1024 bytes, piece index XOR the row within its atom.
__device__ __forceinline__ uint32_t swz128_piece(int r, int p) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + (((p ^ r) & 7) << 4));
}

// NVFP4: alpha * acc + C with one rounding (alpha * acc without C), as the
// other NVFP4 kernels do; MXFP4: acc + C
template <int NX, bool kBF16Out, bool kNv>
__device__ __forceinline__ void store_row(const float (&v)[NX], const float* __restrict__ Cin,
                                          void* __restrict__ Dout, int M, int N, int64_t n, float alpha) {
  if (n >= N) return;
#pragma unroll
  for (int mm = 0; mm < NX; ++mm) {
    if (mm < M) {
      float o = v[mm];
      if (kNv)
        o = Cin != nullptr ? __fmaf_rn(o, alpha, __ldg(Cin + static_cast<int64_t>(mm) * N + n))
                           : __fmul_rn(o, alpha);
      else if (Cin != nullptr)
        o = __fadd_rn(o, __ldg(Cin + static_cast<int64_t>(mm) * N + n));
      if (kBF16Out)
        static_cast<__nv_bfloat16*>(Dout)[static_cast<int64_t>(mm) * N + n] = __float2bfloat16_rn(o);
      else
        static_cast<float*>(Dout)[static_cast<int64_t>(mm) * N + n] = o;
    }
  }
}

// Prefetch of a tensor-map box (same coordinates as the load it stands in
// front of) or of `bytes` of global memory (multiple of 16, 16-byte aligned)
// into L2.  A hint only: nothing completes and no data reaches the CTA.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x),
               "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// L2 prefetch of the weight-scale atoms of work unit u.  Not inlined, like
// prefetch_first_stages below.
__device__ __noinline__ void prefetch_scale_atoms(const uint8_t* sfW, int64_t u, int64_t KS, int KA, int CH,
                                                  int apc) {
  const int64_t tile = u / KS;
  const int ka0 = apc * static_cast<int>(u % KS) * CH;
  const int na = min(apc * CH, KA - ka0);
  if (na > 0) bulk_prefetch_l2(sfW + (tile * KA + ka0) * kSfAtom, static_cast<uint32_t>(na * kSfAtom));
}

// L2 prefetch of the weight boxes and weight-scale atoms of a decode CTA's
// first `stages` units (the coordinates its producer and scale writers load
// them with).  Not inlined: its registers stay out of the kernel's roles.
__device__ __noinline__ void prefetch_first_stages(const CUtensorMap* tmW, const uint8_t* sfW, int64_t u0,
                                                   int64_t u1, int64_t KS, int KA, int stages, int CH,
                                                   int apc) {
  const int64_t npf = u1 - u0 < stages ? u1 - u0 : stages;
  for (int64_t i = 0; i < npf; ++i) {
    const int64_t u = u0 + i;
    const int64_t tile = u / KS;
    const int c0 = static_cast<int>(u % KS) * CH;
    if (CH == 1)
      tma_prefetch_l2_2d(tmW, c0 * kRowBytes, static_cast<int32_t>(tile * 128));
    else
      tma_prefetch_l2_3d(tmW, 0, static_cast<int32_t>(tile * 128), c0);
    const int ka0 = apc * c0;
    const int na = min(apc * CH, KA - ka0);
    if (na > 0) bulk_prefetch_l2(sfW + (tile * KA + ka0) * kSfAtom, static_cast<uint32_t>(na * kSfAtom));
  }
}

// kQ: the activations arrive unquantised (FP32 or BF16, xsrc with row pitch
// ldx; qflags bit 0: BF16, bit 1: 16-byte loads allowed) and are quantised
// stage by stage by the scale-writer warps: each stage's K slice of all
// activation rows goes to MXFP4 codes written straight into the stage's
// shared-memory operand, in the 128-byte swizzle a TMA load would produce,
// and E8M0 codes stored into the tensor-memory scale cells - so the TMA
// moves weights only, and no other kernel or CTA is waited for.  tmX and sfX
// are not used then.
template <int NX, int CH, bool kBF16Out, bool kQ, bool kNv>
__global__ void __launch_bounds__(kDecThreads, 1)
    gemm_mxfp4_decode_kernel(const __grid_constant__ CUtensorMap tmX,
                             const __grid_constant__ CUtensorMap tmW,
                             const uint8_t* __restrict__ sfX, const uint8_t* __restrict__ sfW,
                             const float* __restrict__ Cin, void* __restrict__ Dout, int M, int N,
                             int K, int64_t KS, int64_t U, int64_t smax,
                             float* __restrict__ ws, uint32_t* __restrict__ counters,
                             const void* __restrict__ xsrc, int64_t ldx, int qflags, float alpha) {
  static_assert(!(kQ && kNv), "activations are quantised in the kernel for MXFP4 only");
  constexpr int kStages = Cfg<NX, CH, kNv>::kStages;
  constexpr int kSfCols = Cfg<NX, CH, kNv>::kSfColsPerStage;
  constexpr int kSfBase = Cfg<NX, CH, kNv>::kSfBase;
  constexpr int kTmemCols = Cfg<NX, CH, kNv>::kTmemCols;
  constexpr int kApc = Cfg<NX, CH, kNv>::kAtomsPerChunk;
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
  const int KA = (K / (kNv ? 16 : 32) + 3) / 4;          // scale atoms along K

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1 + 4);   // producer + four scale writers
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.tfull[b]), 1);
      mbar_init(smem_u32(&sm.tempty[b]), 4);
      mbar_init(smem_u32(&sm.xbar[b]), 128);
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
  grid_dep_launch();
  // The weights and weight scales of the first stages go into L2 before the
  // wait for the previous kernel, so that under programmatic dependent
  // launch their DRAM latency overlaps that kernel's tail.  A prefetch only
  // moves lines into L2, where every SM's writes land: the loads after the
  // wait see whatever the previous kernel wrote, prefetched or not.
  if (warp == kProducerWarp && lane == 0) prefetch_first_stages(&tmW, sfW, u0, u1, KS, KA, kStages, CH, kApc);
  grid_dep_wait();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();    // activations: re-read by every CTA
      const uint64_t stream = l2_policy_evict_first(); // weights: read exactly once
      uint32_t it = 0;
      int64_t u = u0;
      for (; u < u1; ++u, ++it) {
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = (it / kStages) & 1u;
        if (sm.abort_flag) break;
        if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        const int64_t tile = u / KS;
        const int c0 = static_cast<int>(u % KS) * CH;    // first 128-byte chunk
        const uint32_t fb = smem_u32(&sm.full[s]);
        // kQ: the activation half of the stage is written by the scale writers
        mbar_arrive_expect_tx(fb, CH * (kQ ? 128 : 128 + NX) * kRowBytes);
        if (CH == 1) {
          tma_load_2d_hint(smem_u32(sm.w[s]), &tmW, fb, c0 * kRowBytes, static_cast<int32_t>(tile * 128), stream);
          if (!kQ) tma_load_2d_hint(smem_u32(sm.x[s]), &tmX, fb, c0 * kRowBytes, 0, keep);
        } else {
          tma_load_3d_hint(smem_u32(sm.w[s]), &tmW, fb, 0, static_cast<int32_t>(tile * 128), c0, stream);
          if (!kQ) tma_load_3d_hint(smem_u32(sm.x[s]), &tmX, fb, 0, 0, c0, keep);
        }
        // the weight-scale atoms of the unit kStages ahead go into L2, so
        // that the scale writers' loads of them hit L2
        if (u + kStages < u1) prefetch_scale_atoms(sfW, u + kStages, KS, KA, CH, kApc);
      }
      drain_fills(sm.full, kStages, it);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
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
        // use n = seg / 2 of this buffer waits for the epilogue's n-th hand-
        // back (the first use of each buffer passes at once)
        if (first && !mbar_wait(smem_u32(&sm.tempty[buf]), ((seg >> 1) & 1u) ^ 1u)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        if (!mbar_wait(smem_u32(&sm.full[s]), ph)) {
          raise_abort(&sm.abort_flag);
          break;
        }
        tc_fence_after();
        const int c0 = ks * CH;
        const uint32_t sfc = tmem + kSfBase + s * kSfCols;
        const uint32_t d = tmem + buf * NX;
        // the first MMA of a segment overwrites the accumulator
        const uint32_t acc0 = first ? 0u : 1u;
        if ((c0 + CH) * kRowBytes <= kbytes) {
          // whole stage: fully unrolled so the MMAs issue back to back
          // (descriptor start addresses advance in 16-byte units)
          const uint64_t w0 = sdesc_kmajor_sw128(smem_u32(sm.w[s]));
          const uint64_t x0 = sdesc_kmajor_sw128(smem_u32(sm.x[s]));
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            const uint32_t sfj = sfc + 8 * kApc * j;   // chunk j: weight atoms, then activation atoms
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t wd = w0 + (j * kSlab) / 16 + 2 * kk;
              const uint64_t xd = x0 + (j * NX * kRowBytes) / 16 + 2 * kk;
              const uint32_t acc = (j == 0 && kk == 0) ? acc0 : 1u;
              if (kNv)   // K = 64 = one atom (four UE4M3 bytes per row) per MMA
                mma_nvf4(d, wd, xd, idesc_nvf4(128, NX), sfj + 4 * kk, sfj + 4 * kApc + 4 * kk, acc);
              else       // K = 64 = half an E8M0 atom: the scale id picks bytes 0-1 or 2-3
                mma_mxf4(d, wd, xd, idesc_mxf4(128, NX, (kk & 1) * 2, (kk & 1) * 2), sfj + 4 * (kk >> 1),
                         sfj + 4 * kApc + 4 * (kk >> 1), acc);
            }
          }
        } else {
          const int nch = min(CH, KC - c0);
          for (int j = 0; j < nch; ++j) {
            const uint64_t wd = sdesc_kmajor_sw128(smem_u32(sm.w[s] + j * kSlab));
            const uint64_t xd = sdesc_kmajor_sw128(smem_u32(sm.x[s] + j * NX * kRowBytes));
            const int rem = kbytes - (c0 + j) * kRowBytes;
            const int nk = min(4, (rem + 31) / 32);
            const uint32_t sfj = sfc + 8 * kApc * j;
            for (int kk = 0; kk < nk; ++kk) {
              const uint32_t acc = (j == 0 && kk == 0) ? acc0 : 1u;
              if (kNv) {
                mma_nvf4(d, wd + 2 * kk, xd + 2 * kk, idesc_nvf4(128, NX), sfj + 4 * kk, sfj + 4 * kApc + 4 * kk,
                         acc);
              } else {
                const uint32_t id = idesc_mxf4(128, NX, (kk & 1) * 2, (kk & 1) * 2);
                mma_mxf4(d, wd + 2 * kk, xd + 2 * kk, id, sfj + 4 * (kk >> 1), sfj + 4 * kApc + 4 * (kk >> 1),
                         acc);
              }
            }
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
  } else if (warp >= kSfWarp0) {
    // ----------------------------------------------------- scale writers
    // Each warp stores the stage's scale atoms into its own quarter of the
    // tensor-memory lanes with tcgen05.st: lane l of every quarter holds
    // bytes [16 l, 16 l + 16) of an atom in four consecutive columns, the
    // image a 32x128b.warpx4 copy would make.  Keeping these stores off the
    // tensor pipe lets the MMAs issue back to back.  A stage's columns are
    // rewritten only after its previous MMAs completed (empty barrier).
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    uint32_t it = 0;
    for (int64_t u = u0; u < u1; ++u, ++it) {
      const int s = static_cast<int>(it % kStages);
      const uint32_t ph = (it / kStages) & 1u;
      if (sm.abort_flag) break;
      if (!mbar_wait(smem_u32(&sm.empty[s]), ph ^ 1u)) {
        raise_abort(&sm.abort_flag);
        break;
      }
      tc_fence_after();
      const int64_t tile = u / KS;
      const int ka0 = kApc * static_cast<int>(u % KS) * CH;
      const int na = min(kApc * CH, KA - ka0);
      const uint4* gw = reinterpret_cast<const uint4*>(sfW + (tile * KA + ka0) * kSfAtom) + lane;
      const uint4* gx = reinterpret_cast<const uint4*>(sfX + static_cast<int64_t>(ka0) * kSfAtom) + lane;
      const uint32_t sfc = lane_base + kSfBase + s * kSfCols;
      if constexpr (kNv) {
        // NVFP4: every load of the stage's atoms is issued before the first
        // store, so the stage waits for one memory latency, not one per
        // chunk (chunk j: weight atoms at columns 32 j + 4 q, activation
        // atoms 16 columns later)
        uint4 vw[4 * CH], vx[4 * CH];
#pragma unroll
        for (int a = 0; a < 4 * CH; ++a) {
          if (a < na) {
            vw[a] = __ldg(gw + a * (kSfAtom / 16));
            vx[a] = __ldg(gx + a * (kSfAtom / 16));
          }
        }
#pragma unroll
        for (int a = 0; a < 4 * CH; ++a) {
          if (a < na) {
            tmem_st_4(sfc + 32 * (a >> 2) + 4 * (a & 3), vw[a]);
            tmem_st_4(sfc + 32 * (a >> 2) + 16 + 4 * (a & 3), vx[a]);
          }
        }
      } else {
        uint4 vw[2 * CH], vx[2 * CH];
#pragma unroll
        for (int a = 0; a < 2 * CH; ++a)
          if (a < na) vw[a] = __ldg(gw + a * (kSfAtom / 16));
        if constexpr (kQ) {
          // This stage's K slice (CH x 256 values) of every activation row,
          // one 32-value block per item, items row-major so that neighbouring
          // threads read neighbouring bytes.  Rows past M and blocks past K/32
          // get zero codes and scale code 127, as a TMA load past the edge
          // and the stand-alone quantiser's padding give.
          constexpr int kBlocks = 8 * CH;                 // 32-value blocks in the slice
          constexpr int kItems = NX * kBlocks / 128;      // per thread
          static_assert(NX * kBlocks % 128 == 0, "whole items per thread");
          const int t = static_cast<int>(threadIdx.x) - kSfWarp0 * 32;
          const int64_t gb0 = static_cast<int64_t>(u % KS) * CH * 8;   // first block of the slice
          const int buf = static_cast<int>(it & 1u);
          uint8_t* xs = sm.x[s];
#pragma unroll
          for (int j = 0; j < kItems; ++j) {
            const int i = t + 128 * j;
            const int r = i / kBlocks, bb = i % kBlocks;
            const int64_t gb = gb0 + bb;
            uint4 codes = make_uint4(0u, 0u, 0u, 0u);
            uint32_t code = 127u;
            if (r < M && gb < K / 32)
              code = quantize_block_mxfp4(xsrc, (qflags & 1) != 0, (qflags & 2) != 0, ldx, r, gb, codes);
            st_shared_v4(smem_u32(xs + (bb >> 3) * NX * kRowBytes) + swz128_piece(r, bb & 7), codes);
            reinterpret_cast<uint8_t*>(&sm.xsc[buf][bb >> 2][r])[bb & 3] = static_cast<uint8_t>(code);
          }
          fence_proxy_async_smem();   // the codes are read by the tensor core (async proxy)
          // all four scale-writer warps have written this stage's codes (a
          // bounded wait: a warp that stopped on an abort cannot hang the rest);
          // buffer it & 1 comes round again two stages later, after every
          // thread has arrived on the stage in between, i.e. read this one
          mbar_arrive(smem_u32(&sm.xbar[buf]));
          if (!mbar_wait(smem_u32(&sm.xbar[buf]), (it >> 1) & 1u)) {
            raise_abort(&sm.abort_flag);
            break;
          }
#pragma unroll
          for (int a = 0; a < 2 * CH; ++a)
            if (a < na)
              vx[a] = make_uint4(lane < NX ? sm.xsc[buf][a][lane] : 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
                                 0x7F7F7F7Fu);
        } else {
#pragma unroll
          for (int a = 0; a < 2 * CH; ++a)
            if (a < na) vx[a] = __ldg(gx + a * (kSfAtom / 16));
        }
#pragma unroll
        for (int a = 0; a < 2 * CH; ++a) {
          if (a < na) {
            tmem_st_4(sfc + 16 * (a >> 1) + 4 * (a & 1), vw[a]);
            tmem_st_4(sfc + 16 * (a >> 1) + 8 + 4 * (a & 1), vx[a]);
          }
        }
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.full[s]));
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int row = warp * 32 + lane;               // weight row within the tile
    const uint32_t lane_taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint32_t seg = 0;
    int64_t u = u0;
    while (u < u1) {
      const int64_t tile = u / KS;
      const int64_t seg_end = min(u1, (tile + 1) * KS);
      const bool whole = (u == tile * KS) && (seg_end == (tile + 1) * KS);
      const uint32_t buf = seg & 1u;
      const int64_t n = tile * 128 + row;
      // Split tile: this CTA holds segment sidx of nseg.  If the other
      // segments are already published (their counter increments are
      // visible), this CTA finishes the tile straight from its registers
      // and skips publishing its own partial.  Otherwise it publishes, and
      // the last contributor adds the partials.  Either way the partials are
      // added in segment order, so the result does not depend on timing.
      int64_t nseg = 1, sidx = 0;
      int nsuf = 0;
      bool fast = false;
      float pre[NX], suf[2][NX];
      if (!whole) {
        const int64_t first_owner = owner(tile * KS, U, G);
        nseg = owner((tile + 1) * KS - 1, U, G) - first_owner + 1;
        sidx = static_cast<int64_t>(blockIdx.x) - first_owner;
        nsuf = static_cast<int>(nseg - 1 - sidx);
        if (nsuf <= 2) {
          if (threadIdx.x == 0)
            sm.fast_flag = (ld_acquire_u32(counters + tile) + 1u == static_cast<uint32_t>(nseg)) ? 1u : 0u;
          asm volatile("bar.sync 1, 128;" ::: "memory");
          fast = sm.fast_flag != 0u;
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (fast) {
            const float* base = ws + tile * smax * NX * 128 + row;
#pragma unroll
            for (int mm = 0; mm < NX; ++mm) pre[mm] = 0.0f;
            for (int64_t sg = 0; sg < sidx; ++sg) {
#pragma unroll
              for (int mm = 0; mm < NX; ++mm) pre[mm] += __ldcg(base + (sg * NX + mm) * 128);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (i < nsuf) {
#pragma unroll
                for (int mm = 0; mm < NX; ++mm) suf[i][mm] = __ldcg(base + ((sidx + 1 + i) * NX + mm) * 128);
              }
            }
          }
        }
      }
      if (sm.abort_flag || !mbar_wait(smem_u32(&sm.tfull[buf]), (seg >> 1) & 1u)) {
        if (!sm.abort_flag) raise_abort(&sm.abort_flag);
        break;
      }
      tc_fence_after();
      float acc[NX];
#pragma unroll
      for (int c = 0; c < NX / 16; ++c) {
        uint32_t r[16];
        tmem_ld_16(lane_taddr + buf * NX + c * 16, r);
        tc_wait_ld_16(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c * 16 + j] = __uint_as_float(r[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tempty[buf]));
      if (whole) {
        store_row<NX, kBF16Out, kNv>(acc, Cin, Dout, M, N, n, alpha);
      } else if (fast) {
        float tot[NX];
#pragma unroll
        for (int mm = 0; mm < NX; ++mm) {
          tot[mm] = pre[mm] + acc[mm];
#pragma unroll
          for (int i = 0; i < 2; ++i)
            if (i < nsuf) tot[mm] += suf[i][mm];
        }
        store_row<NX, kBF16Out, kNv>(tot, Cin, Dout, M, N, n, alpha);
        // leave the workspace zero-filled for the next call
        float* base = ws + tile * smax * NX * 128 + row;
        for (int64_t sg = 0; sg < nseg; ++sg) {
          if (sg == sidx) continue;
#pragma unroll
          for (int mm = 0; mm < NX; ++mm) base[(sg * NX + mm) * 128] = 0.0f;
        }
        if (threadIdx.x == 0) atomicExch(counters + tile, 0u);
      } else {
        float* part = ws + (tile * smax + sidx) * NX * 128;
#pragma unroll
        for (int mm = 0; mm < NX; ++mm) part[mm * 128 + row] = acc[mm];
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (threadIdx.x == 0) {
          const uint32_t prev = atomicAdd(counters + tile, 1u);
          sm.last_flag = (prev + 1 == static_cast<uint32_t>(nseg)) ? 1u : 0u;
          // a counter past its segment count means the workspace was not zero
          if (prev + 1 > static_cast<uint32_t>(nseg)) atomicOr(&g_mxfp4_error, kErrWorkspace);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (sm.last_flag) {
          __threadfence();
          // Sum the segments in order, then zero every slot of this row so
          // the workspace is left zero-filled for any shape.
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
          store_row<NX, kBF16Out, kNv>(tot, Cin, Dout, M, N, n, alpha);
          if (threadIdx.x == 0) atomicExch(counters + tile, 0u);
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
  const size_t smem = (a.nvfp4 ? sizeof(Smem<true>) : sizeof(Smem<false>)) + 1024;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) &&
                       (a.out_bf16 ? (a.N % 8 == 0) : (a.N % 4 == 0));
  auto kern = a.nvfp4 ? (a.out_bf16 ? gemm_mxfp4_kernel<true, true> : gemm_mxfp4_kernel<false, true>)
                      : (a.out_bf16 ? gemm_mxfp4_kernel<true, false> : gemm_mxfp4_kernel<false, false>);
  const cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a.tmA, a.tmB, a.sfA, a.sfB, a.C, a.D,
                    a.M, a.N, a.K, vec_out, a.nvfp4 ? a.alpha : 1.0f);
}

size_t gemm_mxfp4_decode_workspace(int M, int N, int K, int num_sms) {
  const decode::Plan p = decode::make_plan(M, N, K, num_sms);
  if (p.smax <= 1) return 0;
  const size_t floats = static_cast<size_t>(p.tiles * p.smax * p.nx * 128);
  return floats * sizeof(float) + static_cast<size_t>(p.tiles) * sizeof(uint32_t);
}

size_t gemm_mxfp4_act_workspace(int M, int N, int K, int num_sms, size_t* off) {
  // The decode kernel's split-K area (M <= 32) first; unless the kernel
  // quantises as it goes (M <= kActFusedMaxM), the activation codes and
  // scale atoms follow, each at a 256-byte boundary.
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t split = M <= 32 ? gemm_mxfp4_decode_workspace(M, N, K, num_sms) : 0;
  if (off != nullptr) off[0] = off[1] = off[2] = 0;
  if (M <= kActFusedMaxM) return split;
  const size_t codes = static_cast<size_t>(M) * (K / 2);
  const size_t atoms = static_cast<size_t>((M + 127) / 128) * ((K / 32 + 3) / 4) * kSfAtom;
  if (off != nullptr) {
    off[1] = up(split);
    off[2] = off[1] + up(codes);
  }
  return up(split) + up(codes) + atoms;
}

namespace {
template <int NX, int CH, bool BF, bool Q, bool NV>
cudaError_t launch_decode_variant(const Mxfp4GemmArgs& a, const decode::Plan& p, float* ws,
                                  uint32_t* counters, cudaStream_t s) {
  using namespace decode;
  CUtensorMap tmX, tmW;
  std::memset(&tmX, 0, sizeof(tmX));   // not read when the activations come unquantised (Q)
  const uint64_t kb = static_cast<uint64_t>(a.K) / 2;
  if (CH == 1) {
    if ((!Q && !make_kmajor_map(&tmX, a.A, kb, a.M, kb, NX)) || !make_kmajor_map(&tmW, a.B, kb, a.N, kb, 128))
      return cudaErrorInvalidValue;
  } else {
    if ((!Q && !make_kmajor_map_chunked(&tmX, a.A, kb, a.M, kb, NX, CH)) ||
        !make_kmajor_map_chunked(&tmW, a.B, kb, a.N, kb, 128, CH))
      return cudaErrorInvalidValue;
  }
  const size_t smem = sizeof(Smem<NX, CH>) + 1024;
  cudaError_t e = set_smem(gemm_mxfp4_decode_kernel<NX, CH, BF, Q, NV>, smem);
  if (e != cudaSuccess) return e;
  // 16-byte loads of the unquantised activations where alignment allows
  const bool vec = Q && reinterpret_cast<uintptr_t>(a.xsrc) % 16 == 0 && a.ldx % (a.xsrc_bf16 ? 8 : 4) == 0;
  const int qflags = (a.xsrc_bf16 ? 1 : 0) | (vec ? 2 : 0);
  return launch_pdl(gemm_mxfp4_decode_kernel<NX, CH, BF, Q, NV>, dim3(static_cast<unsigned>(p.G)),
                    dim3(kDecThreads), smem, s, tmX, tmW, a.sfA, a.sfB, a.C, a.D, a.M, a.N, a.K, p.KS,
                    p.U, p.smax, ws, counters, a.xsrc, a.ldx, qflags, NV ? a.alpha : 1.0f);
}

template <int NX, int CH, bool Q, bool NV>
cudaError_t launch_decode_out(const Mxfp4GemmArgs& a, const decode::Plan& p, float* ws,
                              uint32_t* counters, cudaStream_t s) {
  return a.out_bf16 ? launch_decode_variant<NX, CH, true, Q, NV>(a, p, ws, counters, s)
                    : launch_decode_variant<NX, CH, false, Q, NV>(a, p, ws, counters, s);
}

template <bool Q, bool NV>
cudaError_t launch_decode_shape(const Mxfp4GemmArgs& a, const decode::Plan& p, float* ws,
                                uint32_t* counters, cudaStream_t s) {
  if (p.nx == 16)
    return p.ch == 1 ? launch_decode_out<16, 1, Q, NV>(a, p, ws, counters, s)
                     : launch_decode_out<16, 4, Q, NV>(a, p, ws, counters, s);
  return p.ch == 1 ? launch_decode_out<32, 1, Q, NV>(a, p, ws, counters, s)
                   : launch_decode_out<32, 2, Q, NV>(a, p, ws, counters, s);
}
}  // namespace

cudaError_t launch_gemm_mxfp4_decode(const Mxfp4GemmArgs& a, int num_sms, cudaStream_t s) {
  using namespace decode;
  const Plan p = make_plan(a.M, a.N, a.K, num_sms);
  float* ws = static_cast<float*>(a.workspace);
  uint32_t* counters =
      ws == nullptr ? nullptr : reinterpret_cast<uint32_t*>(ws + p.tiles * p.smax * p.nx * 128);
  // NVFP4 (a.nvfp4, scales UE4M3 per 16, result times a.alpha) takes
  // quantised activations only
  if (a.nvfp4)
    return a.xsrc != nullptr ? cudaErrorInvalidValue : launch_decode_shape<false, true>(a, p, ws, counters, s);
  return a.xsrc != nullptr ? launch_decode_shape<true, false>(a, p, ws, counters, s)
                           : launch_decode_shape<false, false>(a, p, ws, counters, s);
}

}  // namespace bsg

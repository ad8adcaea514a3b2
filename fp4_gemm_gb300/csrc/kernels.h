// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsg {

// Each kernel translation unit owns one device error word.  read_and_clear
// copies it to the host (synchronously on `s`) and zeroes it.
cudaError_t quantize_error_read_and_clear(cudaStream_t s, uint32_t* out);
cudaError_t gemm_fp8_error_read_and_clear(cudaStream_t s, uint32_t* out);
cudaError_t gemm_mxfp4_error_read_and_clear(cudaStream_t s, uint32_t* out);
cudaError_t mma_peak_error_read_and_clear(cudaStream_t s, uint32_t* out);
cudaError_t gemm_mx_error_read_and_clear(cudaStream_t s, uint32_t* out);
cudaError_t mma_probe_error_read_and_clear(cudaStream_t s, uint32_t* out);

// ------------------------------------------------------------- quantisers
// src_bf16: source is BF16 (else FP32).  fmt: 0 E4M3, 1 E5M2.
cudaError_t launch_quantize_fp8_tile(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                     int64_t ld, int fmt, float fmt_max, uint8_t* q,
                                     float* scales, cudaStream_t s);
cudaError_t launch_quantize_fp8_row(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                    int64_t ld, int fmt, float fmt_max, uint8_t* q, float* scales,
                                    cudaStream_t s);
// MX quantiser.  fmt: 0 E4M3, 1 E5M2 (MXFP8, one code per byte), 2 E2M1
// (MXFP4, two codes per byte); fmt_max: the value a block maximum maps to.
// tc_layout: write scales in the tcgen05 atom layout (with padding) instead
// of row-major.
cudaError_t launch_quantize_mx(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                               int64_t ld, int fmt, float fmt_max, uint8_t* q, uint8_t* sf,
                               bool tc_layout, cudaStream_t s);
// NVFP4: E2M1 codes, one E4M3 scale per 16 along K (row-major or tcgen05
// layout, padding 0), FP32 tensor scale g.
cudaError_t launch_quantize_nvfp4(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                  int64_t ld, float tensor_scale, uint8_t* q, uint8_t* sf,
                                  bool tc_layout, cudaStream_t s);
cudaError_t launch_sf_to_tcgen05(const uint8_t* sf, int64_t rows, int64_t kblocks, uint8_t* out,
                                 cudaStream_t s);

// ------------------------------------------------------------- tensor maps
// 2-D map of a byte matrix (rows x inner_bytes, row pitch `pitch`) loaded in
// boxes of box_rows x 128 bytes with 128-byte swizzling; out of range = 0.
bool make_kmajor_map(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                     uint64_t pitch, uint32_t box_rows);
// 2-D map of a row-major output matrix (rows x cols elements of elem_bytes,
// 2 or 4) stored in boxes of 128 rows x 128 bytes with 128-byte swizzling.
// Needs a 16-byte aligned base and a row pitch that is a multiple of 16 bytes.
bool make_out_map(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols, int elem_bytes);
// 3-D view [chunk][row][128 B] of the same matrix (inner_bytes % 128 == 0):
// one box brings box_chunks consecutive 128-byte chunks of box_rows rows and
// lands as box_chunks canonical (box_rows x 128 B, swizzled) slabs.
bool make_kmajor_map_chunked(CUtensorMap* map, const void* base, uint64_t inner_bytes,
                             uint64_t rows, uint64_t pitch, uint32_t box_rows,
                             uint32_t box_chunks);

// ----------------------------------------------------------------- GEMMs
struct Fp8GemmArgs {
  int M, N, K;
  int afmt, bfmt;            // 0 E4M3, 1 E5M2
  const float* sA;           // scales of A
  bool a_row;                // A scales per 1x128 ([KT][M]) instead of 128x128 ([MT][KT])
  const float* sB;
  bool b_row;
  const float* C;            // optional FP32 addend
  void* D;                   // FP32 / BF16 values, or FP8 codes when out_fp8
  bool out_bf16;
  bool out_fp8;              // quantise the result per 1x128 run of a row
  int qfmt;                  // out_fp8: 0 E4M3, 1 E5M2
  float qmax;                // out_fp8: the value a group's maximum maps to
  float* sD;                 // out_fp8: FP32 scales [ceil(N/128)][M]
  bool pair;                 // CTA-pair kernel (256 x 256 tiles, tcgen05 cta_group::2)
  bool tma_out;              // tmD is valid: D is written by TMA tensor stores
  CUtensorMap tmA, tmB;      // K-major operand maps (box 128 B x rows)
  CUtensorMap tmD;           // output map (box 128 B x 128 rows, 128-byte swizzle)
};
// Whether a problem takes the CTA-pair kernel, and the B box height it needs.
bool gemm_fp8_use_pair(int M, int N, int num_sms);
int gemm_fp8_b_box_rows(bool pair);
cudaError_t launch_gemm_fp8(const Fp8GemmArgs& a, int num_sms, cudaStream_t s);

// Block-scaled GEMM for large shapes (128 x 256 tiles): MXFP8 (FP8 operands,
// E8M0 per 32), MXFP4 (packed E2M1, E8M0 per 32) or NVFP4 (packed E2M1, E4M3
// per 16, times alpha); scales in the tcgen05 layout.
struct MxGemmArgs {
  int M, N, K;
  int kind;                  // 0 MXFP8, 1 MXFP4, 2 NVFP4
  float alpha;               // NVFP4: the sum is multiplied by alpha
  int afmt, bfmt;            // MXFP8: 0 E4M3, 1 E5M2
  const uint8_t* sfA;
  const uint8_t* sfB;
  const float* C;
  void* D;
  bool out_bf16;
  bool pair;                 // CTA-pair kernel (256 x 256 tiles, tcgen05 cta_group::2)
  CUtensorMap tmA, tmB;      // A: box 128 B x 128 rows; B: box 128 B x gemm_mx_b_box_rows(pair)
};
int gemm_mx_b_box_rows(bool pair);
// Whether a large block-scaled problem takes the CTA-pair kernel.
bool gemm_mx_use_pair(int M, int N, int num_sms);
// Whether an FP4 problem takes this kernel rather than the general FP4 one.
bool gemm_mx_fp4_large(int M, int N, int num_sms);
cudaError_t launch_gemm_mx(const MxGemmArgs& a, int num_sms, cudaStream_t s);

struct Mxfp4GemmArgs {
  int M, N, K;
  bool nvfp4;                // E4M3 scales per 16 (general kernel only)
  float alpha;               // nvfp4: the sum is multiplied by alpha
  const uint8_t* sfA;        // tcgen05 layout
  const uint8_t* sfB;
  const float* C;
  void* D;
  bool out_bf16;
  CUtensorMap tmA, tmB;      // packed operands (box 128 B x rows); the decode
                             // launcher encodes its own maps from A and B
  const void* A;
  const void* B;
  void* workspace;           // split-K partials + tile counters (decode path)
  size_t workspace_bytes;
  // decode path with the activations quantised in the kernel (xsrc != null):
  // xsrc M x K, FP32 or BF16, row pitch ldx; A and sfA are not used then
  const void* xsrc;
  int64_t ldx;
  bool xsrc_bf16;
};
cudaError_t launch_gemm_mxfp4(const Mxfp4GemmArgs& a, int num_sms, cudaStream_t s);
// Decode-shaped (small M) MXFP4 GEMM: weights B stream once; A has M <= 32 rows.
size_t gemm_mxfp4_decode_workspace(int M, int N, int K, int num_sms);
cudaError_t launch_gemm_mxfp4_decode(const Mxfp4GemmArgs& a, int num_sms, cudaStream_t s);
// MXFP4 GEMM with on-the-fly activation quantisation.  Up to kActFusedMaxM
// activation rows the decode kernel quantises them stage by stage; above,
// its four scale-writer warps could not keep up with the weight stream, so
// the stand-alone quantiser runs first.  Workspace: the decode kernel's
// split-K area (M <= 32, at off[0] = 0), then for M > kActFusedMaxM the
// activation codes (M x K/2, at off[1]) and scale atoms (ceil(M/128) x
// ceil(K/128) x 512 bytes, at off[2]).
constexpr int kActFusedMaxM = 4;
size_t gemm_mxfp4_act_workspace(int M, int N, int K, int num_sms, size_t* off);

// FP4 GEMM with a BF16 or FP16 scale per 32 along K (codes [K/32][rows]),
// promoted per K block.  A and B are packed E2M1 (rows x K/2 bytes); their
// tensor maps use the 16U4_ALIGN16B type (box 128 elements x 128 rows for A,
// gemm_bs16_b_box_rows() for B).
struct Bs16GemmArgs {
  int M, N, K;               // K % 128 == 0
  bool f16_scales;           // FP16 scale codes (else BF16)
  const uint16_t* sfA;
  const uint16_t* sfB;
  const float* C;
  void* D;
  bool out_bf16;
  bool vec_out;              // D is 16-byte aligned and rows are whole 16-byte pieces
  CUtensorMap tmA, tmB;
};
cudaError_t launch_gemm_bs16(const Bs16GemmArgs& a, int num_sms, cudaStream_t s);
int gemm_bs16_b_box_rows();        // B rows per tile (the B map's box height)
cudaError_t gemm_bs16_error_read_and_clear(cudaStream_t s, uint32_t* out);
// 2-D map of a packed E2M1 matrix (rows x K values, row pitch `pitch` bytes)
// that unpacks on load (16U4_ALIGN16B): box 128 values x box_rows, 128-byte
// swizzle.  Needs K % 128 == 0, a 32-byte aligned base and pitch % 32 == 0.
bool make_fp4_unpack_map(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows,
                         uint64_t pitch, uint32_t box_rows);
// FP4 quantiser with a BF16 / FP16 scale per 32 along K (codes [K/32][rows]).
cudaError_t launch_quantize_fp4_bs16(const void* x, bool src_bf16, int64_t rows, int64_t cols,
                                     int64_t ld, bool f16_scales, uint8_t* q, uint16_t* sf,
                                     cudaStream_t s);

// ------------------------------------------------- tensor-core microbenchmark
// Back-to-back tcgen05.mma from shared memory on every SM; *flops receives
// the floating-point operations the launch performs.  kind: 0 dense FP8,
// 1 block-scaled FP8 (single CTA only), 2 block-scaled FP4.
cudaError_t launch_mma_peak(int kind, bool pair, int64_t iters, int num_sms, cudaStream_t s,
                            int64_t* flops);

// One tcgen05.mma kind::f8f6f4: D[128][16] = A[128][32] . B[16][32]^T + C
// (row-major device arrays; fmt 0 E4M3, 1 E5M2).
cudaError_t launch_mma_probe(const uint8_t* A, int afmt, const uint8_t* B, int bfmt, const float* C,
                             float* D, cudaStream_t s);
// One block-scaled tcgen05.mma of the GEMMs' shape (M128 N256): kind 0
// kind::mxf8f6f4 1X (FP8 formats afmt / bfmt), 1 kind::mxf4 2X, 2
// kind::mxf4nvf4 4X.  A [128][32] / B [256][32] operand bytes as in shared
// memory, sfA [128][4] / sfB [256][4] scale cells, C / D [128][256] FP32.
cudaError_t launch_mma_probe_mx(int kind, const uint8_t* A, const uint8_t* sfA, const uint8_t* B,
                                const uint8_t* sfB, const float* C, float* D, int afmt, int bfmt,
                                cudaStream_t s);
// A kernel whose only wait runs out (the failure-detection self-check).
cudaError_t launch_wait_timeout_check(cudaStream_t s);
cudaError_t watchdog_error_read_and_clear(cudaStream_t s, uint32_t* out);

}  // namespace bsg

/*
 * bsg.h - block-scaled low-precision GEMM on GB300 (sm_103a): the C ABI of
 * libbsg.so.
 *
 * The library computes
 *
 *     D = sum_k (s_A a_k)(s_B b_k) + C          (FP32 accumulation)
 *
 * for FP8 operands (E4M3 / E5M2) with per-tile FP32 scales and for MXFP4
 * operands (E2M1 values, one E8M0 power-of-two scale per 32 elements along K),
 * and the quantisers that produce those operands from FP32 or BF16 sources.
 *
 * Sources of the operations (web pages on the subject; each entry point below
 * names its passage):
 *   "FP8 GEMM on CDNA4"          - per-tile scale max_abs/448, FP32 accumulation,
 *                                  write-back times s_A*s_B (sections 2.2, 3.3, 4.2, 4.4)
 *   "Rubin FP4 GEMM deep dive"   - MXFP4: E2M1, E8M0 per 32 along K, nibble order,
 *                                  A row-major / B column-major (sections 2.1-2.2, 3.1-3.4, 4.2)
 *   "FP8 MMA internals on Hopper"- why per-K-tile promotion into an FP32
 *                                  accumulator is needed
 *
 * Conventions shared by every entry point
 *   - Every pointer argument named as a device buffer is a CUDA device pointer
 *     on the current device; the caller allocates and owns it.  The library
 *     never allocates device memory and never frees a caller's buffer.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every compute call is asynchronous on that stream; buffers
 *     must stay alive until the stream has passed the call.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error status and launches nothing.
 *   - Device-side failures (a bounded wait that ran out) never trap: the
 *     kernel records them in a device error word and returns; read it with
 *     bsg_device_error().
 *   - Matrices are row-major with a leading dimension in elements unless a
 *     comment says otherwise.  Operand B of a GEMM is K x N column-major,
 *     i.e. stored as N rows of K contiguous elements (N x K row-major).
 */
#ifndef BSG_H_
#define BSG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BSG_OK = 0,
  BSG_ERR_INVALID_ARG = 1,   /* null pointer, negative or zero size, bad enum        */
  BSG_ERR_UNSUPPORTED = 2,   /* format / granularity / dtype combination not offered */
  BSG_ERR_ALIGNMENT = 3,     /* pointer or leading dimension not 16-byte aligned     */
  BSG_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, attribute, ...)  */
  BSG_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out (bsg_device_error) */
  BSG_ERR_WORKSPACE = 6      /* workspace missing or smaller than bsg_gemm_workspace_size */
} bsg_status;

typedef enum {
  BSG_E4M3 = 0,              /* FP8, 4-bit exponent, 3-bit mantissa, "fn": max 448, no Inf */
  BSG_E5M2 = 1,              /* FP8, 5-bit exponent, 2-bit mantissa, max 57344            */
  BSG_E2M1 = 2               /* FP4, values {0,.5,1,1.5,2,3,4,6} with sign, 2 per byte,
                                first element in the low nibble                            */
} bsg_format;

typedef enum {
  BSG_F32 = 0,
  BSG_BF16 = 1
} bsg_dtype;

typedef enum {
  /* One FP32 scale per 128 x 128 tile.  Scale array [ceil(R/128)][ceil(C/128)]
     row-major, R = rows of the quantised matrix, C = its K extent.           */
  BSG_SCALE_TILE128x128 = 0,
  /* One FP32 scale per 1 x 128 run of a row.  Stored K-tile major:
     [ceil(C/128)][R], so the scales of one K tile are contiguous.            */
  BSG_SCALE_ROW1x128 = 1,
  /* One E8M0 scale per 1 x 32 block along K (MXFP4); layout per bsg_sf_layout */
  BSG_SCALE_BLOCK1x32_E8M0 = 2,
  /* One E4M3 scale per 1 x 16 block along K (NVFP4); layout per bsg_sf_layout,
     tcgen05 padding bytes 0.                                                  */
  BSG_SCALE_BLOCK1x16_E4M3 = 3,
  /* One BF16 / FP16 scale per 1 x 32 block along K (E2M1 elements; "Rubin
     FP4 GEMM deep dive", section 3.2).  16-bit codes stored K-block major,
     [C/32][R], so one K block's scales are contiguous.                       */
  BSG_SCALE_BLOCK1x32_BF16 = 4,
  BSG_SCALE_BLOCK1x32_F16 = 5
} bsg_scale_gran;

typedef enum {
  /* Canonical E8M0 layout: [R][C/32] bytes, row-major.                        */
  BSG_SF_ROWMAJOR = 0,
  /* The order the block-scaled tensor-core MMA reads scales in: 512-byte
     atoms ordered by (row block of 128, group of 4 K-blocks); inside an atom
     the byte of row r, K-block c is at (r%32)*16 + ((r%128)/32)*4 + (c%4).
     Size ceil(R/128) * ceil(C/128) * 512 bytes; padding bytes hold 127 (1.0).
     bsg_gemm reads MXFP4 scales in this layout only.                          */
  BSG_SF_TCGEN05 = 1
} bsg_sf_layout;

/* ------------------------------------------------------------------------ */
/* bsg_quantize_fp8 - per-tile FP8 quantisation.
 *
 * "FP8 GEMM on CDNA4", section 3.3 (scale = max_abs / 448, each element divided
 * by the scale and stored as FP8) and section 4.2 (warp-level max reduction).
 * For each scale group G (a 128 x 128 tile or a 1 x 128 run, per `gran`):
 *     s_G = max_{x in G} |x| / fmt_max       (FP32, round to nearest; 1.0 if 0)
 *     q   = RNE_satfinite_fmt(x / s_G)       (IEEE FP32 division)
 *
 * x        device, rows x cols source, leading dimension `ld` elements,
 *          FP32 or BF16 per `src`.  Finite values only.
 * fmt      BSG_E4M3 or BSG_E5M2.
 * gran     BSG_SCALE_TILE128x128 or BSG_SCALE_ROW1x128.
 * fmt_max  the value the group maximum maps to; 0 selects the format's own
 *          maximum (448 for E4M3, 57344 for E5M2).  Must be >= 0 and finite.
 * q        device, rows x cols codes, leading dimension `cols` bytes.
 * scales   device, FP32 scales in the layout `gran` describes.
 * Errors: BSG_ERR_INVALID_ARG (null, rows/cols <= 0, ld < cols, bad fmt_max,
 *         more than 65535 * 128 rows for 128 x 128 scales or more than
 *         65535 * 512 columns for 1 x 128 scales),
 *         BSG_ERR_UNSUPPORTED (fmt or gran not FP8), BSG_ERR_CUDA.
 */
bsg_status bsg_quantize_fp8(const void* x, bsg_dtype src, int64_t rows, int64_t cols,
                            int64_t ld, bsg_format fmt, bsg_scale_gran gran, float fmt_max,
                            uint8_t* q, float* scales, void* stream);

/* bsg_quantize_mxfp4 - MXFP4 quantisation.
 *
 * "Rubin FP4 GEMM deep dive", section 4.2 steps 1-3: per block of 32
 * consecutive elements along a row, v = max|x| / 6 (FP32); the E8M0 scale is
 * the power of two nearest to v (linear distance, a tie goes to the larger;
 * v = 0 gives 1.0; codes clamp to [0, 254]); each element is multiplied by the
 * inverse power of two (exact) and rounded to E2M1 (nearest, ties to even,
 * saturating at 6); two codes per byte, first element in the low nibble.
 *
 * x        device, rows x cols source (FP32 or BF16), leading dimension `ld`.
 * cols     K extent, a multiple of 32.
 * q_packed device, rows x cols/2 bytes, leading dimension cols/2.
 * sf       device, E8M0 scales in `layout` (bsg_scale_bytes gives the size).
 * Errors: BSG_ERR_INVALID_ARG (null, sizes, cols % 32), BSG_ERR_CUDA.
 */
bsg_status bsg_quantize_mxfp4(const void* x, bsg_dtype src, int64_t rows, int64_t cols,
                              int64_t ld, uint8_t* q_packed, uint8_t* sf,
                              bsg_sf_layout layout, void* stream);

/* bsg_quantize_mx - MX quantisation with E2M1 (MXFP4) or FP8 (MXFP8) elements.
 *
 * "Rubin FP4 GEMM deep dive", section 2.2 (32 consecutive elements along K
 * share one E8M0 scale) and section 4.2 steps 1-3, with the element format's
 * largest value in place of E2M1's 6 for FP8 elements: per block,
 * v = max|x| / fmt_max (FP32), the E8M0 scale is the power of two nearest to v
 * (as bsg_quantize_mxfp4), and each element times the inverse power of two
 * (exact) is rounded to the element format (nearest, ties to even,
 * saturating).  Taking the E2M1 rule unchanged for FP8 elements is a reading.
 *
 * fmt      BSG_E2M1 (codes packed two per byte, first element in the low
 *          nibble: rows x cols/2 bytes), BSG_E4M3 or BSG_E5M2 (one code per
 *          byte: rows x cols bytes).
 * fmt_max  0 selects the format's own maximum (6, 448, 57344); otherwise any
 *          positive finite value.
 * Other arguments as bsg_quantize_mxfp4.  q must be 8-byte aligned for FP8.
 * Errors: BSG_ERR_INVALID_ARG (null, sizes, cols % 32, bad fmt or fmt_max),
 *         BSG_ERR_ALIGNMENT, BSG_ERR_CUDA.
 */
bsg_status bsg_quantize_mx(const void* x, bsg_dtype src, int64_t rows, int64_t cols, int64_t ld,
                           bsg_format fmt, float fmt_max, uint8_t* q, uint8_t* sf,
                           bsg_sf_layout layout, void* stream);

/* bsg_quantize_nvfp4 - NVFP4 quantisation: E2M1 elements, one E4M3 scale per
 * 16 elements along K, one FP32 tensor scale g.
 *
 * "Rubin FP4 GEMM deep dive", section 5.3 (blocks of 16 give finer scales) and
 * section 2.2 (the block scale kept in a higher-precision format such as FP8).
 * Per block: v = max|x| / 6 and u = v / g (FP32, round to nearest); the scale
 * code is u rounded to E4M3 (nearest even, saturating at 448); the block's
 * scale is s = E4M3(code) * g (FP32); each element is x / s (IEEE FP32
 * division) rounded to E2M1 (nearest even, saturating at 6); a block whose s
 * is 0 stores zero codes.  g (not on the pages) lets the E4M3 scales cover
 * data of any magnitude; pass alpha = g_A * g_B to bsg_gemm_nvfp4.
 *
 * x, src, rows, ld  as bsg_quantize_mxfp4.
 * cols     K extent, a multiple of 16.
 * tensor_scale  g: finite, >= 2^-126.
 * q_packed device, rows x cols/2 bytes (first element in the low nibble),
 *          4-byte aligned.
 * sf       device, E4M3 codes in `layout` (bsg_scale_bytes with
 *          BSG_SCALE_BLOCK1x16_E4M3 gives the size; tcgen05 padding 0).
 * Errors: BSG_ERR_INVALID_ARG (null, sizes, cols % 16, bad g),
 *         BSG_ERR_ALIGNMENT, BSG_ERR_CUDA.
 */
bsg_status bsg_quantize_nvfp4(const void* x, bsg_dtype src, int64_t rows, int64_t cols,
                              int64_t ld, float tensor_scale, uint8_t* q_packed, uint8_t* sf,
                              bsg_sf_layout layout, void* stream);

/* bsg_quantize_fp4_bs16 - E2M1 elements with a 16-bit scale per 32 along K.
 *
 * "Rubin FP4 GEMM deep dive", section 3.2: where the power-of-two E8M0 scale
 * is too coarse, the block scale is kept in FP16 or BF16 at twice the scale
 * bytes; the block of 32 along K and the E2M1 element rule are those of
 * sections 2.2 and 4.2.  Per block:
 *     v  = max |x| / 6                 (FP32, round to nearest)
 *     s  = v rounded to nearest even in BF16 or FP16 (FP16 saturates at 65504)
 *     q  = RNE_satfinite_E2M1(x / s)   (IEEE FP32 division); s = 0 -> codes 0
 *
 * x         device, rows x cols FP32 or BF16 source (leading dimension ld);
 *           finite values only; cols % 32 == 0.
 * gran      BSG_SCALE_BLOCK1x32_BF16 or BSG_SCALE_BLOCK1x32_F16.
 * q_packed  device, rows x cols/2 bytes, first element in the low nibble;
 *           4-byte aligned.
 * sf        device, [cols/32][rows] 16-bit scale codes (bsg_scale_bytes).
 * The GEMM takes these operands through bsg_gemm (E2M1 x E2M1 with the same
 * granularity on both sides, K % 128 == 0, A and B 32-byte aligned).
 * Errors: BSG_ERR_INVALID_ARG, BSG_ERR_UNSUPPORTED (other gran),
 *         BSG_ERR_ALIGNMENT, BSG_ERR_CUDA. */
bsg_status bsg_quantize_fp4_bs16(const void* x, bsg_dtype src, int64_t rows, int64_t cols,
                                 int64_t ld, bsg_scale_gran gran, uint8_t* q_packed, uint16_t* sf,
                                 void* stream);

/* bsg_gemm - block-scaled GEMM D = sum_k (s_A a_k)(s_B b_k) + C.
 *
 * "FP8 GEMM on CDNA4", sections 2.2 (FP32 accumulation), 3.3 and 4.4 (the
 * accumulated result is multiplied by s_A * s_B); "Rubin FP4 GEMM deep dive",
 * sections 2.2 and 3.1 (K-blocked scaling: each K block's partial sum is
 * multiplied by its two scales before it is accumulated).  FP8 scales are not
 * powers of two, so the FP8 path multiplies each 128-wide K tile's partial
 * sum by s_A * s_B and adds it into an FP32 accumulator (the per-K-tile
 * promotion "FP8 MMA internals on Hopper" motivates).  MXFP4 scales are
 * applied by the tensor core.  BF16 / FP16 block scales ("Rubin FP4 GEMM deep
 * dive", section 3.2) are not powers of two either: the E2M1 partial of every
 * 32-wide K block is promoted as fma(s_A * s_B, P, acc), blocks in K order.
 *
 * A   device, M x K codes, row-major: FP8 one byte per element (leading
 *     dimension K bytes), E2M1 packed (K/2 bytes per row).
 * B   device, K x N column-major = N x K row-major, same encoding rules.
 * fa, fb  operand formats: both FP8 (E4M3 / E5M2, any mix) or both E2M1.
 * sA, ga  A's scales: FP8 -> BSG_SCALE_TILE128x128 ([ceil(M/128)][ceil(K/128)])
 *         or BSG_SCALE_ROW1x128 ([ceil(K/128)][M]) (FP32 scales, promoted per
 *         128-wide K tile), or - for both operands together - MXFP8:
 *         BSG_SCALE_BLOCK1x32_E8M0 in the BSG_SF_TCGEN05 layout (applied by
 *         the tensor core, as bsg_quantize_mx writes them); E2M1 ->
 *         BSG_SCALE_BLOCK1x32_E8M0 in the BSG_SF_TCGEN05 layout (MXFP4), or
 *         BSG_SCALE_BLOCK1x16_E4M3 in that layout for both operands (NVFP4,
 *         alpha 1; see bsg_gemm_nvfp4; up to 32 rows the decode-shaped
 *         kernel, which needs the workspace as for MXFP4), or BSG_SCALE_BLOCK1x32_BF16 /
 *         BSG_SCALE_BLOCK1x32_F16 for both operands ([K/32][M] 16-bit codes,
 *         as bsg_quantize_fp4_bs16 writes them).
 * sB, gb  B's scales, same rules with N in place of M.
 * C   device, optional (NULL) FP32 M x N row-major addend.
 * D   device, M x N row-major output, FP32 or BF16 (round to nearest even).
 * workspace, workspace_bytes
 *     device scratch of at least bsg_gemm_workspace_size(...) bytes (may be
 *     NULL when that size is 0).  It must be zero-filled before its first use;
 *     the library leaves it zero-filled after every successful call.  Calls
 *     that share a workspace must not overlap in time.
 * Constraints: M, N, K > 0; K % 16 == 0 for FP8 with FP32 scales, K % 32 == 0
 *     for E8M0 scales; A, B 16-byte aligned (E8M0 scale arrays too); with
 *     16-bit block scales K % 128 == 0 and A, B 32-byte aligned.
 * Errors: BSG_ERR_INVALID_ARG, BSG_ERR_UNSUPPORTED, BSG_ERR_ALIGNMENT,
 *         BSG_ERR_WORKSPACE, BSG_ERR_CUDA.
 */
bsg_status bsg_gemm(int64_t M, int64_t N, int64_t K,
                    const void* A, bsg_format fa, const void* sA, bsg_scale_gran ga,
                    const void* B, bsg_format fb, const void* sB, bsg_scale_gran gb,
                    const float* C, void* D, bsg_dtype out,
                    void* workspace, size_t workspace_bytes, void* stream);

/* bsg_gemm_quantized - the promoted FP8 GEMM with its output quantised in
 * the epilogue (a quantiser fused into the producing GEMM).
 *
 * Computes R = sum_k (s_A a_k)(s_B b_k) + C exactly as bsg_gemm does with FP8
 * operands and FP32 scales (FP32 result before any output rounding), then
 * quantises R the way bsg_quantize_fp8 does with BSG_SCALE_ROW1x128 ("FP8
 * GEMM on CDNA4" section 3.3, the online scale of the next GEMM's
 * activations; "Rubin FP4 GEMM deep dive" section 4.2 step 4, activations
 * quantised at run time): for each 1 x 128 run G of a row of R,
 *     s_G = max_{x in G} |x| / fmt_max   (FP32, round to nearest; 1.0 if 0)
 *     q   = RNE_satfinite_qfmt(x / s_G)  (IEEE FP32 division)
 * so Dq and sD can be passed straight to bsg_gemm as an activation operand
 * with BSG_SCALE_ROW1x128 scales (K = N of this call).
 *
 * A, fa, sA, ga, B, fb, sB, gb, C  as bsg_gemm, FP8 operands with FP32 scales
 *          (BSG_SCALE_TILE128x128 or BSG_SCALE_ROW1x128) only.
 * qfmt     BSG_E4M3 or BSG_E5M2.
 * fmt_max  the value a group's maximum maps to; 0 selects the format's own
 *          maximum (448 / 57344).  Must be in [0, 2^64].
 * Dq       device, M x N codes, leading dimension N bytes (TMA stores when Dq
 *          is 16-byte aligned and N % 16 == 0, a bounds-checked copy else).
 * sD       device, FP32 scales [ceil(N/128)][M] (4-byte aligned).
 * Constraints: M, N, K > 0, K % 16 == 0; A, B 16-byte aligned.
 * Errors: BSG_ERR_INVALID_ARG, BSG_ERR_UNSUPPORTED (non-FP8 operands, E8M0
 *         scales or qfmt), BSG_ERR_ALIGNMENT, BSG_ERR_CUDA.
 */
bsg_status bsg_gemm_quantized(int64_t M, int64_t N, int64_t K,
                              const void* A, bsg_format fa, const void* sA, bsg_scale_gran ga,
                              const void* B, bsg_format fb, const void* sB, bsg_scale_gran gb,
                              const float* C, bsg_format qfmt, float fmt_max,
                              uint8_t* Dq, float* sD, void* stream);

/* bsg_gemm_nvfp4 - NVFP4 GEMM D = alpha * sum_k (s_A a_k)(s_B b_k) + C.
 *
 * A, B: packed E2M1 (M x K/2 and N x K/2 bytes, B = K x N column-major);
 * sA, sB: E4M3 block scales in the BSG_SF_TCGEN05 layout as
 * bsg_quantize_nvfp4 writes them; the tensor core applies them (kind::
 * mxf4nvf4, FP32 accumulation across all of K).  alpha (finite; normally
 * g_A * g_B) multiplies the FP32 sum before the addend C (optional FP32
 * M x N).  D: FP32 or BF16 (nearest even), M x N row-major.  bsg_gemm with
 * BSG_SCALE_BLOCK1x16_E4M3 on both operands is the same with alpha = 1.
 * Up to M = 32 rows that takes the decode-shaped kernel, and so does
 * bsg_gemm_nvfp4_ws below; this entry point has no workspace, so for M <= 32
 * it runs the decode-shaped kernel only when no split-K workspace is needed
 * (bsg_gemm_workspace_size(M, N, K, BSG_E2M1, BSG_E2M1) == 0), else the
 * general kernel.
 * Constraints: K % 32 == 0; A, B, sA, sB 16-byte aligned.
 * Errors: BSG_ERR_INVALID_ARG, BSG_ERR_ALIGNMENT, BSG_ERR_CUDA.
 */
bsg_status bsg_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const void* A, const void* sA,
                          const void* B, const void* sB, float alpha, const float* C, void* D,
                          bsg_dtype out, void* stream);

/* bsg_gemm_nvfp4_ws - bsg_gemm_nvfp4 with a workspace, for the decode shapes
 * of "Rubin FP4 GEMM deep dive" (section 5.3, blocks of 16 with E4M3
 * scales; a memory-bound GEMM whose few activation rows meet a large weight
 * matrix).
 *
 * Same arguments, result and constraints as bsg_gemm_nvfp4, plus workspace,
 * workspace_bytes: device scratch of at least
 * bsg_gemm_workspace_size(M, N, K, BSG_E2M1, BSG_E2M1) bytes (NULL when that
 * is 0), zero-filled before its first use and left zero-filled by every
 * successful call; calls that share a workspace must not overlap in time.
 * For M <= 32 the call runs the decode-shaped kernel: the weights B are the
 * tensor core's 128-row operand and stream from HBM once, and K is split
 * evenly over all SMs (partial sums added in a fixed order, so results do
 * not depend on timing).  Larger M: as bsg_gemm_nvfp4.
 * Errors: as bsg_gemm_nvfp4, plus BSG_ERR_WORKSPACE (a workspace given that
 *     is smaller than needed or not 16-byte aligned).
 */
bsg_status bsg_gemm_nvfp4_ws(int64_t M, int64_t N, int64_t K, const void* A, const void* sA,
                             const void* B, const void* sB, float alpha, const float* C, void* D,
                             bsg_dtype out, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace bsg_gemm needs for this problem (0 if none). */
size_t bsg_gemm_workspace_size(int64_t M, int64_t N, int64_t K, bsg_format fa, bsg_format fb);

/* bsg_gemm_mxfp4_act - MXFP4 GEMM whose activations are quantised on the fly
 * ("Rubin FP4 GEMM deep dive", section 4.2: the BF16 activations of a
 * decode step are cast to MXFP4 per 32-element block right before the GEMM).
 *
 *   D = sum_k (s_A a_k)(s_B b_k) + C,  (s_A, a) = MXFP4(x) per 1 x 32 block
 *
 * x        device, M x K activations, FP32 or BF16 (src), row pitch ldx
 *          elements (ldx >= K); 4- (FP32) or 2-byte (BF16) aligned.  They are
 *          quantised exactly as bsg_quantize_mxfp4 does (E8M0 scale = power of
 *          two nearest max|x| / 6, E2M1 codes, round to nearest even), so D is
 *          bit for bit the D of bsg_quantize_mxfp4 followed by bsg_gemm.
 * B, sB    weights: packed E2M1 (N x K/2 bytes, B = K x N column-major) and
 *          E8M0 scales in the BSG_SF_TCGEN05 layout, 16-byte aligned.
 * C, D     as bsg_gemm (optional FP32 addend; FP32 or BF16 output).
 * workspace  device scratch of at least bsg_gemm_mxfp4_act_workspace_size
 *          bytes, 16-byte aligned, zero-filled before its first use.  It
 *          serves one problem shape (M, N, K): after each call the library
 *          leaves its counters and partial sums zero, but the quantised
 *          activations it holds stay, and another shape would find them
 *          where it expects zeros.  One call at a time per workspace.
 * For M <= 4 one kernel does it all: the decode GEMM quantises each stage's
 * slice of the activations itself, into the shared-memory operand the tensor
 * core reads, while the weights stream.  Larger M runs the quantiser into the
 * workspace, then bsg_gemm (the quantiser's cost grows with M, and above four
 * rows the kernel's quantising warps would slow the weight stream).
 * Constraints: M, N, K > 0, K % 32 == 0.
 * Errors: BSG_ERR_INVALID_ARG, BSG_ERR_ALIGNMENT, BSG_ERR_WORKSPACE,
 *         BSG_ERR_CUDA; a wait that ran out sets the device error word.
 */
bsg_status bsg_gemm_mxfp4_act(int64_t M, int64_t N, int64_t K, const void* x, bsg_dtype src,
                              int64_t ldx, const void* B, const void* sB, const float* C, void* D,
                              bsg_dtype out, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace bsg_gemm_mxfp4_act needs (0 for sizes it rejects). */
size_t bsg_gemm_mxfp4_act_workspace_size(int64_t M, int64_t N, int64_t K);

/* Bytes of the scale array of a rows x cols matrix for a granularity and,
 * for E8M0 scales, a layout (the layout is ignored for FP32 scales). */
size_t bsg_scale_bytes(int64_t rows, int64_t cols, bsg_scale_gran gran, bsg_sf_layout layout);

/* bsg_sf_to_tcgen05 - rewrite row-major E8M0 scales [rows][kblocks] into the
 * BSG_SF_TCGEN05 layout (a permutation plus padding with 127).
 * sf_rowmajor, sf_tc: device buffers; sf_tc holds
 * bsg_scale_bytes(rows, 32*kblocks, BSG_SCALE_BLOCK1x32_E8M0, BSG_SF_TCGEN05). */
bsg_status bsg_sf_to_tcgen05(const uint8_t* sf_rowmajor, int64_t rows, int64_t kblocks,
                             uint8_t* sf_tc, void* stream);

/* bsg_gemm_decode_noalloc - the decode-shaped MXFP4 GEMM (E2M1 x E2M1,
 * M <= 32, same operands, scales, addend and output as bsg_gemm) without a
 * caller-provided workspace.  The pages have no counterpart: this is an
 * interface for callers that cannot allocate device memory, such as a
 * plug-in that a serving runtime hands only its input and output buffers,
 * or a decode loop that keeps cudaMalloc (which may synchronise the device
 * and may fail) out of its steady state.
 *
 * Scratch: a fixed 8 MiB array compiled into the library's device image;
 * every GPU that loads libbsg.so holds it until the process exits.  The
 * first call on a device looks up the array's device address (with that
 * device current), so make that first call before any stream capture.
 * Each call clears the per-tile counters that must start at zero (an
 * asynchronous memset on `stream`) and then runs the decode kernel; nothing
 * is allocated.  The looked-up address is kept for the process's lifetime,
 * so cudaDeviceReset after the first call on a device is not supported.
 * All calls share
 * the one array: calls whose execution overlaps on the GPU (different
 * streams, or different host threads) race and give wrong results.
 * Errors: as bsg_gemm; BSG_ERR_UNSUPPORTED if M > 32; BSG_ERR_WORKSPACE if
 * the problem needs more scratch than 8 MiB (bsg_gemm_workspace_size tells). */
bsg_status bsg_gemm_decode_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* sA,
                                   const void* B, const void* sB, const float* C, void* D,
                                   bsg_dtype out, void* stream);

/* bsg_mma_peak - tensor-core throughput microbenchmark (measurement only).
 *
 * No page gives GB300's FP8 or FP4 tensor rate, and no copy or library GEMM
 * measures it, so the roofline of the GEMMs above needs a measured ceiling.
 * One launch keeps every SM's tensor core busy with `iters` x 4 back-to-back
 * MMAs whose operands sit in shared memory (zero-filled; no global memory
 * traffic, no epilogue; results discarded):
 *   fmt = BSG_E4M3, block_scaled = 0: kind::f8f6f4, E4M3 x E4M3, M128 N256 K32;
 *   fmt = BSG_E4M3, block_scaled = 1: kind::mxf8f6f4.block_scale (UE8M0
 *         scales, scale_vec::1X), M128 N256 K32 (no CTA pairs);
 *   fmt = BSG_E2M1, block_scaled = 1: kind::mxf4.block_scale, M128 N256 K64.
 * pair != 0 runs CTA pairs (cta_group::2, M256 per instruction).
 * *flops (host) receives the floating-point operations of the launch
 * (2*M*N*K per MMA); divide by the launch's duration, timed by the caller
 * with events on `stream`.
 * Errors: BSG_ERR_INVALID_ARG (null flops, iters <= 0 or > 2^20),
 *         BSG_ERR_UNSUPPORTED (other combinations), BSG_ERR_CUDA. */
bsg_status bsg_mma_peak(bsg_format fmt, int block_scaled, int pair, int64_t iters, int64_t* flops,
                        void* stream);

/* bsg_mma_probe - one tensor-core MMA on given operands (verification only).
 *
 * "FP8 MMA internals on Hopper" shows that a single FP8 MMA instruction on
 * H100 is not exact (products aligned to the largest exponent, bits more than
 * 13 places below it dropped, the sum rounded toward zero to 13 fraction
 * bits) and prints test vectors with the bits H100 returns; "Exact models of
 * AMD matrix cores", section 3, models such units from test vectors and
 * random campaigns.  This entry point is the instrument for the same question
 * on this GPU: it runs exactly one tcgen05.mma kind::f8f6f4 (M128 N16 K32,
 * FP32 accumulate) and returns its result:
 *     D[128][16] = A[128][32] . B[16][32]^T + C[128][16]
 * A, B    device, FP8 codes, row-major (B's rows are the N dimension, K
 *         contiguous), formats fa / fb (BSG_E4M3 or BSG_E5M2).
 * C, D    device, FP32, row-major 128 x 16 (C is the accumulator loaded into
 *         tensor memory before the MMA).
 * Errors: BSG_ERR_INVALID_ARG (null), BSG_ERR_UNSUPPORTED (non-FP8 format),
 *         BSG_ERR_ALIGNMENT, BSG_ERR_CUDA. */
/* bsg_mma_probe_mx - one block-scaled tensor-core MMA on given operands and
 * scales (verification only).
 *
 * The block-scaled counterpart of bsg_mma_probe: "Exact models of AMD matrix
 * cores", section 3, fits a matrix unit's arithmetic with test vectors and
 * random campaigns, and "FP8 MMA internals on Hopper" gives the fused
 * dot-add structure such a fit starts from.  Runs exactly one
 *     D[128][256] = sum_k (sA_r a_rk)(sB_c b_ck) + C[128][256]
 * MMA of the shape and tensor-memory scale layout bsg_gemm's block-scaled
 * kernels use, on one CTA:
 *   kind 0  kind::mxf8f6f4.block_scale.scale_vec::1X: K = 32 FP8 values per
 *           row (formats fa, fb: BSG_E4M3 / BSG_E5M2), scale byte 0 of the
 *           row's cell (UE8M0);
 *   kind 1  kind::mxf4.block_scale.scale_vec::2X: K = 64 packed E2M1 values,
 *           bytes 0 and 1 (UE8M0) for elements 0-31 and 32-63;
 *   kind 2  kind::mxf4nvf4.block_scale.scale_vec::4X: K = 64 packed E2M1,
 *           bytes 0-3 (UE4M3) for each 16 elements.
 * A    device, [128][32] bytes: row r's operand bytes in K order (FP8 one per
 *      byte; E2M1 two per byte, first in the low nibble).
 * sfA  device, [128][4] bytes: row r's scale cell.
 * B    device, [256][32] bytes (column c of D = row c of B); sfB [256][4].
 * C    device, [128][256] FP32 accumulator in; D device, [128][256] FP32 out.
 * Errors: BSG_ERR_INVALID_ARG (null, kind not 0-2), BSG_ERR_UNSUPPORTED
 *         (kind 0 with non-FP8 formats), BSG_ERR_CUDA. */
bsg_status bsg_mma_probe_mx(int kind, const uint8_t* A, const uint8_t* sfA, const uint8_t* B,
                           const uint8_t* sfB, const float* C, float* D, bsg_format fa,
                           bsg_format fb, void* stream);

bsg_status bsg_mma_probe(const uint8_t* A, bsg_format fa, const uint8_t* B, bsg_format fb,
                         const float* C, float* D, void* stream);

/* Human-readable name of a status. */
const char* bsg_status_string(bsg_status status);

/* bsg_check_wait_timeout - self-check of the failure detection.
 *
 * Every wait inside the library's kernels is bounded (2 s); a wait that runs
 * out is reported by bsg_device_error as BSG_ERR_TIMEOUT and the kernel
 * returns instead of hanging or trapping.  This call launches one small
 * kernel whose only wait is on a barrier nothing arrives on, so the wait
 * runs out after the limit: the next bsg_device_error returns
 * BSG_ERR_TIMEOUT (and clears it), and the context stays usable.
 * Errors: BSG_ERR_CUDA (launch failure).
 */
bsg_status bsg_check_wait_timeout(void* stream);

/* Synchronise `stream`, then read and clear the device error word.  Returns
 * BSG_OK, BSG_ERR_TIMEOUT if a kernel's bounded wait ran out since the last
 * call, or BSG_ERR_CUDA if the synchronisation itself failed. */
bsg_status bsg_device_error(void* stream);

/* Number of SMs of the current device the library sizes persistent grids by
 * (0 if the query fails). */
int bsg_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* BSG_H_ */

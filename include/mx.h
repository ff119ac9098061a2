/*
 * mx.h -- C ABI of the GB300 (sm_103a) block-scaled quantization and GEMM library
 * (libmxgb.so).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are CALLER-OWNED DEVICE memory.  No call allocates or frees.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream).  No call synchronizes the host.  Kernels are launched with
 *    programmatic dependent launch: one may be scheduled while the previous kernel on the
 *    stream finishes, but it reads no memory before that kernel has completed, so stream
 *    order holds for every input, whichever kernel wrote it.
 *  - Matrices are row-major.  A GEMM computes C[m][n] = sum_k A[m][k] * B[n][k]: both code
 *    operands are K-contiguous ("TN" in column-major BLAS terms).  Column-wise quantized
 *    copies are stored physically transposed, so fprop, dgrad and wgrad all run as this one
 *    product:  fprop  Y  = X W^T : A = X row-wise,   B = W row-wise
 *              dgrad dX  = G W   : A = G row-wise,   B = W column-wise (W^T)
 *              wgrad dW  = G^T X : A = G column-wise, B = X column-wise
 *  - Arguments are validated on the host before anything is launched.  A null pointer, a
 *    shape that is not a multiple of the tile, a misaligned pointer or a bad enum value
 *    returns MX_ERR_INVALID_ARG; a valid but unimplemented combination returns
 *    MX_ERR_UNSUPPORTED; a launch failure returns MX_ERR_CUDA.  The quantizers take at most
 *    65535 tiles of 128 columns (cols <= 8388480); wider inputs return MX_ERR_INVALID_ARG.
 *  - Device-side waits are bounded.  A wait that runs out sets a device error word instead of
 *    hanging; mx_check() reports it as MX_ERR_TIMEOUT.
 *
 * Scale-factor layouts ("GEMM layout", written by the quantizers, read by the GEMMs)
 *  - MX, E8M0, one scale per 32 consecutive elements along K.  For a code matrix Q[R][K]
 *    (R % 128 == 0, K % 128 == 0) the R*K/32 scale bytes form 512-byte chunks, one per
 *    128 rows x 128 elements of K.  Chunk (rb, kc), rb < R/128, kc < K/128, starts at byte
 *    (rb * (K/128) + kc) * 512.  Inside it, the scale of row 128*rb + i and of 32-block
 *    4*kc + j is at byte (i % 32) * 16 + (i / 32) * 4 + j.
 *  - NVFP4, E4M3, one scale per 16 consecutive elements along K: the same 512-byte chunk
 *    shape, but a chunk covers 128 rows x 64 elements of K (4 blocks of 16); chunk (rb, kc),
 *    kc < K/64, starts at byte (rb * (K/64) + kc) * 512, in-chunk offset as above.
 *  - DeepSeek FP32 scales: 1x128 activation tiles are stored k-block-major, s[K/128][R]
 *    (float), so one k-block's scales for consecutive rows are contiguous; 128x128 weight
 *    blocks are stored s[R/128][K/128] (float).
 *  - Packed FP4: element 2i of a row in the low nibble of byte i, element 2i+1 in the high
 *    nibble.
 *
 * Sources (page title and section):
 *  [MX]  "MXFP8 on SM120: software support" (xuesongtap.github.io): sec 0.1 MX block format,
 *        E8M0 scale, q = Q_FP8(x / s); sec 0.3 block-scaled dot product; sec 1.1-1.2 TN/NN/NT
 *        and the fprop/dgrad/wgrad GEMM trio; sec 1.2 row-wise vs column-wise blocks.
 *  [DS]  "Why FP8 training is stable" (magicnetworld.com): sec 4 s = amax/MAX; sec 5 1x128
 *        activation tiles and 128x128 weight blocks; sec 6.3 FP32 promotion every N_C = 128.
 *  [NV]  "NVFP4: high accuracy with 4 bits" (theluyuan.com): sec 5.4 two-level scales;
 *        sec 5.6 worked example; sec 7.3-7.4 block scale outside the sum, global scale in the
 *        epilogue.
 */
#ifndef MXGB_MX_H_
#define MXGB_MX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1,
  MX_ERR_UNSUPPORTED = 2,
  MX_ERR_CUDA = 3,
  MX_ERR_TIMEOUT = 4
} mx_status;

typedef enum { MX_E4M3 = 0, MX_E5M2 = 1, MX_E2M1 = 2 } mx_elem;
typedef enum { MX_SCALE_E8M0 = 0, MX_SCALE_UE4M3 = 1, MX_SCALE_FP32 = 2, MX_SCALE_FP32_POW2 = 3 } mx_scale_fmt;
typedef enum { MX_ROWWISE = 1, MX_COLWISE = 2, MX_BOTH = 3 } mx_layout;
typedef enum { MX_OUT_F32 = 0, MX_OUT_BF16 = 1 } mx_out;

/* Version of this ABI (bumped on any signature or layout change). */
int mx_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* mx_status_string(mx_status s);

/*
 * mx_quantize -- block quantization of a bf16 matrix.  [MX] sec 0.1, [DS] sec 4-5.
 *
 * x[rows][cols]: bf16, row-major, 16-byte aligned.  Blocks run along cols (the reduction
 * axis of the consuming GEMM) for the row-wise copy and along rows for the column-wise copy.
 *
 * Supported combinations (anything else returns MX_ERR_UNSUPPORTED):
 *  1. MX: block = 32, block_rows = 1, elem = MX_E4M3 or MX_E5M2 (MXFP8) or MX_E2M1
 *     (MXFP4, [NV] sec 5.5), sfmt = MX_SCALE_E8M0, layout = ROWWISE, COLWISE or BOTH;
 *     rows % 128 == 0, cols % 128 == 0.
 *     Per block: amax = max |x|; k = clamp(floor(log2 amax) - emax, -127, 127) with emax 8
 *     (E4M3), 15 (E5M2) or 2 (E2M1), k = -127 when amax == 0; scale byte = k + 127;
 *     q = RNE-satfinite(x * 2^-k).  A NaN or Inf in a block gives scale 0xFF and all codes
 *     0x7F (E2M1: 0x7).  With BOTH, both copies come from one read of x.
 *       q_row[rows][cols] u8, s_row: rows*cols/32 bytes in the MX GEMM layout;
 *       q_col[cols][rows] u8 (transposed), s_col: the MX GEMM layout of that [cols][rows]
 *       matrix.  Pointers of a copy that is not requested may be NULL.
 *       MXFP4 codes are packed two per byte, element 2i in the low nibble:
 *       q_row[rows][cols/2], q_col[cols][rows/2].
 *  1b. MX with 2-D weight blocks: block = 32, block_rows = 32, elem = MX_E4M3 or MX_E5M2,
 *     sfmt = MX_SCALE_E8M0 ([MX] sec 1.3): one scale per 32x32 block of x by the rule of 1
 *     over the whole block, stored expanded exactly as in 1 (every 1x32 block of a row-wise
 *     row and of a column-wise row carries its 32x32 block's scale), so mx_gemm consumes it
 *     unchanged; the column-wise codes are the transpose of the row-wise ones.
 *  2. DeepSeek activations: block = 128, block_rows = 1, elem = MX_E4M3,
 *     sfmt = MX_SCALE_FP32, layout = ROWWISE; rows % 128 == 0, cols % 128 == 0.
 *     s = fl32(amax / 448) (1.0 when amax == 0); q = RNE-satfinite(fl32(x / s)).
 *       q_row[rows][cols] u8, s_row float[cols/128][rows].
 *  3. DeepSeek weights: block = 128, block_rows = 128, otherwise as 2.
 *  2/3 with sfmt = MX_SCALE_FP32_POW2: Float8BlockScaling with power-of-two scales ([MX]
 *     sec 1.3): s = 2^k with k the smallest integer such that 448 * 2^k >= amax (clamped to
 *     [-127, 127]; s = 1 when amax == 0), q = RNE-satfinite(x * 2^-k); same layouts as 2/3.
 *     mx_scales_from_fp32_blocks turns these scales into MX scales for mx_gemm.
 *       q_row[rows][cols] u8, s_row float[rows/128][cols/128].
 *     Inputs for 2 and 3 must be finite.
 */
mx_status mx_quantize(const void* x, int64_t rows, int64_t cols, int block, int block_rows,
                      mx_elem elem, mx_scale_fmt sfmt, mx_layout layout,
                      void* q_row, void* s_row, void* q_col, void* s_col, void* stream);

/*
 * mx_quantize_dual -- MX quantization of one bf16 matrix into both element formats at once:
 * E4M3 and E5M2 codes with their E8M0 scales, row-wise and/or column-wise, from a single read of
 * x.  Each output is exactly what mx_quantize (block = 32, MX_SCALE_E8M0) writes for that format.
 * [MX] sec 0.1 (block format; E4M3 and E5M2 are both MXFP8 element encodings) and sec 1.2
 * (row-wise and column-wise copies).  Shapes, alignment and layouts as in mx_quantize; the eight
 * output pointers of the requested copies must be non-NULL.
 */
mx_status mx_quantize_dual(const void* x, int64_t rows, int64_t cols, mx_layout layout,
                           void* q_row_e4m3, void* s_row_e4m3, void* q_col_e4m3, void* s_col_e4m3,
                           void* q_row_e5m2, void* s_row_e5m2, void* q_col_e5m2, void* s_col_e5m2,
                           void* stream);

/*
 * mx_gemm -- MX block-scaled GEMM (MXFP8, MXFP4).  [MX] sec 0.3, [NV] sec 5.5:
 *   C[m][n] = sum_b sA[m][b] sB[n][b] sum_{i<32} qA[m][32b+i] qB[n][32b+i], FP32 accumulate.
 *
 * qa[M][K], qb[N][K]: E4M3 or E5M2 codes (ea, eb), 16-byte aligned; sa, sb: E8M0 scales in
 * the MX GEMM layout.  out: M rows of ldc elements (ldc >= N, ldc % 8 == 0), FP32 or bf16
 * (RNE).  M % 128 == 0, N % 128 == 0, K % 128 == 0.
 * MXFP4: ea = eb = MX_E2M1, qa[M][K/2], qb[N][K/2] packed (element 2i in the low nibble, as
 * mx_quantize writes them), K % 256 == 0.  An E2M1 operand with an FP8 one returns
 * MX_ERR_UNSUPPORTED.
 */
mx_status mx_gemm(const void* qa, const void* sa, mx_elem ea,
                  const void* qb, const void* sb, mx_elem eb,
                  int64_t M, int64_t N, int64_t K,
                  void* out, mx_out out_dtype, int64_t ldc, void* stream);

/*
 * nvfp4_quantize_ex -- NVFP4 with the training options of [DS] sec 13 and [NV] sec 3.2.
 *
 * Same arguments, layouts and limits as nvfp4_quantize, plus:
 *   use_rht = 1: every 1x16 block along cols is first replaced by 0.25 * H16 * (d .* x), H16
 *     the 16x16 Sylvester Hadamard matrix and d_i = -1 where bit i of rht_signs is set (the
 *     random signs are an input; rht_signs <= 0xFFFF).  Computed in FP32 with butterflies in
 *     the order h = 1, 2, 4, 8; the global maximum, block scales and codes are those of the
 *     transformed values.  Operands transformed with the same signs multiply to the same
 *     product (0.25 H16 is orthogonal and symmetric).
 *   rbits != NULL: stochastic rounding of the element codes.  rbits[rows][cols] (u8, 16-byte
 *     aligned) holds one random byte r per element; with y = fl32(x / s_hat), |y| < 6 lying
 *     between E2M1 values lo <= |y| < hi, the code rounds up iff r < floor(256 (|y| - lo) /
 *     (hi - lo)); |y| >= 6 gives 6.  NULL: round to nearest even as nvfp4_quantize.
 * use_rht not 0/1 or rht_signs > 0xFFFF: MX_ERR_INVALID_ARG.
 */
mx_status nvfp4_quantize_ex(const void* x, int64_t rows, int64_t cols, int use_rht, uint32_t rht_signs,
                            const void* rbits, void* q_packed, void* s_ue4m3, float* gscale, void* workspace,
                            void* stream);

/*
 * nvfp4_quantize_2d -- NVFP4 with 16x16 2-D blocks (weights, [DS] sec 13).
 *
 * One E4M3 block scale per 16x16 block of x (the recipe of nvfp4_quantize with the block maximum
 * over 256 elements; same global scale), written for both orientations: q_row[rows][cols/2] and
 * s_row (the NVFP4 GEMM layout of [rows][cols/16]) as nvfp4_quantize writes them, and
 * q_col[cols][rows/2], s_col (the layout of [cols][rows/16]) for the transposed matrix; the two
 * hold the same codes and scales.  rows % 128 == 0, cols % 128 == 0; workspace as for
 * nvfp4_quantize.
 */
mx_status nvfp4_quantize_2d(const void* x, int64_t rows, int64_t cols, void* q_row, void* s_row, void* q_col,
                            void* s_col, float* gscale, void* workspace, void* stream);

/*
 * mx_scales_from_fp32_blocks -- Float8BlockScaling scales in MX form.  [MX] sec 1.3.
 *
 * s: power-of-two FP32 block scales as mx_quantize(block = 128, sfmt = MX_SCALE_FP32_POW2)
 * writes them: block_rows = 1 -> float[cols/128][rows] (1x128 tiles of a [rows][cols] code
 * matrix), block_rows = 128 -> float[rows/128][cols/128] (128x128 blocks); 4-byte aligned.
 * s_e8m0: rows*cols/32 bytes (16-byte aligned), written in the MX GEMM layout of the
 * [rows][cols] code matrix: each 1x32 block gets its 128-block's scale 2^k as the E8M0 code
 * k + 127; a scale that is not exactly 2^k with -127 <= k <= 127 becomes the E8M0 NaN code 0xFF
 * (products that use it are NaN).  The E4M3 codes are passed to mx_gemm as they are.
 * rows % 128 == 0, cols % 128 == 0, block_rows 1 or 128, else MX_ERR_INVALID_ARG.
 */
mx_status mx_scales_from_fp32_blocks(const float* s, int64_t rows, int64_t cols, int block_rows, void* s_e8m0,
                                     void* stream);

/*
 * mx_selftest_wait_timeout -- exercises the failure path of the device-side waits.  Launches one
 * CTA that waits on an mbarrier nothing ever arrives on, through the same bounded wait the GEMM
 * kernels use, with a budget of budget_us microseconds (1 .. 1000000) instead of the kernels'
 * 2 s.  The wait runs out, records its site in the device error word and the kernel returns; the
 * next mx_check() on the stream reports MX_ERR_TIMEOUT (and clears the word).  Nothing faults
 * and the context stays usable.  Returns MX_ERR_INVALID_ARG for a budget out of range.
 */
mx_status mx_selftest_wait_timeout(int64_t budget_us, void* stream);

/*
 * mx_unswizzle_scales / mx_swizzle_scales -- byte permutations between the GEMM scale layout
 * (the chunked layout described at the top of this header, as the quantizers write it and the
 * GEMMs read it) and a plain row-major matrix s_plain[rows][nblocks], one byte per block:
 * nblocks = K/32 for MX (E8M0) scales and K/16 for NVFP4 (E4M3) scales of a [rows][K] code
 * matrix.  For inspecting scales, comparing them with another implementation, or bringing in
 * scales computed elsewhere.  Both buffers are device memory of rows*nblocks bytes and must not
 * overlap; the chunked one 16-byte aligned, the plain one 4-byte aligned.
 * rows % 128 == 0, nblocks % 4 == 0, else MX_ERR_INVALID_ARG.  No arithmetic: bytes move as
 * they are.
 */
mx_status mx_unswizzle_scales(const void* s_gemm, int64_t rows, int64_t nblocks, void* s_plain, void* stream);
mx_status mx_swizzle_scales(const void* s_plain, int64_t rows, int64_t nblocks, void* s_gemm, void* stream);

/*
 * mx_gemm_mxout -- MXFP8 GEMM whose epilogue quantizes its own results for the next product
 * (producer-side fusion of the MX quantization; [MX] sec 0.1 rule, [DS] sec 9 quantizes the
 * activations that feed the next FP8 product before they leave).
 *
 * The product of mx_gemm (same operands, formats and FP32 accumulation), then per 1x32 block of
 * each output row the MX quantization of the FP32 results into out_elem (MX_E4M3 or MX_E5M2):
 * scale byte max(exp(amax) - emax, 0) (0xFF and codes 0x7F when a result is Inf or NaN), codes
 * RNE-satfinite(y * 2^-k).  q_out[M][ldq] u8 codes (ldq >= N, ldq % 16 == 0), s_out: M*N/32
 * bytes in the MX GEMM layout of [M][N] -- exactly the A operand of a following mx_gemm.
 * No bf16 / FP32 output is written.  M % 256 == 0, N % 256 == 0, K % 128 == 0.
 */
mx_status mx_gemm_mxout(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb,
                        int64_t M, int64_t N, int64_t K, mx_elem out_elem, void* q_out, void* s_out, int64_t ldq,
                        void* stream);

/*
 * mx_gemm_mxout_ex -- mx_gemm_mxout with the copies a training step needs ([MX] sec 1.2: a
 * transpose needs its own blocks, scales and codes): layout MX_ROWWISE writes the row-wise copy
 * exactly as mx_gemm_mxout (q_row[M][ldq_row], s_row in the MX GEMM layout of [M][N]);
 * MX_COLWISE writes the column-wise copy -- 32x1 blocks down each column of the result, stored
 * transposed like mx_quantize's column-wise output: q_col[N][ldq_col] codes (ldq_col >= M,
 * ldq_col % 16 == 0) and s_col: M*N/32 bytes in the MX GEMM layout of [N][M], i.e. the operand of
 * a following product that reduces over M; MX_BOTH writes both from the same FP32 results.  Same
 * scale and code rule as mx_gemm_mxout per block.  Pointers of a copy not requested may be NULL.
 * M % 256 == 0, N % 256 == 0, K % 128 == 0.
 */
mx_status mx_gemm_mxout_ex(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb,
                           int64_t M, int64_t N, int64_t K, mx_elem out_elem, mx_layout layout, void* q_row,
                           void* s_row, int64_t ldq_row, void* q_col, void* s_col, int64_t ldq_col, void* stream);

/*
 * mx_gemm_grouped -- MXFP8 expert GEMMs of a mixture-of-experts layer in one launch.  [MX]
 * sec 1.2 (grouped GEMM is its own entry point besides the single GEMMs).
 *
 * groups G (1..1024); group g multiplies rows off[g] .. off[g+1]-1 of A by the g-th block of B:
 *   C[m][n] = sum_b sA[m][b] sB[gN + n][b] sum_{i<32} qA[m][32b+i] qB[gN + n][32b+i]
 * for off[g] <= m < off[g+1], with the block scaling of mx_gemm.
 * qa[M][K] (all groups' rows stacked), sa its E8M0 scales in the MX GEMM layout of [M][K];
 * qb[G*N][K] (block g = rows gN .. gN+N-1), sb the layout of [G*N][K]; out M rows of ldc
 * elements.  group_offsets: device int64[G + 1], 8-byte aligned, read by the kernel (so the
 * expert sizes can come from device-side routing without a host round trip); they must satisfy
 * off[0] = 0, off[G] = M, off[g] <= off[g+1] and off[g] % 128 == 0 (an empty group is allowed).
 * Offsets that break this make the call do nothing and mx_check return MX_ERR_INVALID_ARG.
 * M % 128 == 0, N % 256 == 0, K % 128 == 0, element formats as mx_gemm: MXFP8 (E4M3 / E5M2) or
 * MXFP4 (both MX_E2M1, codes packed as mx_quantize writes them, K % 256 == 0).
 */
mx_status mx_gemm_grouped(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb,
                          const int64_t* group_offsets, int64_t groups, int64_t M, int64_t N, int64_t K, void* out,
                          mx_out out_dtype, int64_t ldc, void* stream);

/*
 * nvfp4_gemm_grouped -- NVFP4 expert GEMMs in one launch: group g computes, for its rows
 * off[g] <= m < off[g+1],  C[m][n] = s_gA * s_gB[g] * sum_b sA[m][b] sB[gN + n][b] sum_{i<16} qA qB
 * ([NV] sec 7.3-7.4; each expert's weights are quantized as their own tensor, so each has its own
 * global scale).  qa[M][K/2] packed E2M1 with sa in the NVFP4 GEMM layout of [M][K] and one global
 * scale ga (device float); qb[G*N][K/2] with sb the layout of [G*N][K] and gb: device float[G].
 * group_offsets as mx_gemm_grouped.  M % 128 == 0, N % 256 == 0, K % 256 == 0.
 */
mx_status nvfp4_gemm_grouped(const void* qa, const void* sa, const float* ga, const void* qb, const void* sb,
                             const float* gb, const int64_t* group_offsets, int64_t groups, int64_t M, int64_t N,
                             int64_t K, void* out, mx_out out_dtype, int64_t ldc, void* stream);

/*
 * nvfp4_gemm_grouped_ex -- nvfp4_gemm_grouped with, when ga_per_group == 1, one global scale of A
 * per group: ga is then a device float[G] and group g's results are scaled by ga[g] * gb[g] (the
 * tokens routed to each expert quantized as a tensor of their own, e.g. by nvfp4_quantize_grouped
 * with the same offsets).  ga_per_group == 0 is nvfp4_gemm_grouped; any other value returns
 * MX_ERR_INVALID_ARG.
 */
mx_status nvfp4_gemm_grouped_ex(const void* qa, const void* sa, const float* ga, int ga_per_group, const void* qb,
                                const void* sb, const float* gb, const int64_t* group_offsets, int64_t groups,
                                int64_t M, int64_t N, int64_t K, void* out, mx_out out_dtype, int64_t ldc,
                                void* stream);

/*
 * fp8_blockwise_gemm_grouped -- the DeepSeek FP8 expert GEMMs of a mixture-of-experts layer in one
 * launch ([DS] sec 5, 6.3; group layout as mx_gemm_grouped): group g computes, for its rows
 * off[g] <= m < off[g+1], C[m][n] = sum_kb sA[kb][m] sB[gN/128 + n/128][kb] P_kb[m][n], with P_kb
 * the exact FP32 sum of qA qB over k-block kb (promotion every 128 of K, as fp8_blockwise_gemm).
 * qa[M][K] E4M3 with sa float[K/128][M] (1x128 tiles); qb[G*N][K] E4M3, the experts' [N][K]
 * weights stacked, with sb float[G*N/128][K/128] (their 128x128 blocks stacked the same way, as
 * one mx_quantize(block=128, block_rows=128) of the stacked weights gives).  group_offsets as
 * mx_gemm_grouped.  M % 128 == 0, N % 256 == 0, K % 128 == 0, 1 <= G <= 1024; out as for mx_gemm.
 */
mx_status fp8_blockwise_gemm_grouped(const void* qa, const float* sa, const void* qb, const float* sb,
                                     const int64_t* group_offsets, int64_t groups, int64_t M, int64_t N, int64_t K,
                                     void* out, mx_out out_dtype, int64_t ldc, void* stream);

/* Bytes of caller-owned device workspace nvfp4_quantize needs (>= 16). */
size_t nvfp4_workspace_bytes(int64_t rows, int64_t cols);

/*
 * nvfp4_quantize -- NVFP4 two-level quantization.  [NV] sec 5.4, 5.6.
 *   pass 1: amax over the whole tensor; s_g = fl32(amax / 2688) (1.0 if amax == 0),
 *           written to *gscale (device float).
 *   pass 2: per 16 consecutive elements along cols: t = fl32(fl32(bamax / 6) / s_g);
 *           c = E4M3 RNE-satfinite(t); s_hat = fl32(dec(c) * s_g);
 *           q = E2M1 RNE-satfinite(fl32(x / s_hat)) (0 when s_hat == 0).
 * x[rows][cols] bf16 (finite); q_packed[rows][cols/2] u8; s_ue4m3: rows*cols/16 bytes in the
 * NVFP4 GEMM layout; workspace: nvfp4_workspace_bytes() bytes, 16-byte aligned, contents
 * need not be initialised (the call clears it on `stream`).  rows % 128 == 0,
 * cols % 64 == 0.
 */
mx_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols,
                         void* q_packed, void* s_ue4m3, float* gscale,
                         void* workspace, void* stream);

/*
 * nvfp4_quantize_grouped -- NVFP4 quantization of G row groups of one bf16 matrix, each group a
 * tensor of its own (the weights or tokens of MoE experts; [NV] sec 5.4 applied per group): group
 * g, rows off[g] <= r < off[g+1], gets its own amax and global scale gscale[g].  The results equal
 * G calls of nvfp4_quantize on the groups' row slices, bit for bit: q_packed and s_ue4m3 hold the
 * codes and scale chunks of the whole [rows][cols] matrix in the NVFP4 GEMM layout, group g's in
 * its own rows (the layout nvfp4_gemm_grouped reads for B, whose gb is this gscale).
 * group_offsets: device int64[G + 1], 0 = off[0] <= off[1] <= ... <= off[G] = rows, all multiples
 * of 128; an empty group gets gscale 1.0.  Offsets that break this contract make the next
 * mx_check() report MX_ERR_INVALID_ARG; the outputs are then unspecified, but no access leaves
 * the caller's buffers.  gscale: device float[G]; workspace: 4 * G bytes (at least 16), 16-byte
 * aligned, cleared by the call on `stream`.  1 <= G <= 1024, rows % 128 == 0, cols % 64 == 0.
 */
mx_status nvfp4_quantize_grouped(const void* x, int64_t rows, int64_t cols, const int64_t* group_offsets,
                                 int64_t groups, void* q_packed, void* s_ue4m3, float* gscale, void* workspace,
                                 void* stream);

/*
 * nvfp4_gemm -- NVFP4 block-scaled GEMM.  [NV] sec 7.3-7.4:
 *   C[m][n] = gA * gB * sum_b sA[m][b] sB[n][b] sum_{i<16} qA qB, FP32 accumulate; the two
 *   global scales (device floats written by nvfp4_quantize) are applied in the epilogue.
 * qa[M][K/2], qb[N][K/2] packed E2M1; sa, sb in the NVFP4 GEMM layout.
 * M % 128 == 0, N % 128 == 0, K % 256 == 0; out as for mx_gemm.
 */
mx_status nvfp4_gemm(const void* qa, const void* sa, const float* ga,
                     const void* qb, const void* sb, const float* gb,
                     int64_t M, int64_t N, int64_t K,
                     void* out, mx_out out_dtype, int64_t ldc, void* stream);

/*
 * fp8_blockwise_gemm -- DeepSeek-style FP8 GEMM with FP32 promotion.  [DS] sec 6.3:
 *   for every 128-wide k-block kb: P = sum_{k in kb} qA[m][k] qB[n][k] (tensor cores, FP32),
 *   acc += sA[kb][m] * sB[n/128][kb] * P in FP32 registers.
 * qa[M][K], qb[N][K] E4M3; sa float[K/128][M] (1x128 tiles, k-block-major);
 * sb float[N/128][K/128] (128x128 blocks).  M % 128 == 0, N % 128 == 0, K % 128 == 0.
 */
mx_status fp8_blockwise_gemm(const void* qa, const float* sa,
                             const void* qb, const float* sb,
                             int64_t M, int64_t N, int64_t K,
                             void* out, mx_out out_dtype, int64_t ldc, void* stream);

/*
 * nvfp4_quantize_noalloc -- the same NVFP4 quantization as nvfp4_quantize, for callers that
 * cannot allocate device memory (for example a plug-in inside a host whose allocator owns all of
 * the GPU's memory, or a launch path that must never call cudaMalloc because it synchronizes the
 * device).  It takes no workspace and allocates nothing: its scratch is a 64 KB array inside
 * libmxgb.so that every GPU which loads the library keeps until the process exits.  The pages
 * have no counterpart to this entry point; it exists only for such callers.
 *
 * Arguments and results are those of nvfp4_quantize (identical codes, scales and gscale).
 * Limit: rows <= 262144 (the array holds one partial maximum per 16 rows); larger inputs return
 * MX_ERR_INVALID_ARG.  The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.  The address is cached
 * per device ordinal, so the library assumes that every call on a device runs in the CUDA
 * runtime's primary context of that device (the context the runtime API and PyTorch use); a
 * caller that makes its own driver-API contexts must not call this entry point from them.  All
 * calls share the one array: calls that overlap on the GPU (different streams, or different host
 * threads, without ordering between them) race and may produce wrong results.  Each call writes every scratch slot
 * it reads before reading it, so nothing left by an earlier call needs clearing.
 */
mx_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols,
                                 void* q_packed, void* s_ue4m3, float* gscale, void* stream);

/* Bytes of the scale tensor mx_quantize / nvfp4_quantize write for a [rows][cols] input:
 * block 32 + E8M0 -> rows*cols/32 (block_rows 1, and 32: 2-D blocks are stored expanded);
 * block 16 + UE4M3 -> rows*cols/16; block 128 + FP32 or FP32_POW2 -> 4*rows*cols/128
 * (block_rows 1) or 4*(rows/128)*(cols/128) (block_rows 128).  0 if the combination is not
 * supported. */
size_t mx_scale_bytes(int64_t rows, int64_t cols, int block, int block_rows, mx_scale_fmt sfmt);

/*
 * mx_check -- synchronizes `stream`, then reads and clears the library's device error word.
 * Returns MX_ERR_TIMEOUT if a kernel's bounded wait ran out since the last check,
 * MX_ERR_INVALID_ARG if the only event was a grouped GEMM whose device offsets broke their
 * contract, MX_ERR_CUDA on a pending CUDA error, MX_OK otherwise.  This is the only call that
 * synchronizes.
 */
mx_status mx_check(void* stream);

/* Number of SMs the GEMM kernels size their persistent grids for (0 before the first call
 * that launches a GEMM on the current device). */
int mx_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* MXGB_MX_H_ */

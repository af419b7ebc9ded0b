/*
 * fp8moe -- FP8 / MXFP8 quantization and scaled grouped GEMM for the
 * Mixture-of-Experts training hot path, for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is a plain device pointer unless marked
 * "host"; sizes are element counts.  The caller owns and allocates every
 * buffer.  The library allocates no device memory: its only device state is
 * one status word in static device memory per device, and TMA descriptors
 * are passed to kernels by value.
 *
 * Streams.  Every call is asynchronous on the given stream (NULL = legacy
 * default stream) and never synchronizes, except fp8moe_get_device_status.
 * No call reads the routing offsets on the host: grouped kernels schedule
 * experts on the device.
 *
 * Errors.  A problem visible on the host (null pointer, bad size, alignment,
 * an unsupported combination) makes the call return an error before any
 * launch and leaves the outputs untouched.  A problem only visible on the
 * device (offsets that decrease, exceed M, do not end at M, or break a
 * multiple-of-32 rule; a pipeline wait that runs out) sets the sticky
 * device status word; the outputs of that launch are then unspecified.
 * Read and clear it with fp8moe_get_device_status.
 *
 * Alignment.  Every data pointer must be 16-byte aligned.
 *
 * Sources (the library follows the behaviour these pages describe):
 *  [AMD-FP8]  "FP8 Training on AMD GPUs with TorchTitan and TorchAO:
 *             Upstreaming Performance Improvements", as summarised by
 *             aitrends.kr (Korean), aihirek.info (Hungarian) and aixai.ru
 *             (Russian).
 *  [SCOUT]    "Accelerating Llama4 Scout training with TorchAO MXFP8 MoE
 *             primitives", as summarised by aitrends.kr (Korean).
 */
#ifndef FP8MOE_H
#define FP8MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* fp8moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  FP8MOE_OK = 0,
  FP8MOE_ERR_INVALID_ARG = 1,     /* null pointer, negative or inconsistent size */
  FP8MOE_ERR_ALIGNMENT = 2,       /* pointer not 16-byte aligned, bad multiple */
  FP8MOE_ERR_UNSUPPORTED = 3,     /* e.g. e4m3fnuz with MXFP8 or with the GEMM */
  FP8MOE_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed */
  FP8MOE_ERR_DEVICE_OFFSETS = 5,  /* device: offsets invalid (read via get_device_status) */
  FP8MOE_ERR_TIMEOUT = 6,         /* device: a bounded pipeline wait ran out */
  FP8MOE_ERR_SCRATCH_LIMIT = 7,   /* host: the problem needs more than the static scratch */
  FP8MOE_ERR_CONCURRENT = 8       /* device: launches in flight at once shared a work counter */
} fp8moe_status;

typedef enum {
  FP8MOE_E4M3FN = 0,   /* max 448, NaN = S.1111.111, signed zero      */
  FP8MOE_E4M3FNUZ = 1  /* max 240, no NaN/Inf values, unsigned zero   */
} fp8moe_fp8_kind;

typedef enum {
  FP8MOE_ROWWISE = 0,   /* fp32 scale per row / per (expert, column)  */
  FP8MOE_MXFP8 = 1,     /* e8m0 scale per 1x32 block, 128x4-tiled     */
  FP8MOE_TENSORWISE = 2, /* one fp32 scale per tensor                 */
  FP8MOE_BLOCKWISE = 3   /* fp32 scale per 1x128 / 128x128 tile        */
} fp8moe_recipe;

enum { FP8MOE_SCALES_ROWMAJOR = -2, FP8MOE_NO_GROUPS = -1, FP8MOE_GROUP_ROWS = 0, FP8MOE_GROUP_COLS = 1 };

/* Largest number of groups (experts) a call with offsets accepts. */
enum { FP8MOE_MAX_GROUPS = 1024 };

/* ------------------------------------------------------------------------
 * Rowwise FP8 quantization.  [AMD-FP8] aihirek.info "A Triton-kernelok
 * csökkentették a kvantálás költségét"; aixai.ru "Три уровня оптимизации
 * Triton-ядер": absmax per row -> scale -> apply -> clamp -> cast, fused in
 * one pass (one read of x, one write of q).
 *
 * x      [R, C] bf16, row stride ldx elements (ldx >= C, ldx % 8 == 0)
 * q      [R, C] fp8 codes of `kind`, dense (row stride C); C % 16 == 0
 * scale_inv [R] fp32: the dequantization scale fl(1/s), where
 *        s = fl(fp8_max / max(amax_row, 1e-12)) and q = enc(fl(x * s))
 *        (round to nearest even, saturating at +-fp8_max).
 * kind   FP8MOE_E4M3FN or FP8MOE_E4M3FNUZ (quantize-only mode; [AMD-FP8]
 *        aixai.ru "Тихая порча градиентов": the wrong maximum silently clips).
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_quantize_rowwise(const void* x, int64_t R, int64_t C, int64_t ldx,
                                      int kind, void* q, float* scale_inv,
                                      fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Colwise FP8 quantization of 3D expert weights or of routed rows.
 * [AMD-FP8] aixai.ru "MoE: почему DeepSeek-V3 ломал пайплайн" (a column
 * scale per expert) and "Три уровня оптимизации" (the backward colwise
 * scales kernel: transposed output written through on-chip staging, single
 * pass, no .t().contiguous() copy).
 *
 * offs == NULL (dense): x is [E, R, C] bf16 contiguous; the absmax runs over
 *   R for every (e, c).  scale_inv is [E, C].  q is [E, C, R] when
 *   transpose_out (R contiguous: the K-major operand of a GEMM contracting
 *   over R), else [E, R, C].
 * offs != NULL (jagged): x is [R, C] bf16 contiguous; offs is a device int32
 *   [E] of cumulative exclusive group ends (group e = rows
 *   [offs[e-1], offs[e]), offs[-1] = 0, offs[E-1] must equal R).  The
 *   absmax runs over each group's rows for every column; an empty group
 *   gets scale_inv = fl(1 / fl(fp8_max / 1e-12)).  q is
 *   [C, fp8moe_jagged_t_cols(R, E)] when transpose_out, with group e in
 *   columns [P_e, P_e + g_e), P_e = sum_{j<e} round_up(g_j, 32), every
 *   other column 0; else [R, C].  1 <= E <= FP8MOE_MAX_GROUPS.
 * C % 16 == 0; dense transposed output also needs R % 16 == 0.
 * Transposed output runs as one pass over x and writes scale_inv directly:
 * dense, in thread-block clusters that exchange column maxima through
 * distributed shared memory; jagged, one CTA per group strip, the CTAs
 * taking strips from a device work counter (one of 16 slots, chosen per
 * launch in turn: 16 or more such launches in flight at once on different
 * streams, or replays of one captured launch running concurrently, can
 * meet in a slot, which sets FP8MOE_ERR_CONCURRENT in the device status and
 * leaves the outputs invalid).  Untransposed output uses
 * scale_inv as the scratch of the column maxima during the call
 * (stream-ordered; it holds the scales when the call's work completes).
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_quantize_colwise_3d(const void* x, int64_t E, int64_t R, int64_t C,
                                         const int32_t* offs, int transpose_out, int kind,
                                         void* q, float* scale_inv, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Tensorwise FP8 quantization: one scale for the whole tensor.  [AMD-FP8]
 * aixai.ru "Скейлы: от тензора до микроблока" (the coarsest of the four
 * granularities; tensorwise, rowwise, blockwise, MXFP8).  Same arithmetic as
 * rowwise with the absolute maximum over every element.
 *
 * x and the output layouts as fp8moe_quantize_colwise_3d: dense [E, R, C]
 * (offs NULL) or routed rows [R, C] with offs [E] over R; transpose_out 0
 * writes q in x's layout, 1 writes [E, C, R] (dense) or the group-padded
 * [C, fp8moe_jagged_t_cols(R, E)] (jagged, E <= FP8MOE_MAX_GROUPS; zero
 * padding), the operand layouts of the rowwise / tensorwise grouped GEMMs.  scale_inv: one fp32
 * (4-byte aligned), the dequantization scale 1/s; it is used as scratch by
 * the call (stream-ordered).  Alignment: x, q 16 bytes; C % 16 == 0 when
 * transposed, (dense) R % 16 == 0 when transposed.  kind: e4m3fn or fnuz.
 * The plain layout runs as one cooperative launch of one CTA per SM: it
 * starts once every SM can take one of its CTAs (work on other streams
 * that occupies SMs delays it), and each CTA holds the SM's whole TMEM.
 * A wait inside it that exceeds 2 s sets FP8MOE_ERR_TIMEOUT in the device
 * status.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_quantize_tensorwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                                         int transpose_out, int kind, void* q, float* scale_inv,
                                         fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Blockwise FP8 quantization: one fp32 scale per tile.  [AMD-FP8] aixai.ru
 * "Скейлы: от тензора до микроблока" (blockwise: a scale per tile of fixed
 * size, between rowwise and MXFP8).  The pages give no tile size; tiles are
 * 1 x 128 along the contracting dimension for activations and gradients,
 * 128 x 128 for expert weights, 128 tokens per group for the operands of
 * wgrad.  Per tile, the rowwise arithmetic: s = fl(fp8_max / max(amax,
 * 1e-12)), q = enc(fl(x * s)) (RNE, saturating), scale_inv = fl(1 / s).
 *
 * _rows:   x [R, C] bf16, C % 128 == 0 -> q [R, C], scale_inv [C/128, R]
 *          (tile-index major: the scales of one tile column are contiguous).
 *          The row operand of forward (A over K) and dgrad (dY over N).
 * _weight: w [E, N, K] bf16, N % 128 == K % 128 == 0 -> q [E, N, K] (forward
 *          operand) and / or qt [E, K, N] (the transposed dgrad operand; the
 *          same codes), scale_inv [E, N/128, K/128] serving both.  Either
 *          output may be NULL.
 * _tokens: x [M, C] bf16 routed rows, offs [E] device (multiples of 32,
 *          offs[E-1] = M), C % 16 == 0 -> qt [C, M] (tokens contiguous: the
 *          wgrad operand) and scale_inv [fp8moe_blockwise_token_blocks(M, E),
 *          C]: row b holds the scales of token block b, the blocks of group
 *          0 first (block j of group e = tokens [start + 128 j, min(end,
 *          start + 128 (j + 1)))); rows past the real block count are not
 *          written.  scale_inv 16-byte aligned.  Invalid offsets set
 *          FP8MOE_ERR_DEVICE_OFFSETS and write nothing.
 * kind: e4m3fn or fnuz (the GEMM takes e4m3fn).
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_quantize_blockwise_rows(const void* x, int64_t R, int64_t C, int kind, void* q,
                                             float* scale_inv, fp8moe_stream_t stream);
fp8moe_status fp8moe_quantize_blockwise_weight(const void* w, int64_t E, int64_t N, int64_t K, int kind, void* q,
                                               void* qt, float* scale_inv, fp8moe_stream_t stream);
int64_t fp8moe_blockwise_token_blocks(int64_t M, int64_t E);
fp8moe_status fp8moe_quantize_blockwise_tokens(const void* x, int64_t M, int64_t C, const int32_t* offs, int64_t E,
                                               int kind, void* qt, float* scale_inv, fp8moe_stream_t stream);

/* Width (columns) of the transposed jagged colwise output: round_up(M + 31*E, 16). */
int64_t fp8moe_jagged_t_cols(int64_t M, int64_t E);

/* ------------------------------------------------------------------------
 * MXFP8 quantization along dim 0 (the contiguous dimension).  [SCOUT] MXFP8
 * layout diagram: e4m3 data, one e8m0 scale per 1x32 block.
 * x [B*R, C] bf16 contiguous (B batches of R rows), C % 32 == 0.
 * q [B*R, C] e4m3fn codes; scale [B*R, C/32] e8m0 bytes, row-major.
 * Scale rule: e = clamp(floor(log2(amax)) - 8, -127, 127), byte = e + 127
 * (amax = 0 gives byte 0); q = enc_e4m3fn(x * 2^-e), RNE, saturating.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_mxfp8_quantize_dim0(const void* x, int64_t B, int64_t R, int64_t C,
                                         void* q, uint8_t* scale, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 quantization along dim 1 with transposed output.  [SCOUT] section
 * details: dynamic quantization in forward and backward, with the layout
 * change along the contracting dimension of the weight gradient.
 * x [B, R, C] bf16 contiguous, R % 32 == 0, C % 16 == 0.
 * qt [B, C, R] e4m3fn codes; scale [B, C, R/32] e8m0 bytes (blocks of 32
 * consecutive rows of one column).  Routed rows whose groups are multiples
 * of 32 need no offsets here: no block straddles two groups.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_mxfp8_quantize_dim1(const void* x, int64_t B, int64_t R, int64_t C,
                                         void* qt, uint8_t* scale, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 quantization along either or both dimensions, with the scales
 * written directly in the layout the grouped GEMM consumes (no separate
 * swizzle pass).  [SCOUT] section details: forward and backward quantize the
 * same tensors (activations, weights, gradients) along the dimension their
 * GEMM contracts over, and the scales go to the 128x4 layout; [AMD-FP8]
 * aixai.ru "Три уровня оптимизации": fewer passes through HBM.  With both
 * directions requested, one launch reads x once and writes both (4 bytes
 * moved per element instead of 6); with one, that direction's own pass.
 *
 * x [B, R, C] bf16 contiguous, R % 32 == 0 (when dim1 is produced), C % 32 == 0.
 * Either direction may be skipped by passing NULL codes.
 *   dim0: q0 [B, R, C] e4m3fn; s0 = scales of [B, R, C/32] in layout s0_layout:
 *         FP8MOE_SCALES_ROWMAJOR (plain [B, R, C/32]), FP8MOE_NO_GROUPS
 *         (128x4 tiles per batch, as fp8moe_swizzle_scales_128x4), or
 *         FP8MOE_GROUP_ROWS (B == 1, offs [E] over R).
 *   dim1: q1 [B, C, R] e4m3fn; s1 = scales of [B, C, R/32] in layout s1_layout:
 *         FP8MOE_SCALES_ROWMAJOR, FP8MOE_NO_GROUPS, or FP8MOE_GROUP_COLS
 *         (B == 1, offs [E] over R, multiples of 32).
 * Codes and the scale bytes of real blocks are bit-identical to
 * fp8moe_mxfp8_quantize_dim0 / dim1 followed by fp8moe_swizzle_scales_128x4;
 * the padding bytes of a swizzled scale buffer are not written (the grouped
 * GEMM never lets them reach a stored output; zero the buffer first if they
 * must be zero).  Invalid device offsets set FP8MOE_ERR_DEVICE_OFFSETS and
 * write nothing.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_mxfp8_quantize_dual(const void* x, int64_t B, int64_t R, int64_t C, const int32_t* offs,
                                         int64_t E, void* q0, uint8_t* s0, int s0_layout, void* q1, uint8_t* s1,
                                         int s1_layout, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * 128x4 tiled scale layout for tcgen05 block-scaled MMA.  [SCOUT] section
 * details and the caption of its 128x4 tile layout table: a dedicated kernel
 * converts row-major scales into 128x4 tiles.
 *
 * Input s: [B, R, Cs] bytes, row-major.  Output: for each batch, the matrix
 * padded to whole tiles, tile (rb, cb) at byte ((rb * CB) + cb) * 512 and
 * element (r, c) of a tile at (r % 32) * 16 + (r / 32) * 4 + c.
 * group_axis:
 *   FP8MOE_NO_GROUPS  plain, B >= 1 batches, offs ignored (may be NULL).
 *   FP8MOE_GROUP_ROWS B == 1; offs [E] (device) splits the R rows; each
 *                     group starts a new 128-row block (forward / dgrad).
 *   FP8MOE_GROUP_COLS B == 1; offs [E] (device) splits the *contracting
 *                     elements* (32 per scale column; boundaries multiples of
 *                     32); each group starts a new 4-column block (wgrad).
 * Every byte of the output (fp8moe_swizzled_scales_bytes) is written: pads
 * and unused tiles are 0.
 * ------------------------------------------------------------------------ */
int64_t fp8moe_swizzled_scales_bytes(int64_t B, int64_t R, int64_t Cs, int64_t E, int group_axis);
fp8moe_status fp8moe_swizzle_scales_128x4(const uint8_t* s, int64_t B, int64_t R, int64_t Cs,
                                          const int32_t* offs, int64_t E, int group_axis,
                                          uint8_t* out, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Scaled grouped GEMM, one launch over all experts, groups from device
 * offsets.  [AMD-FP8] aixai.ru "MoE: почему DeepSeek-V3 ломал пайплайн"
 * (row scales for activations, column scales per expert for weights, an
 * offsets tensor, one launch); [SCOUT] MoE forward diagram (2D input, 3D
 * weights, grouped by offsets); aixai.ru "Что такое FP8-обучение" (three
 * GEMMs per linear layer).  Output bf16, fp32 accumulation on tcgen05
 * tensor cores.  Only e4m3fn operands.
 *
 * forward:  out[m, :] = A[m, :] . W[e]^T  for m in group e
 *   a [M, K] e4m3, w [E, N, K] e4m3, out [M, N] bf16.
 *   MXFP8:   a_scale = fp8moe_swizzle_scales_128x4 of [M, K/32], GROUP_ROWS;
 *            w_scale = swizzle of [E, N, K/32], NO_GROUPS, B = E.
 *   ROWWISE: a_scale fp32 [M]; w_scale fp32 [E, N].
 *   TENSORWISE: a_scale, w_scale one fp32 each (fp8moe_quantize_tensorwise);
 *            operand layouts as ROWWISE in every mode.
 * dgrad:    dA[m, :] = dY[m, :] . Wt[e]^T  (contraction over N)
 *   dy [M, N], wt [E, K, N] (the transposed weight from colwise / dim1
 *   quantization), out [M, K].  Scales as forward with (K <-> N).
 * wgrad:    dW[e] = dYt[:, group e] . At[:, group e]^T (contraction over
 *   the routed tokens of group e; an empty group gives dW[e] = 0)
 *   dyt [N, Mt], at [K, Mt], out [E, N, K].
 *   MXFP8:   Mt = M, offs multiples of 32; scales = swizzle of [N, M/32] and
 *            [K, M/32] with GROUP_COLS.
 *   ROWWISE: Mt = fp8moe_jagged_t_cols(M, E), the group-padded layout of
 *            fp8moe_quantize_colwise_3d; scales fp32 [E, N] and [E, K].
 * BLOCKWISE (N % 128 == K % 128 == 0): operands and scales from
 *   fp8moe_quantize_blockwise_*: forward a = _rows(A) with a_scale
 *   [K/128, M], w = _weight q with w_scale [E, N/128, K/128]; dgrad dy =
 *   _rows(dY) with [N/128, M], wt = _weight qt with the same w_scale; wgrad
 *   (M % 32 == 0, offsets multiples of 32) dyt, at = _tokens(dY), _tokens(A)
 *   with [blocks, N] and [blocks, K] (16-byte aligned).  Each 128-element
 *   k-block's product is scaled by its row and column scales and summed in
 *   fp32.
 * Sizes: M >= 0, N % 16 == 0, K % 32 == 0 (MXFP8) or K % 16 == 0 (rowwise),
 * E >= 1.  MXFP8 offsets must be multiples of 32 (device-checked).
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_scaled_grouped_mm_fwd(int recipe, const void* a, const void* a_scale,
                                           const void* w, const void* w_scale,
                                           const int32_t* offs, int64_t E, int64_t M,
                                           int64_t N, int64_t K, void* out,
                                           fp8moe_stream_t stream);
fp8moe_status fp8moe_scaled_grouped_mm_dgrad(int recipe, const void* dy, const void* dy_scale,
                                             const void* wt, const void* wt_scale,
                                             const int32_t* offs, int64_t E, int64_t M,
                                             int64_t N, int64_t K, void* out,
                                             fp8moe_stream_t stream);
fp8moe_status fp8moe_scaled_grouped_mm_wgrad(int recipe, const void* dyt, const void* dyt_scale,
                                             const void* at, const void* at_scale,
                                             const int32_t* offs, int64_t E, int64_t M,
                                             int64_t N, int64_t K, void* out,
                                             fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 grouped GEMM with the activation quantized in the GEMM's prologue.
 * [SCOUT] section details (the _to_mxfp8_then_scaled_grouped_mm primitive:
 * bf16 activations are quantized to MXFP8 on the fly and fed to the scaled
 * grouped GEMM); [AMD-FP8] aixai.ru "Три уровня оптимизации" (fewer passes
 * through HBM).  Same results as fp8moe_mxfp8_quantize_dim0 of the bf16
 * operand (scales swizzled with GROUP_ROWS) followed by the MXFP8
 * fp8moe_scaled_grouped_mm_fwd / _dgrad, bit for bit: the kernel's
 * producer stages the bf16 A tiles in shared memory and four warps turn each
 * into e4m3 codes and e8m0 scales (the dim0 rule) right where the tensor
 * cores read them, so the fp8 copy of A never goes through HBM.
 *
 * forward: a [M, K] bf16 routed rows (groups from offs, multiples of 32),
 *   w [E, N, K] e4m3 with w_scale as for the MXFP8 forward; out [M, N] bf16.
 * dgrad:   dy [M, N] bf16, wt [E, K, N] e4m3 with wt_scale as for the MXFP8
 *   dgrad; out [M, K] bf16.
 * a_q / a_s (dy_q / dy_s): optional (both NULL or both given) copies of the
 * quantized operand, codes [M, K] ([M, N]) and row-major e8m0 scales
 * [M, K/32] ([M, N/32]), written by the kernel (rows past M are not).
 * The contracting dimension must be a multiple of 32; N % 16 == K % 16 == 0;
 * 1 <= E <= FP8MOE_MAX_GROUPS; every pointer 16-byte aligned.  Device-side
 * offset errors as the MXFP8 grouped GEMM.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_mxfp8_grouped_mm_fwd_quant_a(const void* a, const void* w, const void* w_scale,
                                                  const int32_t* offs, int64_t E, int64_t M, int64_t N, int64_t K,
                                                  void* out, void* a_q, uint8_t* a_s, fp8moe_stream_t stream);
fp8moe_status fp8moe_mxfp8_grouped_mm_dgrad_quant_a(const void* dy, const void* wt, const void* wt_scale,
                                                    const int32_t* offs, int64_t E, int64_t M, int64_t N, int64_t K,
                                                    void* out, void* dy_q, uint8_t* dy_s, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 MoE expert layer as two composites: dynamic MXFP8 quantization of
 * the bf16 operands followed by the scaled grouped GEMMs.  [SCOUT] section
 * details (the _to_mxfp8_then_scaled_grouped_mm primitive quantizes the
 * input activations and the weights to MXFP8 on the fly and then runs the
 * scaled grouped GEMM; dynamic quantization applies in forward and
 * backward, the weight gradient along its contracting dimension);
 * [AMD-FP8] aixai.ru "Три уровня оптимизации" (the backward reads operands
 * already laid out for its GEMMs instead of transposed copies).
 *
 * Forward: A [M, K] bf16 routed rows (groups from offs [E], multiples of
 * 32), W [E, N, K] bf16.  One dual-direction quantization of A and one of W
 * (each reads its tensor once), then out [M, N] bf16 = the grouped GEMM
 * forward.  The dim1 codes and scales of A and of W (the operands of wgrad
 * and dgrad) are kept in the workspace for the backward.
 * Backward: dY [M, N] bf16 -> one dual-direction quantization, then
 * dA [M, K] = dgrad(dY, W^T saved) and dW [E, N, K] = wgrad(dY^T, A^T
 * saved); either output may be NULL to skip its GEMM.
 * Results are bit-identical to the same chain of fp8moe_mxfp8_quantize_dual
 * and fp8moe_scaled_grouped_mm_* calls.
 * workspace: caller-owned device memory of fp8moe_mxfp8_moe_workspace_bytes
 * (16-byte aligned), passed unchanged from the forward to the backward on
 * the same stream (or after it completes); the backward overwrites the
 * forward-only part of it.  Sizes: M, N, K multiples of 32, 1 <= E <=
 * FP8MOE_MAX_GROUPS.  Device-side offset errors as the calls it chains.
 * ------------------------------------------------------------------------ */
int64_t fp8moe_mxfp8_moe_workspace_bytes(int64_t E, int64_t M, int64_t N, int64_t K);
fp8moe_status fp8moe_mxfp8_moe_fwd(const void* a, const void* w, const int32_t* offs, int64_t E, int64_t M,
                                   int64_t N, int64_t K, void* out, void* workspace, int64_t workspace_bytes,
                                   fp8moe_stream_t stream);
fp8moe_status fp8moe_mxfp8_moe_bwd(const void* dy, const int32_t* offs, int64_t E, int64_t M, int64_t N,
                                   int64_t K, void* workspace, int64_t workspace_bytes, void* da, void* dw,
                                   fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Token routing into expert groups and back.  [AMD-FP8] aixai.ru "MoE:
 * почему DeepSeek-V3 ломал пайплайн" (tokens are routed to their experts by
 * an offsets tensor before the fused quantization and the one-launch grouped
 * GEMM); the MoE layer configurations pad every group to a multiple of 32
 * rows.
 *
 * fp8moe_route_permute: x [T, H] bf16, topk_idx [T, k] int32 expert ids in
 * [0, E).  Writes a [fp8moe_route_rows(T, k, E), H] bf16: group e holds the
 * (t, j) pairs with topk_idx[t, j] == e in increasing (t, j) order starting
 * at a 32-aligned row, followed by zero rows up to the next multiple of 32;
 * the last group also takes the remaining rows (all zero).  offs [E] int32:
 * the cumulative ends (multiples of 32, offs[E-1] = the row count), the
 * offsets of the grouped GEMMs and of the grouped MXFP8 scale layouts.
 * row_of [T, k] int32: the row of each (t, j).  topk_w [T, k] fp32 or NULL:
 * when given, the copied rows are bf16(w * x) (the backward of a weighted
 * combine).  Ids outside [0, E) set FP8MOE_ERR_DEVICE_OFFSETS; their rows are
 * not written (row_of = -1).  workspace: caller-owned device memory of
 * fp8moe_route_workspace_bytes(T, k, E) bytes.  Alignment: x, a 16 bytes,
 * H % 8 == 0; 1 <= E <= 1024.
 *
 * fp8moe_route_unpermute: y [rows, N] bf16 (a grouped GEMM output), row_of as
 * above -> out [T, N] bf16 with out[t] = sum over j (in order, fp32) of
 * w[t, j] * y[row_of[t, j]] (w = 1 when topk_w is NULL: the backward of
 * permute).  Alignment: y, out 16 bytes, N % 8 == 0.
 * ------------------------------------------------------------------------ */
int64_t fp8moe_route_rows(int64_t T, int64_t k, int64_t E);
int64_t fp8moe_route_workspace_bytes(int64_t T, int64_t k, int64_t E);
fp8moe_status fp8moe_route_permute(const void* x, int64_t T, int64_t H, const int32_t* topk_idx,
                                   const float* topk_w, int64_t k, int64_t E, void* a, int32_t* offs,
                                   int32_t* row_of, void* workspace, int64_t workspace_bytes,
                                   fp8moe_stream_t stream);
fp8moe_status fp8moe_route_unpermute(const void* y, int64_t T, int64_t N, const int32_t* row_of,
                                     const float* topk_w, int64_t k, void* out, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8moe_route_permute without a caller workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory when they route, such as a runtime whose device memory is
 * planned up front into a fixed arena with no room set aside for the
 * routing scratch, or code on a path where a cudaMalloc is not allowed
 * (it can synchronize the device and can fail under memory pressure).
 *
 * Arguments, results, layouts and errors as fp8moe_route_permute, minus the
 * workspace: the call uses the library's own scratch, a static device array
 * of FP8MOE_ROUTE_STATIC_SCRATCH_BYTES (1 MiB) that every device loading
 * the library holds until the process exits.  A problem whose scratch,
 * fp8moe_route_workspace_bytes(T, k, E), exceeds it is rejected on the host
 * with FP8MOE_ERR_SCRATCH_LIMIT before any launch (for E = 256 experts, up
 * to about a million (token, slot) pairs fit).  The call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call on a device shares the one array and leaves its
 * contents behind; each call writes every scratch word it reads before
 * reading it, so nothing needs to start at zero.  Calls whose work overlaps
 * on the GPU (two streams, or two host threads) race on the array: order
 * them on one stream, or synchronize between them.
 * ------------------------------------------------------------------------ */
enum { FP8MOE_ROUTE_STATIC_SCRATCH_BYTES = 1 << 20 };
fp8moe_status fp8moe_route_permute_noalloc(const void* x, int64_t T, int64_t H, const int32_t* topk_idx,
                                           const float* topk_w, int64_t k, int64_t E, void* a, int32_t* offs,
                                           int32_t* row_of, fp8moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Device status.  After the work already queued on `stream`, takes the
 * sticky device error code of the current device (an fp8moe_status value, 0
 * if none) and clears it in one atomic exchange on the device, then
 * synchronizes `stream` and returns the code in *out_code.  An error that a
 * kernel on another stream sets meanwhile is never lost: it is either taken
 * by this call or left for the next one.  The pages' failure mode is silent
 * ([AMD-FP8] aixai.ru "Тихая порча градиентов"); this makes device-side
 * problems visible instead.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_get_device_status(fp8moe_stream_t stream, int32_t* out_code);

/* ------------------------------------------------------------------------
 * Testing hook of the failure-detection path (no counterpart on the pages).
 * Arms a one-shot flag: the next fp8moe_scaled_grouped_mm_* launch of the
 * process (MXFP8, rowwise or tensorwise recipe) has its first pair of CTAs
 * keep its first accumulator, so the epilogue's bounded wait (2 s) runs out
 * and the launch sets FP8MOE_ERR_TIMEOUT.  Every CTA still waits for its own
 * copies and MMAs before it releases its tensor memory, so the context stays
 * usable.  No environment variable and no other call can stall a launch.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_testing_stall_next_gemm(void);

/* ------------------------------------------------------------------------
 * Testing hook of the failure-detection path of fp8moe_quantize_tensorwise
 * (no counterpart on the pages).  Arms a one-shot flag: the next plain-
 * layout tensorwise launch of the process (the one-launch kernel) has its
 * first CTA skip counting itself in at the grid-wide meeting, so every
 * CTA's bounded wait (2 s) runs out and the launch sets FP8MOE_ERR_TIMEOUT
 * (its codes and scale are then not valid).  Every CTA still waits for its
 * own copies and releases its tensor memory, so the context stays usable.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_testing_stall_next_tensorwise(void);

/* ------------------------------------------------------------------------
 * Testing hook of the failure-detection path of the warp-specialised
 * quantizers (no counterpart on the pages): fp8moe_mxfp8_quantize_dual with
 * both directions and at least 128 columns, and fp8moe_quantize_colwise_3d of
 * routed rows with transposed output.  Arms a one-shot flag: the next such
 * launch of the process never loads one tile (the dual quantizer: the first
 * CTA's first tile; the routed-rows colwise kernel: the first tile of its
 * first unit, whichever CTA takes it), so the consumer warps waiting for it
 * run out of their bounded wait (2 s) and the launch sets
 * FP8MOE_ERR_TIMEOUT (its outputs are then not valid).  The CTA's producer
 * still waits (bounded) for the loads it issued, so no copy is in flight when
 * it exits and the context stays usable.
 * ------------------------------------------------------------------------ */
fp8moe_status fp8moe_testing_stall_next_quant_ring(void);

/* Static string for a status code. */
const char* fp8moe_status_string(int status);

/* Library version, (major << 16) | minor. */
int fp8moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8MOE_H */

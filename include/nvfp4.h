/*
 * nvfp4.h -- C ABI of the NVFP4 linear-layer library for one GB300 (sm_103a).
 *
 * The library quantizes bf16 tensors to NVFP4 and multiplies NVFP4 operands
 * on the tcgen05 tensor cores.  Sources (page title, section):
 *  [FS]  "Full-Stack FP4" (academ.us 2607.04422): Sec. 2 Preliminaries (NVFP4
 *        format x^ = x_E2M1 * s * s_g, blocks of 1x16 or 16x16, the three
 *        linear GEMMs); Sec. 3.2 Eq. (1)-(2) (Q_1x16, Q_16x1, Q_16x16 operands
 *        of Fprop/Dgrad/Wgrad, H16^r random Hadamard on the Wgrad inputs);
 *        Appendix 7 (E2M1 bins, RTN and SR).
 *  [NV]  "Pretraining Large Language Models with NVFP4" (paperlayer
 *        2509.25149v2): Sec. 2 NVFP4 Format (block amax -> FP4 max, E4M3
 *        block scale, FP32 tensor scale); Sec. 4 Training Methodology (RNE for
 *        weights and activations, SR on gradients, RHT on Wgrad inputs, 2D
 *        weight scaling, FP4 GEMMs with BF16/FP32 outputs); B.4 (RHT scale
 *        computed in the rotated space, H H^T = I).
 *  [OT]  "OptiTrain-FP4" README (github mirror): E2M1 code table, Sylvester
 *        Hadamard recursion, 1/sqrt(N) normalisation.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE memory owned by the caller.  The library
 *    allocates no memory and keeps no state between calls except one device
 *    status word (see nvfp4_device_error).  It is safe to call from several
 *    host threads.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Arguments are validated on the host before any
 *    launch; an error return means nothing was enqueued, except
 *    NVFP4_ERR_CUDA, which reports a failed launch.  No C++ exception crosses
 *    the ABI.
 *  - bf16 inputs are row-major with a leading dimension in elements.  Inputs
 *    must be finite; NaN or Inf inputs give unspecified codes.
 *  - Numbers are bit-exact with the documented arithmetic (below); the
 *    repository's CPU oracle implements the same arithmetic independently.
 *
 * Encoded operand (nvfp4_tensor)
 *  A logical matrix [rows][cols] whose cols run along the GEMM reduction
 *  dimension, stored as:
 *   codes  : [rows][ld_codes] bytes; element (r, c) is the 4-bit E2M1 code in
 *            byte codes[r*ld_codes + c/2], low nibble for even c.  Code bits:
 *            sign (bit 3), exponent (bits 2:1, bias 1), mantissa (bit 0);
 *            magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 for codes 0..7 [OT].
 *   scales : one E4M3 (bias 7, max 448) block scale per 16 consecutive
 *            elements of a row, in the tensor-core tile layout.  With
 *            j = c / 16 and S4 = ceil(cols / 64):
 *              offset(r, j) = ((r / 128) * S4 + j / 4) * 512
 *                             + (r % 32) * 16 + ((r / 32) % 4) * 4 + j % 4
 *            in a buffer of nvfp4_scale_bytes(rows, cols) bytes.  Padding
 *            bytes (rows >= `rows` or j >= cols/16) are written as 0 by the
 *            quantizer.  With 16x16 scaling the tile scale is repeated on each
 *            of the tile's 16 rows.
 *   amax   : 1 float, the tensor amax the scale was derived from (may be NULL).
 *   global_scale : 1 float, the decode scale s_g; never leaves the device.
 *  Decoding: x^(r, c) = e2m1(code) * e4m3(scale) * s_g [FS Sec. 2].
 *
 * Quantizer arithmetic (binary32, round-to-nearest-even, no fused ops)
 *  1. amax_t = max |t| over the tensor, t = x, or t = U x per 16-block along
 *     the emitted orientation's reduction dimension when the RHT is on
 *     [NV B.4: the scale is computed in the rotated space].
 *  2. S_enc = 2688 / amax_t (448 * 6: the tensor amax maps onto the largest
 *     E4M3 scale times the largest E2M1 value) [NV Sec. 2]; S_enc = 1 when
 *     amax_t = 0, FLT_MAX on overflow; s_g = 1 / S_enc.
 *  3. per block: s_b = E4M3_rne_satfinite((amax_b / 6) * S_enc) [NV Sec. 2:
 *     the block amax maps onto the FP4 maximum 6]; amax_b is over the 1x16
 *     block or the 16x16 tile of x.
 *  4. r_b = S_enc / s_b (0 if s_b = 0); v = t * r_b.  When r_b overflows to
 *     +inf (S_enc saturated near FLT_MAX and s_b < 1: tensor amaxes below
 *     about 4e-33), v = (t * S_enc) / s_b instead, each operation rounded
 *     once, so that zeros stay signed zeros [FS Sec. 2: the encode divides
 *     by s_b * s_g].
 *  5. RNE: nearest E2M1 value, ties to the even mantissa, |v| > 6 -> 6 [NV
 *     Sec. 4].  SR [FS App. 7]: round |v| up from grid point c_k to c_k+1 iff
 *     (float)r < ((|v| - c_k) / step_k) * 2^16, r 16 random bits (so
 *     P(up) = ceil(frac * 2^16) / 2^16); |v| >= 6 -> 6.  The code's sign bit is
 *     the sign bit of v.
 *  6. Random bits of element idx: Philox4x32-10 (Salmon et al., SC'11) block
 *     with key = (seed lo32, seed hi32), counter = (g lo32, g hi32,
 *     stream_id lo32, stream_id hi32), g = idx / 8; the element takes word
 *     (idx / 2) % 4, low 16 bits for even idx, high 16 bits for odd idx.
 *     idx = r * cols + c in the emitted logical matrix (for 16x16 scaling: the
 *     row-wise index of x, so that both orientations share one draw per
 *     element).
 *  7. RHT [FS Eq. (2), NV Sec. 4, OT]: U = H16 * D / 4, D = diag(-1 where bit
 *     i of rht_sign_mask is set); computed as: negate per D, butterfly stages
 *     s = 0, 1, 2, 3 mapping (t[i], t[i ^ 2^s]) (i without bit s) to
 *     (t[i] + t[i ^ 2^s], t[i] - t[i ^ 2^s]), then multiply by 0.25.
 *
 * Orientations
 *  ROWWISE emits the logical matrix x [rows][cols]; COLWISE emits x^T
 *  [cols][rows], i.e. 1x16 blocks run down 16 consecutive rows of x (Q_16x1
 *  of [FS Eq. (2)]).  For the three GEMMs of a linear layer Y = X W^T:
 *   Fprop  Y  = X  W^T   : A = X rowwise,  B = W rowwise
 *   Dgrad  dX = dY W     : A = dY rowwise, B = W colwise (16x16: same codes)
 *   Wgrad  dW = dY^T X   : A = dY colwise, B = X colwise (RHT on both, same D)
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nvfp4_stream_t;   /* a cudaStream_t */

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,   /* NULL pointer, bad enum, inconsistent tensor */
    NVFP4_ERR_SHAPE = 2,         /* a dimension breaks the format (cols % 16 ...) */
    NVFP4_ERR_ALIGNMENT = 3,     /* a pointer or leading dimension is misaligned */
    NVFP4_ERR_UNSUPPORTED = 4,   /* valid but not implemented (e.g. 2D + RHT) */
    NVFP4_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    NVFP4_ERR_TIMEOUT = 6,       /* a kernel gave up on a bounded wait */
    NVFP4_ERR_WORKSPACE = 7      /* workspace missing or too small */
} nvfp4_status;

/* Block scaling.  NVFP4_SCALE_1X16_46 is 1x16 blocks with 4/6 adaptive
 * scaling [FS related work: 4/6 scaling, MSE-optimal adaptive block scales;
 * the rule is not printed there]: each block is encoded with its amax mapped
 * to 6 (the plain 1x16 scale) and with its amax mapped to 4 (scale
 * E4M3(RN(amax_b / 4) * S_enc)), both with RNE, and keeps the candidate with
 * the smaller sum_i (x_i * S_enc - e2m1(q_i) * s)^2 (binary32, index order,
 * fused multiply-adds; the 6 candidate on a tie); with SR the chosen scale is
 * then used for the stochastic encode.  The output format is unchanged. */
typedef enum { NVFP4_SCALE_1X16 = 0, NVFP4_SCALE_16X16 = 1, NVFP4_SCALE_1X16_46 = 2 } nvfp4_scaling;
typedef enum { NVFP4_ROUND_RNE = 0, NVFP4_ROUND_SR = 1 } nvfp4_rounding;
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_FP32 = 1 } nvfp4_dtype;
enum { NVFP4_ROWWISE = 1, NVFP4_COLWISE = 2 };   /* bit mask of orientations to emit */

typedef struct {
    uint8_t *codes;          /* device, [rows][ld_codes] bytes */
    uint8_t *scales;         /* device, nvfp4_scale_bytes(rows, cols) bytes, tile layout */
    float   *amax;           /* device, 1 float, or NULL */
    float   *global_scale;   /* device, 1 float: s_g */
    int64_t  rows;           /* logical rows */
    int64_t  cols;           /* logical columns = reduction dimension */
    int64_t  ld_codes;       /* bytes between rows of codes */
} nvfp4_tensor;

/* Bytes of the scale buffer of a [rows][cols] operand (tile layout above). */
NVFP4_API size_t nvfp4_scale_bytes(int64_t rows, int64_t cols);

/* Bytes of device workspace nvfp4_quantize / nvfp4_rht_quantize need. */
NVFP4_API size_t nvfp4_quantize_workspace_size(int64_t rows, int64_t cols, int orientations);

/*
 * nvfp4_quantize -- quantize x (bf16, [rows][ld_x], row-major) to NVFP4
 * without the Hadamard transform [FS Sec. 2; NV Sec. 2, Sec. 4].
 *  scaling      1x16 blocks (activations, gradients), 1x16 blocks with 4/6
 *               adaptive scales, or 16x16 tiles (weights).
 *  rounding     RNE (weights, activations) or SR (gradients).
 *  seed, stream_id  select the Philox stream of SR (ignored for RNE); use a
 *               different stream_id for each quantization of one tensor.
 *  orientations NVFP4_ROWWISE and/or NVFP4_COLWISE.
 *  out_row      ROWWISE output: rows = rows, cols = cols (NULL if not emitted).
 *  out_col      COLWISE output: rows = cols, cols = rows (NULL if not emitted).
 *  workspace    device scratch of nvfp4_quantize_workspace_size() bytes,
 *               16-byte aligned; used only during this call's kernels.
 * Requirements (else the status in brackets):
 *  cols % 16 == 0 [SHAPE]; COLWISE or 16x16: rows % 16 == 0 [SHAPE];
 *  x 16-byte aligned, ld_x % 8 == 0, ld_x >= cols [ALIGNMENT / SHAPE];
 *  codes 16-byte aligned, ld_codes % 16 == 0, ld_codes >= cols/2 of the
 *  emitted orientation [ALIGNMENT / SHAPE]; scales 16-byte aligned; at most
 *  2^32 - 1 blocks of 16 per orientation [UNSUPPORTED].
 * Both orientations of one call share the tensor amax (no RHT) and write it
 * to both tensors.
 */
NVFP4_API nvfp4_status nvfp4_quantize(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                            nvfp4_scaling scaling, nvfp4_rounding rounding,
                            uint64_t seed, uint64_t stream_id, int orientations,
                            const nvfp4_tensor *out_row, const nvfp4_tensor *out_col,
                            void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_rht_quantize -- as nvfp4_quantize, with the 16-point random Hadamard
 * transform U = H16 * D / 4 applied along the reduction dimension of each
 * emitted orientation before scaling [FS Eq. (2); NV Sec. 4, B.4].  Each
 * orientation gets its own amax and s_g, both taken in the rotated space.
 * Pass the same rht_sign_mask for the two operands of one Wgrad GEMM: U^T U = I
 * cancels in the product.  16x16 scaling with the RHT is NVFP4_ERR_UNSUPPORTED
 * (the pages apply the RHT to the 1x16-scaled Wgrad inputs only).
 */
NVFP4_API nvfp4_status nvfp4_rht_quantize(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                nvfp4_scaling scaling, nvfp4_rounding rounding,
                                uint64_t seed, uint64_t stream_id, int orientations,
                                const nvfp4_tensor *out_row, const nvfp4_tensor *out_col,
                                uint16_t rht_sign_mask,
                                void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_requantize_col_rht -- Wgrad's second operand re-quantized from the
 * forward pass's quantized input [FS Sec. 3.2 Eq. (2): Q_16x1(H16^T Q_1x16(X))],
 * so that Wgrad uses the same quantized activations as Fprop.  in_row is a
 * ROWWISE 1x16 operand ([rows][cols], e.g. from nvfp4_quantize); each value
 * is dequantized to binary32 as RN(RN(e2m1 * s_b) * s_g), the 16-point RHT
 * U = H16 * D / 4 is applied along the rows (16 consecutive rows of a
 * column), and the result is quantized col-wise with 1x16 blocks along the
 * rows into out_col ([cols][rows], K-major along rows) with its own tensor
 * amax and s_g, RNE or SR as for nvfp4_rht_quantize (stream_id selects the
 * Philox stream).  Two kernels: an amax pass and an encode pass over the FP4
 * input (0.5625 B read per element each).
 * Requirements: rows % 16 == 0 and cols % 16 == 0 [SHAPE]; in_row and
 * out_col as for nvfp4_quantize's outputs and not sharing codes, scales or
 * s_g [INVALID_ARG]; workspace of nvfp4_quantize_workspace_size() bytes.
 */
NVFP4_API nvfp4_status nvfp4_requantize_col_rht(const nvfp4_tensor *in_row, nvfp4_rounding rounding,
                                                uint64_t seed, uint64_t stream_id, uint16_t rht_sign_mask,
                                                const nvfp4_tensor *out_col, void *workspace,
                                                size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_row_col_rht -- the two operands a linear layer takes from one
 * activation or output gradient x [FS Sec. 2, Eq. (1)-(2); NV Sec. 4: the RHT
 * goes to the Wgrad inputs only]: the ROWWISE 1x16 operand without the
 * transform (Fprop / Dgrad) and the COLWISE 1x16 operand with the RHT along
 * the rows of x (Wgrad).  Both outputs are required.  The results are
 * bit-identical to
 *   nvfp4_quantize(x, ..., NVFP4_SCALE_1X16, rounding, seed, stream_row,
 *                  NVFP4_ROWWISE, out_row, NULL, ...)
 *   nvfp4_rht_quantize(x, ..., NVFP4_SCALE_1X16, rounding, seed, stream_col,
 *                      NVFP4_COLWISE, NULL, out_col, rht_sign_mask, ...)
 * but one amax pass and one encode pass over x serve both (two reads of x
 * instead of four).
 * Requirements, workspace and errors as nvfp4_quantize with both
 * orientations (rows % 16 == 0, cols % 16 == 0).
 */
NVFP4_API nvfp4_status nvfp4_quantize_row_col_rht(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                nvfp4_rounding rounding, uint64_t seed,
                                uint64_t stream_row, uint64_t stream_col,
                                uint16_t rht_sign_mask,
                                const nvfp4_tensor *out_row, const nvfp4_tensor *out_col,
                                void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_gemm -- D = A * B^T with NVFP4 operands and FP32 accumulation
 * [FS Sec. 2; NV Sec. 4: FP4 inputs, BF16 or FP32 outputs]:
 *   D[m][n] = s_gA * s_gB * sum_k e2m1(a_mk) s_A(m, k/16) e2m1(b_nk) s_B(n, k/16)
 *  A            [M][K] operand (A->rows = M, A->cols = K).
 *  B            [N][K] operand (B->rows = N, B->cols = K).
 *  D            device, row-major [M][ldd] of out_dtype (bf16 or fp32).
 *  workspace    unused by the current kernels; may be NULL.
 * Requirements: K % 16 == 0 [SHAPE]; ldd >= N [SHAPE]; codes and scales
 * 16-byte aligned, ld_codes % 16 == 0, D aligned to its element size
 * [ALIGNMENT].  Rows of D that start on a 16-byte boundary are written with
 * vector stores.  Only the N columns of each row are written: the padding
 * after them (up to ldd) keeps its contents.  M = 0 or N = 0 enqueues
 * nothing; K = 0 writes D = 0.
 * The kernel's pipeline waits are bounded; a wait that runs out records a
 * timeout which nvfp4_device_error() reports.
 */
NVFP4_API nvfp4_status nvfp4_gemm(const nvfp4_tensor *A, const nvfp4_tensor *B, void *D, int64_t ldd,
                        nvfp4_dtype out_dtype, void *workspace, size_t workspace_bytes,
                        nvfp4_stream_t stream);

/*
 * nvfp4_gemm_amax -- nvfp4_gemm with BF16 output that also takes, in its
 * epilogue, the two tensor amaxes the quantization of D needs [FS App. 9:
 * quantization fused with the operation that produces its input]:
 *  amax_out[0]  max |D| over the BF16 outputs (the row-wise operand's amax);
 *  amax_out[1]  max |U d| over the 16-row blocks d of each column of D, with
 *               U = H16 * diag(rht_sign_mask) / 4 (the col-wise RHT operand's
 *               amax), in the rounding order of nvfp4_quantize_row_col_rht.
 * amax_out is device memory (2 floats, 4-byte aligned), overwritten.  Feed it
 * to nvfp4_quantize_row_col_rht_amax with the same mask: the result equals
 * nvfp4_quantize_row_col_rht of D without its amax pass.
 * Requirements as nvfp4_gemm plus: M % 16 == 0 [SHAPE]; D 16-byte aligned
 * and ldd % 8 == 0 [ALIGNMENT].
 */
NVFP4_API nvfp4_status nvfp4_gemm_amax(const nvfp4_tensor *A, const nvfp4_tensor *B, void *D, int64_t ldd,
                                       float *amax_out, uint16_t rht_sign_mask, void *workspace,
                                       size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_row_col_rht_amax -- nvfp4_quantize_row_col_rht with the two
 * tensor amaxes given (amax_in[0] plain, amax_in[1] rotated; device memory,
 * e.g. from nvfp4_gemm_amax): one encode pass over x, no amax pass, no
 * workspace.  Codes and scales are bit-identical to nvfp4_quantize_row_col_rht
 * when amax_in holds the true maxima.
 */
NVFP4_API nvfp4_status nvfp4_quantize_row_col_rht_amax(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                                       nvfp4_rounding rounding, uint64_t seed, uint64_t stream_row,
                                                       uint64_t stream_col, uint16_t rht_sign_mask,
                                                       const float *amax_in, const nvfp4_tensor *out_row,
                                                       const nvfp4_tensor *out_col, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_lora -- nvfp4_gemm plus the BF16 low-rank branch of a LoRA-SVD
 * linear projection [FS Sec. 3.2 Eq. (1): Y = Q(X) Q(W_res)^T + beta (X L1^T) L2^T,
 * dX = Q(dY) Q(W_res) + beta (dY L2) L1; fused into the GEMM as FS App. 9
 * discusses]:
 *   D = s_gA * s_gB * (A B^T) + beta * U V^T
 *  U            device, BF16 [M][ldu] row-major, r columns (e.g. X L1^T).
 *  V            device, BF16 [N][ldv] row-major, r columns (e.g. L2).
 *  r            the rank, a multiple of 64 up to 4096 [UNSUPPORTED otherwise].
 *  beta         finite FP32 scalar.
 *  workspace    device scratch of nvfp4_gemm_lora_workspace_size(M, r) bytes,
 *               16-byte aligned: holds U * beta / (s_gA s_gB) in BF16.
 * The low-rank product runs on the tensor cores (BF16 MMAs into the same FP32
 * accumulator, after the tile's FP4 MMAs), so U is rounded once more to BF16
 * after scaling (relative error 2^-9 on that term).  K = 0 is UNSUPPORTED.
 * Other requirements and errors as nvfp4_gemm; U and V 16-byte aligned,
 * ldu, ldv multiples of 8 and >= r [ALIGNMENT / SHAPE].
 */
NVFP4_API size_t nvfp4_gemm_lora_workspace_size(int64_t M, int64_t r);
NVFP4_API nvfp4_status nvfp4_gemm_lora(const nvfp4_tensor *A, const nvfp4_tensor *B, void *D, int64_t ldd,
                                       nvfp4_dtype out_dtype, const void *U, int64_t ldu, const void *V,
                                       int64_t ldv, int64_t r, float beta, void *workspace,
                                       size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_axpby -- the NVFP4 GEMM plus a scaled C term, as the Newton-
 * Schulz iteration of the Root optimizer combines its products [FS Sec. 3.4:
 * B_k = b A_k + c qA_k qA_k^16x1, X_k+1 = a X_k + qB_k qX_k^16x1]:
 *   D = alpha * (s_gA * s_gB * A B^T) + beta * C
 * per element in binary32: RN(acc * RN(RN(s_gA * s_gB) * alpha)) + RN(beta * c),
 * then one rounding to out_dtype.
 *  C            device, row-major [M][ldc] of out_dtype; read only when
 *               beta != 0 (may be NULL then).  C may be D itself (same
 *               leading dimension): every element is read before it is
 *               written; any other overlap is undefined.
 *  alpha, beta  finite FP32 scalars [INVALID_ARG].
 * Requirements and errors as nvfp4_gemm, plus ldc >= N [SHAPE] and C aligned
 * to its element size [ALIGNMENT]; K = 0 is UNSUPPORTED.
 */
NVFP4_API nvfp4_status nvfp4_gemm_axpby(const nvfp4_tensor *A, const nvfp4_tensor *B, void *D, int64_t ldd,
                                        nvfp4_dtype out_dtype, float alpha, const void *C, int64_t ldc,
                                        float beta, void *workspace, size_t workspace_bytes,
                                        nvfp4_stream_t stream);

/*
 * nvfp4_newton_schulz_step -- one NVFP4 Newton-Schulz iteration of the Root
 * (Muon) optimizer, with every matrix product an NVFP4 GEMM [FS Sec. 3.4, the
 * quantized NS iteration]:
 *   qX = Q_1x16(X H),  A = qX qX^T
 *   qA = Q_1x16(A H),  qA' = Q_16x1(H^T A),  B = b A + c qA qA'
 *   qB = Q_1x16(B H),  qX' = Q_16x1(H^T X),  X_out = a X + qB qX'
 * Every quantization is RNE with 4/6 adaptive block scales
 * (NVFP4_SCALE_1X16_46) and the RHT H = H16 * D / 4 with D from rht_sign_mask
 * along the product's reduction dimension (one mask for the whole step, so
 * H H^T = I cancels in each product).  A and B are BF16 [m][m]; X and X_out
 * are BF16 [m][n] row-major (ldx, ld_out in elements).  The page's
 * shape-optimised (a, b, c) are not printed: the caller passes them.
 *  workspace    device scratch of nvfp4_newton_schulz_workspace_size(m, n)
 *               bytes, 16-byte aligned.  After the call it begins with A
 *               (bf16, row stride m) and, at byte offset 256 * ceil(2 m^2 /
 *               256), B; the rest (the five quantized operands) is internal.
 * Work on `stream`: three quantize calls and three GEMMs.  X_out may be X
 * itself (same leading dimension).
 * Requirements: m % 16 == 0, n % 16 == 0, m, n > 0 [SHAPE]; X and X_out
 * 16-byte aligned with leading dimensions multiples of 8 and >= n
 * [ALIGNMENT / SHAPE]; finite a, b, c [INVALID_ARG].
 */
NVFP4_API size_t nvfp4_newton_schulz_workspace_size(int64_t m, int64_t n);
NVFP4_API nvfp4_status nvfp4_newton_schulz_step(const void *X, int64_t m, int64_t n, int64_t ldx, float a,
                                                float b, float c, uint16_t rht_sign_mask, void *X_out,
                                                int64_t ld_out, void *workspace, size_t workspace_bytes,
                                                nvfp4_stream_t stream);

/*
 * nvfp4_dequantize -- y = e2m1(code) * s_b * s_g for every element of q
 * [FS Sec. 2], rounded once (nearest even) to out_dtype; y is row-major
 * [q->rows][ldy].  Requirements: y 16-byte aligned, ldy * sizeof(out) % 16 == 0.
 */
NVFP4_API nvfp4_status nvfp4_dequantize(const nvfp4_tensor *q, void *y, int64_t ldy,
                              nvfp4_dtype out_dtype, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_noalloc -- nvfp4_quantize for callers that cannot provide
 * device scratch memory (no counterpart on the pages: this is an interface
 * convenience of this library).  Some callers cannot allocate or be handed a
 * workspace: a plugin whose host runtime owns all device memory and passes it
 * only inputs and outputs, or code that must not call cudaMalloc once it is
 * running (allocation can synchronize the device or fail under memory
 * pressure).  This entry point allocates nothing: it uses a 32 KiB scratch
 * array compiled into the library (held on every GPU that loads the library
 * until the process exits) and otherwise behaves exactly like nvfp4_quantize
 * with the same arguments, workspace aside.
 *  - The first call on a device looks up the scratch's device address (one
 *    cudaGetSymbolAddress with that device current); make that first call
 *    before any stream capture on the device.  The address is cached per
 *    device and CUDA context: after a device reset (or a primary context
 *    released and created again) the next call looks it up again, so make
 *    that call outside a capture as well.
 *  - Every call shares the one scratch array and it keeps the previous call's
 *    contents (each call writes the amax partials it reads, so nothing needs
 *    clearing).  Calls that overlap on the GPU -- on different streams, or
 *    from several host threads -- race on it: serialize them.
 *  - A shape whose workspace would exceed the 32 KiB scratch returns
 *    NVFP4_ERR_WORKSPACE; every shape nvfp4_quantize accepts fits today.
 */
NVFP4_API nvfp4_status nvfp4_quantize_noalloc(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                              nvfp4_scaling scaling, nvfp4_rounding rounding,
                                              uint64_t seed, uint64_t stream_id, int orientations,
                                              const nvfp4_tensor *out_row, const nvfp4_tensor *out_col,
                                              nvfp4_stream_t stream);

/* Human-readable name of a status. */
NVFP4_API const char *nvfp4_status_string(nvfp4_status status);

/*
 * Synchronize `stream`, then read and clear the device status word that
 * kernels set when a bounded wait runs out.  Returns NVFP4_OK,
 * NVFP4_ERR_TIMEOUT, or NVFP4_ERR_CUDA if the synchronization failed.
 */
NVFP4_API nvfp4_status nvfp4_device_error(nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */

/*
 * nvfp4_oracle.h -- plain, slow CPU oracle for the NVFP4 linear-layer pipeline.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this code.  It shares no source with
 * the CUDA library: no headers, tables, constants or helpers.
 *
 * Every floating-point step is a single IEEE-754 binary32 (or binary64 where
 * stated) operation with round-to-nearest-even; the build uses
 * -ffp-contract=off so no multiply-add is fused.
 *
 * Sources (page title, section):
 *  - "Full-Stack FP4" (academ.us 2607.04422), Sec. 2 Preliminaries: NVFP4 is
 *    E2M1 values times an E4M3 block scale s (blocks of 1x16 or 16x16) times
 *    an FP32 global scale s_g; decode x^ = x_E2M1 * s * s_g.
 *  - same page, Sec. 3.2 Eq. (1)-(2): Fprop/Dgrad/Wgrad operand quantizers
 *    Q_1x16, Q_16x1, Q_16x16 and the 16x16 random Hadamard H16^r.
 *  - same page, Appendix 7: E2M1 bins/steps, RTN error <= step/2, SR rounds
 *    up with probability d/step.
 *  - "Pretraining Large Language Models with NVFP4" (paperlayer 2509.25149v2)
 *    Sec. 2 NVFP4 Format and Sec. 4 / B.4: block amax maps to the FP4 maximum,
 *    FP32 tensor scale keeps block scales inside E4M3, round-to-nearest-even,
 *    RHT scale computed in the rotated space, H H^T = I.
 *  - "OptiTrain-FP4" README (github mirror): E2M1 enumeration with bias 1,
 *    Sylvester recursion H_2k = [[H_k, H_k], [H_k, -H_k]], 1/sqrt(N) norm.
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *    easy as 1, 2, 3" (SC'11).  The pages do not name the generator.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* E2M1 code (4 bits: sign, 2 exponent, 1 mantissa) -> value. */
double oracle_e2m1_value(uint8_t code);
/* Nearest E2M1 value of v, ties to the even mantissa, saturating at 6. */
uint8_t oracle_e2m1_rne(float v);
/* Stochastic rounding of v with a 16-bit random value (low 16 bits). */
uint8_t oracle_e2m1_sr(float v, uint32_t rand16);

/* E4M3 (FN variant, bias 7, max 448, 0x7F = NaN) code -> value. */
double oracle_e4m3_value(uint8_t code);
/* Nearest E4M3 code of a finite x >= 0, ties to even, saturating at 448. */
uint8_t oracle_e4m3_rne_satfinite(float x);

/* Philox4x32-10 block function. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* The 16 random bits that stochastic rounding of element `idx` uses. */
uint32_t oracle_sr_bits(uint64_t seed, uint64_t stream_id, uint64_t idx);

/* y = (1/4) * H16 * D * x, D = diag(bit i of sign_mask ? -1 : +1). */
void oracle_rht16(const float x[16], uint16_t sign_mask, float y[16]);

/* Encode scale S_enc and decode scale s_g from the tensor amax. */
void oracle_tensor_scale(float amax, float *s_enc, float *s_g);

/* Orientation of an encoded operand. */
enum { ORACLE_ROWWISE = 1, ORACLE_COLWISE = 2 };

/*
 * Tensor amax of the values one orientation encodes: max |x| without RHT,
 * max |U x_block| over the blocks along that orientation's reduction
 * dimension with RHT.  x is bf16 bit patterns, [rows][ld] row-major.
 */
float oracle_amax(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                  int orientation, int use_rht, uint16_t sign_mask);

/*
 * Quantize logical rows [lr0, lr1) of one orientation.  The logical matrix is
 * x itself (ROWWISE, [rows][cols]) or its transpose (COLWISE, [cols][rows]);
 * its columns are the reduction dimension.  amax is oracle_amax() of the
 * same orientation.  Output: codes [(lr1-lr0)][Lc/2] (lower column index in
 * the low nibble) and scales [(lr1-lr0)][Lc/16] row-major, Lc = logical cols.
 * scaling: 0 = 1x16 blocks, 1 = 16x16 tiles of x, 2 = 1x16 blocks with the
 * 4/6 choice (amax mapped to 6 or to 4, whichever RNE candidate is closer).
 * rounding: 0 RNE, 1 SR.
 * Returns 0 on success, nonzero on a bad shape.
 */
int oracle_quantize_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                         int scaling, int rounding, int use_rht, uint16_t sign_mask,
                         uint64_t seed, uint64_t stream_id, int orientation,
                         float amax, int64_t lr0, int64_t lr1,
                         uint8_t *codes, uint8_t *scales);

/* Dequantize [rows][cols] (row-major scales [rows][cols/16]) to binary64. */
void oracle_dequantize(const uint8_t *codes, const uint8_t *scales, float s_g,
                       int64_t rows, int64_t cols, double *out);

/* Round binary64 to bfloat16 (nearest, ties to even) in a single step. */
uint16_t oracle_round_bf16(double v);
/* oracle_round_bf16 of each of n values. */
void oracle_round_bf16_array(const double *v, int64_t n, uint16_t *out);

/*
 * y[i][n] = s_gA*s_gB * sum_k (e2m1(a)*s_A)(e2m1(b)*s_B) in binary64 for the
 * listed rows of A (all rows if row_ids is NULL), and abs_sum the same sum of
 * absolute products (NULL to skip).  A is [M][K] codes / [M][K/16] scales,
 * B is [N][K], both contiguous.
 */
void oracle_gemm_f64(const uint8_t *a_codes, const uint8_t *a_scales, float a_sg,
                     const uint8_t *b_codes, const uint8_t *b_scales, float b_sg,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *row_ids, int64_t n_rows,
                     double *y, double *abs_sum);

/* Element-wise array forms of the scalar encoders above (same arithmetic). */
void oracle_e2m1_rne_array(const float *v, int64_t n, uint8_t *codes);
void oracle_e2m1_sr_array(const float *v, const uint32_t *rand16, int64_t n, uint8_t *codes);
void oracle_e4m3_rne_satfinite_array(const float *x, int64_t n, uint8_t *codes);

/* Threads the OpenMP loops use (1 without OpenMP). */
int oracle_num_threads(void);

/*
 * Wgrad's second operand from the forward's quantized input ("Full-Stack
 * FP4", Sec. 3.2 Eq. (2)): dequantize the row-wise 1x16 operand (codes
 * [rows][cols/2], row-major scales [rows][cols/16], s_g) to binary32, apply
 * the RHT along the rows and quantize col-wise with 1x16 blocks along the
 * rows.  Logical rows [lr0, lr1) of the [cols][rows] output; amax < 0
 * computes the tensor amax (returned in *amax_out).  Returns 0 on success.
 */
int oracle_requantize_col_rht(const uint8_t *codes, const uint8_t *scales, float s_g,
                              int64_t rows, int64_t cols, int rounding, uint16_t sign_mask,
                              uint64_t seed, uint64_t stream_id, float amax,
                              int64_t lr0, int64_t lr1, uint8_t *out_codes, uint8_t *out_scales,
                              float *amax_out);

#ifdef __cplusplus
}
#endif
#endif

/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 linear-layer pipeline.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
 * CPU-baseline leg are its only users.  It shares no code with the CUDA
 * library.  Build: -O2 -ffp-contract=off, no fast-math; OpenMP only across
 * independent output rows / elements.
 *
 * The citations name the page and the section each step follows; see
 * nvfp4_oracle.h for the list of pages.
 *
 * Readings of points the pages leave open (each is a proposal the CUDA path
 * must match bit for bit):
 *  - tensor scale: S_enc = (448*6) / amax_t, s_g = 1 / S_enc, S_enc = 1 when
 *    amax_t = 0 and FLT_MAX when the quotient overflows;
 *  - block scale: s_b = E4M3_rne_satfinite((amax_b / 6) * S_enc);
 *  - encode multiplier r_b = S_enc / s_b (0 when s_b = 0), v = x * r_b;
 *    when that quotient overflows (S_enc near FLT_MAX, s_b < 1: a tensor
 *    amax below about 4e-33), v = (x * S_enc) / s_b, each operation rounded
 *    once, so that zeros stay (signed) zeros and the rest keep their size;
 *  - RNE ties go to the even mantissa; the code's sign bit is v's sign bit;
 *  - SR: round up iff (float)u < frac * 2^16, frac = d / step, u a 16-bit
 *    random value;
 *  - Philox key = (seed lo, seed hi), counter = (g lo, g hi, stream lo,
 *    stream hi), g = idx >> 3; element idx takes 16 bits of word
 *    (idx >> 1) & 3, the low half for even idx; idx = row * cols + col of
 *    the emitted logical matrix (the row-wise index of x for 16x16 scaling);
 *  - RHT butterfly: D first, stages s = 0..3 pairing (i, i ^ 2^s) into
 *    (a + b, a - b) with a at the lower index, then * 0.25.
 */
#include "nvfp4_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* E2M1 ("OptiTrain-FP4" README, FP4 grid enumeration: sign, 2 exponent
 * bits, 1 mantissa bit, bias 1; codes 0..7 are 0, .5, 1, 1.5, 2, 3, 4, 6). */
static const float kE2M1Magnitude[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

double oracle_e2m1_value(uint8_t code)
{
    double mag = (double)kE2M1Magnitude[code & 7u];
    return (code & 8u) ? -mag : mag;
}

/* Round to nearest, ties to even ("Pretraining LLMs with NVFP4", Sec. 4,
 * round-to-nearest-even for weights and activations).  Written as a plain
 * nearest-point search over the grid; values above 6 land on 6. */
uint8_t oracle_e2m1_rne(float v)
{
    uint8_t sign = signbit(v) ? 8u : 0u;
    double a = fabs((double)v);
    if (a >= 6.0)                    /* beyond the grid: saturate at 6 */
        return (uint8_t)(sign | 7u);
    int best = 0;
    double best_dist = fabs(a - (double)kE2M1Magnitude[0]);
    for (int k = 1; k < 8; ++k) {
        double dist = fabs(a - (double)kE2M1Magnitude[k]);
        /* equal distance: keep the code whose mantissa bit is 0 */
        if (dist < best_dist || (dist == best_dist && (k & 1) == 0)) {
            best = k;
            best_dist = dist;
        }
    }
    return (uint8_t)(sign | (uint8_t)best);
}

/* Stochastic rounding ("Full-Stack FP4", Appendix 7: for u in [c_k, c_k+1]
 * with d = u - c_k, round up to c_k+1 with probability d / step_k).  The
 * probability is realised with a 16-bit random value r: up iff
 * (float)r < frac * 2^16, so P(up) = ceil(frac * 2^16) / 2^16. */
uint8_t oracle_e2m1_sr(float v, uint32_t rand16)
{
    uint8_t sign = signbit(v) ? 8u : 0u;
    float a = fabsf(v);
    if (a >= 6.0f)
        return (uint8_t)(sign | 7u);
    int k = 0;
    while (k < 6 && !(a < kE2M1Magnitude[k + 1]))
        ++k;                                             /* c_k <= a < c_k+1 */
    float d = a - kE2M1Magnitude[k];                     /* exact: c_k >= a/2 or c_k = 0 */
    float step = kE2M1Magnitude[k + 1] - kE2M1Magnitude[k];  /* a power of two */
    float frac = d / step;                               /* exact */
    float u16 = (float)(rand16 & 0xFFFFu);               /* exact, < 2^16 */
    int up = u16 < frac * 65536.0f;                      /* both sides exact */
    return (uint8_t)(sign | (uint8_t)(k + up));
}

/* ------------------------------------------------------------------ */
/* E4M3, FN variant: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 = NaN, largest finite 448 ("Pretraining LLMs
 * with NVFP4", Sec. 2: E4M3 block scales). */
double oracle_e4m3_value(uint8_t code)
{
    unsigned e = (code >> 3) & 0xFu;
    unsigned m = code & 7u;
    double mag;
    if (e == 0xFu && m == 7u)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);                        /* subnormal: m/8 * 2^-6 */
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return (code & 0x80u) ? -mag : mag;
}

/* Nearest finite non-negative E4M3 value (codes 0x00..0x7E), ties to the
 * even code; everything at or beyond 448 lands on 448 (satfinite). */
uint8_t oracle_e4m3_rne_satfinite(float x)
{
    double a = (double)x;
    if (a >= 448.0)                  /* satfinite */
        return 0x7Eu;
    int best = 0;
    double best_dist = fabs(a - oracle_e4m3_value(0));
    for (int c = 1; c <= 0x7E; ++c) {
        double dist = fabs(a - oracle_e4m3_value((uint8_t)c));
        if (dist < best_dist || (dist == best_dist && (c & 1) == 0)) {
            best = c;
            best_dist = dist;
        }
    }
    return (uint8_t)best;
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32->64
 * multiplies with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by the
 * Weyl constants W0 = 0x9E3779B9, W1 = 0xBB67AE85 between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

uint32_t oracle_sr_bits(uint64_t seed, uint64_t stream_id, uint64_t idx)
{
    uint64_t g = idx >> 3;                       /* one Philox block per 8 elements */
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)stream_id,
                       (uint32_t)(stream_id >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    uint32_t word = out[(idx >> 1) & 3u];
    return (idx & 1u) ? (word >> 16) : (word & 0xFFFFu);
}

/* ------------------------------------------------------------------ */
/* 16-point random Hadamard transform U = H16 * D / 4 ("Full-Stack FP4",
 * Sec. 3.2 Eq. (2), H16^r; "OptiTrain-FP4", U = H D / sqrt(N); "Pretraining
 * LLMs with NVFP4" B.4, H H^T = I).  H16 is the Sylvester matrix, applied as
 * an in-place fast Walsh-Hadamard butterfly in binary32. */
void oracle_rht16(const float x[16], uint16_t sign_mask, float y[16])
{
    float t[16];
    for (int i = 0; i < 16; ++i)
        t[i] = ((sign_mask >> i) & 1u) ? -x[i] : x[i];
    for (int s = 0; s < 4; ++s) {
        int h = 1 << s;
        for (int i = 0; i < 16; ++i) {
            if (i & h)
                continue;
            float a = t[i], b = t[i | h];
            t[i] = a + b;
            t[i | h] = a - b;
        }
    }
    for (int i = 0; i < 16; ++i)
        y[i] = t[i] * 0.25f;
}

/* ------------------------------------------------------------------ */
/* Tensor scale ("Pretraining LLMs with NVFP4", Sec. 2: the FP32 tensor scale
 * keeps block scales representable in E4M3; A.2: global scaling first, then
 * block scaling, decode scales stored for the GEMM).  The tensor amax maps
 * onto the largest product of an E4M3 scale and an E2M1 value, 448 * 6. */
void oracle_tensor_scale(float amax, float *s_enc, float *s_g)
{
    float s = (amax == 0.0f) ? 1.0f : 2688.0f / amax;
    if (isinf(s))
        s = FLT_MAX;
    *s_enc = s;
    *s_g = 1.0f / s;
}

/* ------------------------------------------------------------------ */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* The matrix being quantized: bf16 bit patterns, or binary32 values (a
 * dequantized operand), [rows][ld] row-major. */
struct source {
    const uint16_t *bf16;
    const float *f32;
    int64_t ld;
};

static float src_elem(const struct source *x, int64_t r, int64_t c)
{
    return x->f32 ? x->f32[r * x->ld + c] : bf16_bits_to_float(x->bf16[r * x->ld + c]);
}

/* Element j of logical row lr of one orientation. */
static float logical_elem(const struct source *x, int orientation, int64_t lr, int64_t j)
{
    if (orientation == ORACLE_ROWWISE)
        return src_elem(x, lr, j);
    return src_elem(x, j, lr);
}

static float amax_src(const struct source *x, int64_t rows, int64_t cols,
                      int orientation, int use_rht, uint16_t sign_mask);

float oracle_amax(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                  int orientation, int use_rht, uint16_t sign_mask)
{
    struct source src = {x, NULL, ld};
    return amax_src(&src, rows, cols, orientation, use_rht, sign_mask);
}

static float amax_src(const struct source *x, int64_t rows, int64_t cols,
                      int orientation, int use_rht, uint16_t sign_mask)
{
    int64_t lrows = (orientation == ORACLE_ROWWISE) ? rows : cols;
    int64_t lcols = (orientation == ORACLE_ROWWISE) ? cols : rows;
    float amax = 0.0f;
    if (!use_rht) {
#pragma omp parallel for reduction(max : amax) schedule(static)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c) {
                float a = fabsf(src_elem(x, r, c));
                if (a > amax)
                    amax = a;
            }
        return amax;
    }
    /* with the RHT the scale lives in the rotated space ("Pretraining LLMs
     * with NVFP4", B.4) */
#pragma omp parallel for reduction(max : amax) schedule(static)
    for (int64_t lr = 0; lr < lrows; ++lr) {
        for (int64_t b = 0; b < lcols / 16; ++b) {
            float blk[16], rot[16];
            for (int t = 0; t < 16; ++t)
                blk[t] = logical_elem(x, orientation, lr, 16 * b + t);
            oracle_rht16(blk, sign_mask, rot);
            for (int t = 0; t < 16; ++t) {
                float a = fabsf(rot[t]);
                if (a > amax)
                    amax = a;
            }
        }
    }
    return amax;
}

static int quantize_src(const struct source *x, int64_t rows, int64_t cols,
                        int scaling, int rounding, int use_rht, uint16_t sign_mask,
                        uint64_t seed, uint64_t stream_id, int orientation,
                        float amax, int64_t lr0, int64_t lr1,
                        uint8_t *codes, uint8_t *scales);

int oracle_quantize_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                         int scaling, int rounding, int use_rht, uint16_t sign_mask,
                         uint64_t seed, uint64_t stream_id, int orientation,
                         float amax, int64_t lr0, int64_t lr1,
                         uint8_t *codes, uint8_t *scales)
{
    struct source src = {x, NULL, ld};
    return quantize_src(&src, rows, cols, scaling, rounding, use_rht, sign_mask, seed, stream_id,
                        orientation, amax, lr0, lr1, codes, scales);
}

/* The value the E2M1 encoder rounds: x / (s_b * s_g) = x * S_enc / s_b,
 * evaluated as v = x * r_b with r_b = S_enc / s_b ("Full-Stack FP4", Sec. 2:
 * x^ = x_E2M1 * s * s_g, so the encode divides by s * s_g).  When r_b
 * overflows to +inf (S_enc close to FLT_MAX and s_b < 1), x * r_b would be
 * +-inf for every non-zero x and NaN for x = +-0; the quotient is then taken
 * as (x * S_enc) / s_b, whose intermediate stays finite. */
static float encode_value(float x, float r_b, float s_enc, float sb)
{
    if (isinf(r_b))
        return (x * s_enc) / sb;
    return x * r_b;
}

static int quantize_src(const struct source *x, int64_t rows, int64_t cols,
                        int scaling, int rounding, int use_rht, uint16_t sign_mask,
                        uint64_t seed, uint64_t stream_id, int orientation,
                        float amax, int64_t lr0, int64_t lr1,
                        uint8_t *codes, uint8_t *scales)
{
    if (orientation != ORACLE_ROWWISE && orientation != ORACLE_COLWISE)
        return 1;
    int64_t lrows = (orientation == ORACLE_ROWWISE) ? rows : cols;
    int64_t lcols = (orientation == ORACLE_ROWWISE) ? cols : rows;
    if (lcols % 16 != 0 || lr0 < 0 || lr1 > lrows || lr0 > lr1)
        return 2;
    if (scaling < 0 || scaling > 2)
        return 5;
    if (scaling == 1 && (rows % 16 != 0 || cols % 16 != 0))
        return 3;
    if (scaling == 1 && use_rht)
        return 4;

    float s_enc, s_g;
    oracle_tensor_scale(amax, &s_enc, &s_g);
    int64_t nblk = lcols / 16;

#pragma omp parallel for schedule(static)
    for (int64_t lr = lr0; lr < lr1; ++lr) {
        uint8_t *crow = codes + (lr - lr0) * (lcols / 2);
        uint8_t *srow = scales + (lr - lr0) * nblk;
        for (int64_t b = 0; b < nblk; ++b) {
            float blk[16];
            for (int t = 0; t < 16; ++t)
                blk[t] = logical_elem(x, orientation, lr, 16 * b + t);
            if (use_rht) {
                float rot[16];
                oracle_rht16(blk, sign_mask, rot);
                memcpy(blk, rot, sizeof blk);
            }

            /* block amax: the 1x16 block, or the 16x16 tile of x that holds it
             * ("Full-Stack FP4", Sec. 2: blocks of 16x16 or 1x16) */
            float amax_b = 0.0f;
            if (scaling != 1) {
                for (int t = 0; t < 16; ++t)
                    if (fabsf(blk[t]) > amax_b)
                        amax_b = fabsf(blk[t]);
            } else {
                int64_t r0 = (orientation == ORACLE_ROWWISE) ? (lr / 16) * 16 : 16 * b;
                int64_t c0 = (orientation == ORACLE_ROWWISE) ? 16 * b : (lr / 16) * 16;
                for (int64_t i = 0; i < 16; ++i)
                    for (int64_t j = 0; j < 16; ++j) {
                        float a = fabsf(src_elem(x, r0 + i, c0 + j));
                        if (a > amax_b)
                            amax_b = a;
                    }
            }

            /* block amax -> FP4 maximum 6 ("Pretraining LLMs with NVFP4", Sec. 2) */
            float sb32 = (amax_b / 6.0f) * s_enc;
            uint8_t sb_code = oracle_e4m3_rne_satfinite(sb32);
            float sb = (float)oracle_e4m3_value(sb_code);
            float r_b = (sb == 0.0f) ? 0.0f : s_enc / sb;

            /* 4/6 adaptive scaling ("Full-Stack FP4", Sec. 1 and related
             * work: 4/6 adds MSE-optimal adaptive block scaling; the rule is
             * not printed).  Reading: the block is also encoded with its amax
             * mapped to 4; each candidate is encoded with RNE and measured by
             * sum_i (x_i S_enc - e2m1(q_i) s)^2 in binary32 (x_i S_enc and
             * the difference rounded once each, the squares accumulated in
             * index order by fused multiply-adds); the 4 candidate is kept
             * only when strictly closer.  With SR the chosen scale is then
             * used for the stochastic encode. */
            if (scaling == 2) {
                float sb32_4 = (amax_b / 4.0f) * s_enc;
                uint8_t code4 = oracle_e4m3_rne_satfinite(sb32_4);
                float sb4 = (float)oracle_e4m3_value(code4);
                float r4 = (sb4 == 0.0f) ? 0.0f : s_enc / sb4;
                float err6 = 0.0f, err4 = 0.0f;
                for (int t = 0; t < 16; ++t) {
                    float xs = blk[t] * s_enc;
                    float g6 = (float)oracle_e2m1_value(oracle_e2m1_rne(encode_value(blk[t], r_b, s_enc, sb)));
                    float g4 = (float)oracle_e2m1_value(oracle_e2m1_rne(encode_value(blk[t], r4, s_enc, sb4)));
                    float d6 = xs - g6 * sb;
                    float d4 = xs - g4 * sb4;
                    err6 = fmaf(d6, d6, err6);
                    err4 = fmaf(d4, d4, err4);
                }
                if (err4 < err6) {
                    sb_code = code4;
                    r_b = r4;
                    sb = sb4;
                }
            }
            srow[b] = sb_code;

            for (int t = 0; t < 16; t += 2) {
                uint8_t q[2];
                for (int u = 0; u < 2; ++u) {
                    int64_t j = 16 * b + t + u;
                    float v = encode_value(blk[t + u], r_b, s_enc, sb);
                    if (rounding == 0) {
                        q[u] = oracle_e2m1_rne(v);
                    } else {
                        uint64_t idx;
                        if (scaling == 1)   /* row-wise index of x, both orientations */
                            idx = (orientation == ORACLE_ROWWISE)
                                      ? (uint64_t)(lr * cols + j)
                                      : (uint64_t)(j * cols + lr);
                        else
                            idx = (uint64_t)(lr * lcols + j);
                        q[u] = oracle_e2m1_sr(v, oracle_sr_bits(seed, stream_id, idx));
                    }
                }
                crow[(16 * b + t) / 2] = (uint8_t)(q[0] | (q[1] << 4));
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Decode x^ = x_E2M1 * s * s_g ("Full-Stack FP4", Sec. 2). */
void oracle_dequantize(const uint8_t *codes, const uint8_t *scales, float s_g,
                       int64_t rows, int64_t cols, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = codes[r * (cols / 2) + c / 2];
            uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xFu);
            double s = oracle_e4m3_value(scales[r * (cols / 16) + c / 16]);
            out[r * cols + c] = oracle_e2m1_value(code) * s * (double)s_g;
        }
}

/* ------------------------------------------------------------------ */
/* Wgrad's second operand re-quantized from the forward's quantized input
 * ("Full-Stack FP4", Sec. 3.2 Eq. (2): Q_16x1(H16^T Q_1x16(X))).  The row-wise
 * operand (codes [rows][cols/2], scales [rows][cols/16] row-major, s_g) is
 * dequantized to binary32, x^ = RN(RN(e2m1 * s_b) * s_g) (the first product is
 * exact), and then quantized like oracle_quantize_rows with the RHT in the
 * COLWISE orientation: 16 consecutive rows of a column form a block, the
 * output is [cols][rows] (K-major along rows).  amax < 0 asks for the tensor
 * amax of the rotated dequantized values; it is returned in *amax_out. */
int oracle_requantize_col_rht(const uint8_t *codes, const uint8_t *scales, float s_g,
                              int64_t rows, int64_t cols, int rounding, uint16_t sign_mask,
                              uint64_t seed, uint64_t stream_id, float amax,
                              int64_t lr0, int64_t lr1, uint8_t *out_codes, uint8_t *out_scales,
                              float *amax_out)
{
    if (rows % 16 != 0 || cols % 16 != 0)
        return 2;
    float *xf = (float *)malloc((size_t)(rows * cols) * sizeof(float));
    if (!xf)
        return 6;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = codes[r * (cols / 2) + c / 2];
            uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xFu);
            float g = (float)oracle_e2m1_value(code);
            float sb = (float)oracle_e4m3_value(scales[r * (cols / 16) + c / 16]);
            float gs = g * sb;
            xf[r * cols + c] = gs * s_g;
        }
    struct source src = {NULL, xf, cols};
    if (amax < 0.0f)
        amax = amax_src(&src, rows, cols, ORACLE_COLWISE, 1, sign_mask);
    if (amax_out)
        *amax_out = amax;
    int rc = quantize_src(&src, rows, cols, 0, rounding, 1, sign_mask, seed, stream_id, ORACLE_COLWISE,
                          amax, lr0, lr1, out_codes, out_scales);
    free(xf);
    return rc;
}

uint16_t oracle_round_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return 0x7FC0u;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                    /* a = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;                /* 8 significant bits */
    if (qexp < -133)                 /* bf16 subnormal quantum 2^-133 */
        qexp = -133;
    double q = rint(ldexp(a, -qexp)); /* nearest, ties to even */
    double r = ldexp(q, qexp);
    if (r > 3.3895313892515355e38)   /* beyond the largest finite bf16 */
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;              /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void oracle_round_bf16_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_round_bf16(v[i]);
}

/* ------------------------------------------------------------------ */
/* y = s_gA s_gB sum_k (e2m1(a_k) s_A)(e2m1(b_k) s_B): the three linear-layer
 * GEMMs with FP4 inputs ("Full-Stack FP4", Sec. 2 Linear projection;
 * "Pretraining LLMs with NVFP4", Sec. 4 Mixed precision).  Every product is
 * exact in binary64; the sum runs k = 0 .. K-1 in binary64. */
void oracle_gemm_f64(const uint8_t *a_codes, const uint8_t *a_scales, float a_sg,
                     const uint8_t *b_codes, const uint8_t *b_scales, float b_sg,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *row_ids, int64_t n_rows,
                     double *y, double *abs_sum)
{
    double e2m1[16], e4m3[256];
    for (int c = 0; c < 16; ++c)
        e2m1[c] = oracle_e2m1_value((uint8_t)c);
    for (int c = 0; c < 256; ++c)
        e4m3[c] = oracle_e4m3_value((uint8_t)c);
    double sg = (double)a_sg * (double)b_sg;   /* exact: 48 significant bits */
    int64_t nr = row_ids ? n_rows : M;

#pragma omp parallel for schedule(static)
    for (int64_t idx = 0; idx < nr * N; ++idx) {
        int64_t i = idx / N, n = idx % N;
        int64_t m = row_ids ? row_ids[i] : i;
        const uint8_t *ac = a_codes + m * (K / 2), *as = a_scales + m * (K / 16);
        const uint8_t *bc = b_codes + n * (K / 2), *bs = b_scales + n * (K / 16);
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            uint8_t ca = (k & 1) ? (uint8_t)(ac[k / 2] >> 4) : (uint8_t)(ac[k / 2] & 0xFu);
            uint8_t cb = (k & 1) ? (uint8_t)(bc[k / 2] >> 4) : (uint8_t)(bc[k / 2] & 0xFu);
            double pa = e2m1[ca] * e4m3[as[k / 16]];
            double pb = e2m1[cb] * e4m3[bs[k / 16]];
            double p = pa * pb;
            acc += p;
            acc_abs += fabs(p);
        }
        y[i * N + n] = acc * sg;
        if (abs_sum)
            abs_sum[i * N + n] = acc_abs * sg;
    }
}

void oracle_e2m1_rne_array(const float *v, int64_t n, uint8_t *codes)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        codes[i] = oracle_e2m1_rne(v[i]);
}

void oracle_e2m1_sr_array(const float *v, const uint32_t *rand16, int64_t n, uint8_t *codes)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        codes[i] = oracle_e2m1_sr(v[i], rand16[i]);
}

void oracle_e4m3_rne_satfinite_array(const float *x, int64_t n, uint8_t *codes)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        codes[i] = oracle_e4m3_rne_satfinite(x[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

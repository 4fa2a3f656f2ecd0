// device_common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a).
//
// Inline-PTX wrappers for mbarrier, TMA (cp.async.bulk*) and tcgen05, plus the
// bit-level helpers of the NVFP4 format (E2M1 codes, E4M3 block scales, the
// tile layout of the scale buffer).  Format facts: "Full-Stack FP4", Sec. 2
// (x^ = x_E2M1 * s * s_g, 16-element blocks, E4M3 s, FP32 s_g); the byte and
// bit layouts are the ones documented in include/nvfp4.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace nvfp4 {

// ---------------------------------------------------------------- scales ---
// Offset of block scale (r, j) in the tile layout: 128-row x 4-scale tiles of
// 512 bytes, rows interleaved as (r % 32) * 16 + ((r / 32) % 4) * 4.
__host__ __device__ __forceinline__ uint64_t scale_offset(uint32_t r, uint32_t j, uint32_t s4) {
    return ((uint64_t)(r >> 7) * s4 + (j >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u +
           (j & 3u);
}

// ------------------------------------------------------------ conversions ---
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3 (FN) encode of a finite non-negative value: nearest, ties to even,
// saturating at 448.
__device__ __forceinline__ uint32_t e4m3_encode_satfinite(float x) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(x));
    return pair & 0xFFu;
}

// E4M3 decode of a non-negative code (exact).
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0) return __uint2float_rn(m) * 0.001953125f;       // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));     // 2^(e-7) * (1 + m/8)
}

// Eight values -> eight E2M1 codes (RNE, saturating), element 0 in the low
// nibble.  The conversion keeps each value's sign bit also when the value
// rounds to zero (-0, -0.1 and -1e-40 give 0x8 on sm_103a) and rounds ties
// to the even code, which is the oracle's rule; the GPU tests check both.
__device__ __forceinline__ uint32_t e2m1_rne_x8(const float* v) {
    uint32_t out;
    asm("{\n\t"
        ".reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t"
        "}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// Stochastic rounding of one value to the E2M1 grid with 16 random bits
// ("Full-Stack FP4", Appendix 7: round up with probability d / step): up iff
// r16 < frac * 2^16, i.e. iff r16 < ceil(frac * 2^16).
//
// Done on the FP32 bit pattern.  In each binade [2^e, 2^(e+1)) with e >= 0
// the E2M1 grid keeps one mantissa bit, so frac is the low 22 mantissa bits
// over 2^22, and adding ((2^16 - 1 - r16) << 6) + 63 to the pattern carries
// into bit 22 exactly when r16 < ceil(frac * 2^16); clearing the low 22 bits
// then leaves the rounded value.  Below 1 the grid {0, 0.5, 1} is that of
// [1, 2) shifted by one and halved: z = (|v| + 1) / 2, one fused multiply-add
// rounded upward (which keeps ceil(frac * 2^16): float spacing there, 2^-24,
// is finer than 2^-18), lies in [0.5, 1) where the same addition applies,
// and 2 z - 1 maps the rounded z back.  max(|v|, (|v| + 1) / 2) selects z
// exactly when |v| < 1; the rounded value q maps back as q - sat(1 - q),
// which is 2 q - 1 for q in [0.5, 1) and q from 1 up (every step exact),
// on the FMA pipe (the kernels that round stochastically are bound by the
// integer/logic pipe, where a min would run).  The result is |v|'s rounded value with v's sign: a grid value, or
// a value >= 6 (|v| > 6 can round to 8 or 12), which the saturating RNE
// conversion e2m1_rne_x8 then turns into the code without rounding, so no
// clamp to 6 is needed.  With finite v, |v| here stays below 9 (the block
// scale's E4M3 rounding error is at most 1/2 of its smallest subnormal step).
__device__ __forceinline__ uint32_t sr_addend_lo(uint32_t w) { return ((~w << 6) & 0x3FFFC0u) | 63u; }
__device__ __forceinline__ uint32_t sr_addend_hi(uint32_t w) { return (~w >> 10) | 63u; }

// Both addends of one Philox word, 0x3FFFFF - 64 r for r = its low and its
// high 16 bits (the same values as sr_addend_lo / sr_addend_hi), as integer
// multiply-adds: they run on the FMA pipe while the rounding itself keeps
// the integer ALU busy.
__device__ __forceinline__ void sr_addends(uint32_t w, uint32_t& lo, uint32_t& hi) {
    uint32_t h16, t;
    asm("mul.hi.u32 %0, %1, 65536;" : "=r"(h16) : "r"(w));
    asm("mad.lo.u32 %0, %1, 4294967232, 4194303;" : "=r"(hi) : "r"(h16));       // 0x3FFFFF - 64 h16
    asm("mad.lo.u32 %0, %1, 4194304, 4194303;" : "=r"(t) : "r"(h16));            // 0x3FFFFF + 2^22 h16
    asm("mad.lo.u32 %0, %1, 4294967232, %2;" : "=r"(lo) : "r"(w), "r"(t));     // 0x3FFFFF - 64 (w - 2^16 h16)
}

__device__ __forceinline__ float e2m1_sr_grid(float v, uint32_t addend) {
    const float a = fabsf(v);
    const float z = fmaxf(a, __fmaf_ru(a, 0.5f, 0.5f));
    const float zt = __uint_as_float((__float_as_uint(z) + addend) & 0xFFC00000u);
    const float q = __fsub_rn(zt, __saturatef(__fmaf_rn(zt, -1.0f, 1.0f)));
    return __uint_as_float(__float_as_uint(q) | (__float_as_uint(v) & 0x80000000u));
}

// --------------------------------------------------------------- Philox ----
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies; the key is bumped by the Weyl constants between
// rounds.  The ten round keys depend only on the seed, so the host forms them
// once and the kernels read them from their parameters (no registers, no
// per-round key additions).
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};

__host__ __device__ __forceinline__ PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        k.k0[r] = a;
        k.k1[r] = b;
        a += 0x9E3779B9u;
        b += 0xBB67AE85u;
    }
    return k;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k.k0[r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k.k1[r],
                       (uint32_t)p0);
    }
    return c;
}

// The Philox block of SR elements 8g .. 8g+7: element 8g + i takes 16 bits of
// word i / 2, the low half for even i.
__device__ __forceinline__ uint4 sr_words4(const PhiloxKeys& keys, uint64_t stream_id, uint64_t g) {
    return philox4x32_10(
        make_uint4((uint32_t)g, (uint32_t)(g >> 32), (uint32_t)stream_id, (uint32_t)(stream_id >> 32)), keys);
}

// ------------------------------------------------------------------ RHT ----
// The sign flips D of the RHT as XOR words on packed bf16 pairs, formed on
// the host and read from the kernel parameters, so that each flip is one XOR
// of a loaded word: col[i] flips both values of a word when bit i of the
// mask is set (two columns of row i, the transform running down the
// columns); row[k] flips the low value by bit 2k and the high value by bit
// 2k + 1 (columns 2k and 2k + 1 of one row, the transform along the row).
struct RhtSigns {
    uint32_t col[16];
    uint32_t row[8];
};

__host__ __device__ inline RhtSigns rht_signs(uint32_t mask) {
    RhtSigns s;
    for (int i = 0; i < 16; ++i) s.col[i] = ((mask >> i) & 1u) ? 0x80008000u : 0u;
    for (int k = 0; k < 8; ++k)
        s.row[k] = (((mask >> (2 * k)) & 1u) ? 0x00008000u : 0u) | (((mask >> (2 * k + 1)) & 1u) ? 0x80000000u : 0u);
    return s;
}

// t <- H16 * D * t (without the 1/4): negate per mask, butterfly stages 0..3.
// With bf16 inputs every value here is a multiple of 2^-133, so t / 4 is
// exact even when subnormal: max|t| / 4 is the amax of the scaled transform,
// and RN((t / 4) r) = RN(t (r / 4)) whenever r / 4 is exact.
__device__ __forceinline__ void rht16_unscaled(float* t, uint32_t sign_mask) {
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __uint_as_float(__float_as_uint(t[i]) ^ (((sign_mask >> i) & 1u) << 31));
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & (1 << s)) continue;
            const float a = t[i], b = t[i | (1 << s)];
            t[i] = __fadd_rn(a, b);
            t[i | (1 << s)] = __fsub_rn(a, b);
        }
    }
}

// rht16_unscaled on two blocks at once, as packed binary32 pairs (a[i], b[i]):
// each lane of add.rn.f32x2 / sub.rn.f32x2 rounds like the scalar operation,
// so the results are those of two rht16_unscaled calls, in half the
// instructions.
__device__ __forceinline__ void rht16_unscaled_x2(float* a, float* b, uint32_t sign_mask) {
    uint64_t t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t sgn = ((sign_mask >> i) & 1u) << 31;
        asm("mov.b64 %0, {%1, %2};"
            : "=l"(t[i])
            : "r"(__float_as_uint(a[i]) ^ sgn), "r"(__float_as_uint(b[i]) ^ sgn));
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & (1 << s)) continue;
            uint64_t sum, dif;
            asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(t[i]), "l"(t[i | (1 << s)]));
            asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dif) : "l"(t[i]), "l"(t[i | (1 << s)]));
            t[i] = sum;
            t[i | (1 << s)] = dif;
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(t[i]));
        a[i] = __uint_as_float(lo);
        b[i] = __uint_as_float(hi);
    }
}

// rht16_unscaled of one block with stages 0-2 on packed pairs (t[i], t[i + 8])
// (stage s < 3 pairs i with i ^ 2^s in both halves alike) and stage 3, which
// pairs the two halves, in scalar: the same operations in the same order.
__device__ __forceinline__ void rht16_unscaled_packed(float* t, uint32_t sign_mask) {
    uint64_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = __float_as_uint(t[i]) ^ (((sign_mask >> i) & 1u) << 31);
        const uint32_t hi = __float_as_uint(t[i + 8]) ^ (((sign_mask >> (i + 8)) & 1u) << 31);
        asm("mov.b64 %0, {%1, %2};" : "=l"(p[i]) : "r"(lo), "r"(hi));
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i & (1 << s)) continue;
            uint64_t sum, dif;
            asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(p[i]), "l"(p[i | (1 << s)]));
            asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dif) : "l"(p[i]), "l"(p[i | (1 << s)]));
            p[i] = sum;
            p[i | (1 << s)] = dif;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(p[i]));
        t[i] = __fadd_rn(__uint_as_float(lo), __uint_as_float(hi));
        t[i + 8] = __fsub_rn(__uint_as_float(lo), __uint_as_float(hi));
    }
}

__device__ __forceinline__ void scale16(float* t, float f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __fmul_rn(t[i], f);
}

// ------------------------------------------------------------ tensor scale -
struct TensorScale {
    float s_enc, s_g;
};

// S_enc = 2688 / amax (1 if amax == 0, FLT_MAX on overflow), s_g = 1 / S_enc.
__device__ __forceinline__ TensorScale tensor_scale(float amax) {
    float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(2688.0f, amax);
    if (isinf(s)) s = 3.402823466e38f;
    return {s, __fdiv_rn(1.0f, s)};
}

// RN(a / 6) for a >= 0 without a division: q0 = RN(a * RN(1/6)), the exact
// remainder a - 6 q0 by one fused multiply-add, and one correction step
// q0 + remainder * RN(1/6) (Markstein's method for division by a constant,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", 1990).  An exhaustive comparison with IEEE division on sm_103a
// over every non-negative float found it exact from 2^-125 up; below that
// the quotient is subnormal and the division is done as such.
__device__ __forceinline__ float div6_rn(float a) {
    if (a < 0x1p-125f) return __fdiv_rn(a, 6.0f);
    const float c6 = 0x1.555556p-3f;
    const float q0 = __fmul_rn(a, c6);
    const float r = __fmaf_rn(-q0, 6.0f, a);
    return __fmaf_rn(r, c6, q0);
}

// Block scale code and encode multiplier r_b from the block amax.
__device__ __forceinline__ uint32_t block_scale(float amax_b, float s_enc, float* r_b) {
    const float sb32 = __fmul_rn(div6_rn(amax_b), s_enc);
    const uint32_t code = e4m3_encode_satfinite(sb32);
    const float sb = e4m3_decode(code);
    *r_b = (sb == 0.0f) ? 0.0f : __fdiv_rn(s_enc, sb);
    return code;
}

// The multipliers r_b = S_enc / s_b of all 127 finite non-negative E4M3
// codes, for a CTA to look up instead of dividing per block (the same single
// division, done once per code).  Threads 0..127 fill it; callers sync.
__device__ __forceinline__ void fill_rb_table(float* table, float s_enc, float mult = 1.0f) {
    if (threadIdx.x < 128) {
        const float sb = e4m3_decode(threadIdx.x);
        table[threadIdx.x] =
            (threadIdx.x == 0 || threadIdx.x == 127) ? 0.0f : __fmul_rn(__fdiv_rn(s_enc, sb), mult);
    }
}

// Whether an RHT encode may take the transform's 1/4 into its multipliers
// (table entries r_b / 4): exact for every code when the smallest r_b,
// S_enc / 448, is at least 2^-124, so that r_b / 4 stays normal.  Otherwise
// (tensor amax above about 1.3e38) the 1/4 is applied to the values.
__device__ __forceinline__ bool rht_quarter_foldable(float s_enc) { return __fdiv_rn(s_enc, 448.0f) >= 0x1p-124f; }

// fill_rb_table by threads [first, first + 128).
__device__ __forceinline__ void fill_rb_table_at(float* table, float s_enc, uint32_t first, float mult = 1.0f) {
    const uint32_t c = threadIdx.x - first;
    if (threadIdx.x >= first && c < 128) {
        const float sb = e4m3_decode(c);
        table[c] = (c == 0 || c == 127) ? 0.0f : __fmul_rn(__fdiv_rn(s_enc, sb), mult);
    }
}

__device__ __forceinline__ uint32_t block_scale_tab(float amax_b, float s_enc, const float* table, float* r_b) {
    const float sb32 = __fmul_rn(div6_rn(amax_b), s_enc);
    const uint32_t code = e4m3_encode_satfinite(sb32);
    *r_b = table[code];
    return code;
}

// The values of eight E2M1 codes (element 0 in the low nibble), signed.
__device__ __forceinline__ void e2m1_decode_x8(uint32_t w, float* g) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float lo, hi;
        asm("{\n\t"
            ".reg .b8 t;\n\t"
            ".reg .b32 h2;\n\t"
            ".reg .f16 l, h;\n\t"
            "cvt.u8.u32 t, %2;\n\t"
            "cvt.rn.f16x2.e2m1x2 h2, t;\n\t"
            "mov.b32 {l, h}, h2;\n\t"
            "cvt.f32.f16 %0, l;\n\t"
            "cvt.f32.f16 %1, h;\n\t"
            "}"
            : "=f"(lo), "=f"(hi)
            : "r"(w >> (8 * k)));
        g[2 * k] = lo;
        g[2 * k + 1] = hi;
    }
}

// The two E2M1 codes of one byte (low nibble first), as values.
__device__ __forceinline__ void e2m1_decode_byte(uint32_t b, float& lo, float& hi) {
    asm("{\n\t"
        ".reg .b8 t;\n\t"
        ".reg .b32 h2;\n\t"
        ".reg .f16 l, h;\n\t"
        "cvt.u8.u32 t, %2;\n\t"
        "cvt.rn.f16x2.e2m1x2 h2, t;\n\t"
        "mov.b32 {l, h}, h2;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, h;\n\t"
        "}"
        : "=f"(lo), "=f"(hi)
        : "r"(b));
}

// The values the E2M1 encoder rounds, v_i = RN(t_i * r_b) (x / (s_b s_g) with
// x^ = x_E2M1 * s_b * s_g: "Full-Stack FP4", Sec. 2).  When r_b = S_enc / s_b
// has overflowed to +inf (S_enc saturated near FLT_MAX and a block scale below
// 1, i.e. tensor amaxes below about 4e-33), t_i * r_b would be +-inf for every
// non-zero t_i and NaN for zeros; such blocks take v_i = RN(RN(t_i * s_mult) /
// s_b) instead, with s_mult = S_enc (times 1/4 when t holds the RHT's values
// before its 1/4, which the multipliers then carry).  The test costs one
// comparison per block.
// (v may be t itself.)  kGuard = false leaves the test out: kernels take
// that form whenever multiplier_may_overflow(S_enc) is false, i.e. for every
// tensor amax above about 4e-33.
// Whether S_enc / s_b can overflow for some E4M3 code: the smallest positive
// s_b is 2^-9, so not while S_enc < FLT_MAX * 2^-9 (about 6.6e35, a tensor
// amax above about 4e-33).  Conservative: a true answer only selects the
// checked form of encode_values.
__device__ __forceinline__ bool multiplier_may_overflow(float s_enc) { return s_enc >= 6.0e35f; }

template <int N, bool kGuard = true>
__device__ __forceinline__ void encode_values(const float* t, float r_b, uint32_t code, float s_mult, float* v) {
    if (kGuard && r_b > 3.402823466e38f) {
        const float sb = e4m3_decode(code);
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = __fdiv_rn(__fmul_rn(t[i], s_mult), sb);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = __fmul_rn(t[i], r_b);
    }
}

// 4/6 adaptive scaling of one 1x16 block (the oracle's reading of the 4/6
// scaling "Full-Stack FP4" names): the block's amax mapped to 6 (the plain
// scale) or to 4, each candidate encoded with RNE and measured by
// sum_i (x_i S_enc - e2m1(q_i) s)^2 in binary32, accumulated in index order by
// fused multiply-adds; the 4 candidate only when strictly closer.  t holds the
// values the multipliers of `table` apply to and xs_mult * t_i = x_i S_enc
// (both carry the RHT's 1/4 when it is folded into the multipliers).  Returns
// the chosen scale code and its multiplier in *r_b; with rne_codes, also the
// chosen candidate's RNE codes (as encode16<false> packs them: the same
// values, so an RNE caller need not encode the block again).
template <bool kGuard = true>
__device__ __forceinline__ uint32_t block_scale_46(const float* t, float amax_b, float s_enc, float xs_mult,
                                                   const float* table, float* r_b, uint2* rne_codes = nullptr) {
    float r6;
    const uint32_t c6 = block_scale_tab(amax_b, s_enc, table, &r6);
    const uint32_t c4 = e4m3_encode_satfinite(__fmul_rn(__fmul_rn(amax_b, 0.25f), s_enc));
    const float r4 = table[c4];
    const float sb6 = e4m3_decode(c6), sb4 = e4m3_decode(c4);
    float v6[16], v4[16];
    encode_values<16, kGuard>(t, r6, c6, xs_mult, v6);
    encode_values<16, kGuard>(t, r4, c4, xs_mult, v4);
    float g6[16], g4[16];
    const uint2 q6 = make_uint2(e2m1_rne_x8(v6), e2m1_rne_x8(v6 + 8));
    const uint2 q4 = make_uint2(e2m1_rne_x8(v4), e2m1_rne_x8(v4 + 8));
    e2m1_decode_x8(q6.x, g6);
    e2m1_decode_x8(q6.y, g6 + 8);
    e2m1_decode_x8(q4.x, g4);
    e2m1_decode_x8(q4.y, g4 + 8);
    // d = RN(x S_enc - g s) in one fused multiply-add: g s is exact (at most
    // 2 + 4 significant bits, between 2^-10 and 2688), so this is the
    // rounded difference of the exact product.  The two candidates' sums
    // advance together as one packed pair (e6, e4): each lane of
    // fma.rn.f32x2 rounds like the scalar fused multiply-add, in index order.
    uint64_t e;
    asm("mov.b64 %0, {%1, %1};" : "=l"(e) : "r"(0u));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float xs = __fmul_rn(t[i], xs_mult);
        const float d6 = __fmaf_rn(-g6[i], sb6, xs);
        const float d4 = __fmaf_rn(-g4[i], sb4, xs);
        uint64_t d;
        asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(d6), "f"(d4));
        asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(e) : "l"(d), "l"(e));
    }
    float e6, e4;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(e6), "=f"(e4) : "l"(e));
    if (e4 < e6) {
        *r_b = r4;
        if (rne_codes) *rne_codes = q4;
        return c4;
    }
    *r_b = r6;
    if (rne_codes) *rne_codes = q6;
    return c6;
}

// Encode the 16 values t of one block with multiplier r_b (scale code `code`;
// s_mult as for encode_values): codes in a uint2 (element 0 in the low nibble
// of byte 0).  idx_base is the SR index of element 0 (a multiple of 16 for
// 1x16 blocks).
template <bool kSR, bool kGuard = true>
__device__ __forceinline__ uint2 encode16(const float* t, float r_b, uint32_t code, float s_mult,
                                          const PhiloxKeys& keys, uint64_t stream_id, uint64_t idx_base) {
    float v[16];
    encode_values<16, kGuard>(t, r_b, code, s_mult, v);
    if constexpr (!kSR) {
        return make_uint2(e2m1_rne_x8(v), e2m1_rne_x8(v + 8));
    } else {
        const uint4 r0 = sr_words4(keys, stream_id, idx_base >> 3);
        const uint4 r1 = sr_words4(keys, stream_id, (idx_base >> 3) + 1);
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float q[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            uint32_t alo, ahi;
            sr_addends(w[k], alo, ahi);
            q[2 * k] = e2m1_sr_grid(v[2 * k], alo);
            q[2 * k + 1] = e2m1_sr_grid(v[2 * k + 1], ahi);
        }
        return make_uint2(e2m1_rne_x8(q), e2m1_rne_x8(q + 8));
    }
}

// ------------------------------------------------------------ reductions ---
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Max over `n` partial maxima, computed by the whole block; every thread gets
// the result.  `red` is __shared__ float[32].
__device__ __forceinline__ float block_max_of(const float* __restrict__ partials, int n, float* red) {
    float m = 0.0f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, partials[i]);
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float r = red[0];
    __syncthreads();
    return r;
}

// Block-wide max written to partials[blockIdx.x] by thread 0.
__device__ __forceinline__ void block_max_store(float m, float* __restrict__ partials, float* red) {
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) partials[blockIdx.x] = v;
    }
}

// --------------------------------------------------------------- memory ----
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread for up to `hint_ns` (it resumes as
// soon as the phase completes): a waiting thread then takes no issue slots
// from the warps sharing its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete, giving up after timeout_ns.
// Returns false on timeout; the caller records it.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait_sleep(a, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// ------------------------------------------------------------------ TMA ----
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// --------------------------------------------------------------- cluster ---
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA of the cluster.  Default semantics: a
// release.cluster arrive costs hundreds of cycles more under memory traffic.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (mbarrier.test_wait).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait on a barrier given by its shared-memory address; the first probe
// does not block (the common case on the MMA issuer's path: already complete).
__device__ __forceinline__ bool mbar_wait_addr(uint32_t a, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_test_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait_sleep(a, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// mbar_wait for barriers that also receive arrivals from the peer CTA.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait_sleep(a, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA tile load whose completion is counted on an mbarrier of the pair's
// leader CTA (cta_group::2 form).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, uint32_t leader_bar, int32_t x,
                                                 int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(leader_bar), "r"(x), "r"(y)
        : "memory");
}

// 3-D TMA tile load completing on an mbarrier of this CTA.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y,
                                            int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// TMA tile store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------- tcgen05 pair ---
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A * B^T issued by the pair's leader: M = 256 split over the two
// CTAs' shared memory and tensor memory, B's N rows split over the two CTAs.
__device__ __forceinline__ void mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// The four K = 64 MMAs of one 256-deep stage.  Descriptors are built from
// their 32-bit low words (start address >> 4 in the low 14 bits, which never
// carry: shared memory is below 256 KiB) and the common high word, so the
// issuing thread spends as few instructions as possible between MMAs.
// B's descriptor is kBOff address units after A's; per K step A and B advance
// 32 bytes (2 units) and the scale columns by 4 (A) and 8 (B), B's scales
// starting 16 columns after A's.
template <bool kAccumulate, uint32_t kBOff>
__device__ __forceinline__ void mma_nvf4_pair_stage(uint32_t d_tmem, uint32_t a_lo, uint32_t desc_hi, uint32_t idesc,
                                                    uint32_t sf_col) {
    asm volatile(
        "{\n\t"
        ".reg .b32 a1, a2, a3, b0, b1, b2, b3, sa1, sa2, sa3, sb0, sb1, sb2, sb3;\n\t"
        ".reg .b64 da0, da1, da2, da3, db0, db1, db2, db3;\n\t"
        ".reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "add.u32 a1, %1, 2;\n\tadd.u32 a2, %1, 4;\n\tadd.u32 a3, %1, 6;\n\t"
        "add.u32 b0, %1, %6;\n\tadd.u32 b1, b0, 2;\n\tadd.u32 b2, b0, 4;\n\tadd.u32 b3, b0, 6;\n\t"
        "add.u32 sa1, %4, 4;\n\tadd.u32 sa2, %4, 8;\n\tadd.u32 sa3, %4, 12;\n\t"
        "add.u32 sb0, %4, 16;\n\tadd.u32 sb1, %4, 24;\n\tadd.u32 sb2, %4, 32;\n\tadd.u32 sb3, %4, 40;\n\t"
        "mov.b64 da0, {%1, %2};\n\tmov.b64 da1, {a1, %2};\n\tmov.b64 da2, {a2, %2};\n\tmov.b64 da3, {a3, %2};\n\t"
        "mov.b64 db0, {b0, %2};\n\tmov.b64 db1, {b1, %2};\n\tmov.b64 db2, {b2, %2};\n\tmov.b64 db3, {b3, %2};\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da0, db0, %3, [%4], [sb0], p;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da1, db1, %3, [sa1], [sb1], 1;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da2, db2, %3, [sa2], [sb2], 1;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da3, db3, %3, [sa3], [sb3], 1;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_lo), "r"(desc_hi), "r"(idesc), "r"(sf_col), "n"(kAccumulate ? 1 : 0), "n"(kBOff)
        : "memory");
}

// Arrive on the mbarrier at the same offset in every CTA of `cta_mask` once
// this thread's pair MMAs so far have completed.
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// tc_commit_pair_multicast on a barrier given by its shared-memory address.
__device__ __forceinline__ void tc_commit_pair_multicast_addr(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(cta_mask)
        : "memory");
}

// --------------------------------------------------------------- tcgen05 ---
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), version 1 at bit 46, swizzle mode at 61.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 / 32 registers per thread -> 32 lanes x 16 / 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace nvfp4

// quantize.cu -- NVFP4 quantizer kernels for sm_103a.
//
// One quantize call is two HBM passes over the bf16 input:
//   pass 1 (amax): every CTA of a persistent grid writes the max |t| of its
//     share to a workspace slot (t = x, or the 16-point RHT of x along the
//     emitted orientation's reduction dimension: "Pretraining LLMs with
//     NVFP4", B.4, the scale is computed in the rotated space);
//   pass 2 (encode): every CTA reduces those slots to the tensor amax, derives
//     S_enc and s_g ("Pretraining LLMs with NVFP4", Sec. 2: FP32 tensor scale,
//     block amax -> FP4 max 6, E4M3 block scale) and encodes its blocks to
//     packed E2M1 codes by RNE or Philox SR ("Full-Stack FP4", Appendix 7).
// Layouts: row-wise blocks are 16 consecutive elements of a row (Q_1x16);
// col-wise blocks are 16 consecutive rows of a column, emitted transposed
// (Q_16x1 of "Full-Stack FP4" Eq. (2)); 16x16 tiles share one scale (Q_16x16).
#include <cuda_runtime.h>

#include <type_traits>

#include "device_common.cuh"
#include "bounds.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

enum class Pass { kAmax, kEncode };

struct Target {
    uint8_t* codes;
    int64_t ld_codes;
    uint8_t* scales;
    uint32_t s4;        // 4-scale groups per logical row
    float* amax;
    float* sg;
    Extent xc, xs;      // the bytes of codes and scales the call may write
};

// Stores into an orientation's codes (logical row r, byte offset off) and
// scales (byte index idx), through the bounds check of the debug build.
template <typename T>
__device__ __forceinline__ void put_codes(const Target& t, int64_t r, int64_t off, const T& v) {
    store_out(reinterpret_cast<T*>(t.codes + r * t.ld_codes + off), v, t.xc);
}
template <typename T>
__device__ __forceinline__ void put_scales(const Target& t, uint32_t idx, const T& v) {
    store_out(reinterpret_cast<T*>(t.scales + idx), v, t.xs);
}

// Tensor scale from the amax partials; CTA 0 publishes amax and s_g.
__device__ __forceinline__ TensorScale load_tensor_scale(const float* partials, int n, float* red,
                                                         const Target& t0, const Target* t1) {
    const float amax = block_max_of(partials, n, red);
    const TensorScale ts = tensor_scale(amax);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (t0.sg) {
            if (t0.amax) *t0.amax = amax;
            *t0.sg = ts.s_g;
        }
        if (t1 && t1->sg) {
            if (t1->amax) *t1->amax = amax;
            *t1->sg = ts.s_g;
        }
    }
    return ts;
}

// ----------------------------------------------------------- row-wise -----
struct RowArgs {
    const uint16_t* x;
    int64_t ld_x;
    uint32_t bpr;      // blocks of 16 per row (cols / 16)
    uint32_t total;    // rows * bpr
    Target out;
    const float* partials_in;
    int n_partials;
    float* partials_out;
    uint32_t mask;
    RhtSigns sg;                 // the mask's sign flips as XOR words
    PhiloxKeys keys;             // SR round keys of the seed
    uint64_t stream;
};

// One thread = one 1x16 block: two 16-byte loads, RHT in registers (optional),
// block amax, E4M3 scale, 8 bytes of codes.
// kS46: 4/6 adaptive block scales (block_scale_46).
template <Pass P, bool kRHT, bool kSR, bool kS46 = false>
__global__ void __launch_bounds__(kThreads) rowwise_kernel(const RowArgs a) {
    __shared__ float red[32];
    __shared__ float rb_table[128];
    TensorScale ts{1.0f, 1.0f};
    bool fold = false;   // the RHT's 1/4 lives in the multipliers (rht_quarter_foldable)
    if constexpr (P == Pass::kEncode) {
        ts = load_tensor_scale(a.partials_in, a.n_partials, red, a.out, nullptr);
        if constexpr (kRHT) fold = rht_quarter_foldable(ts.s_enc);
        fill_rb_table(rb_table, ts.s_enc, fold ? 0.25f : 1.0f);
        __syncthreads();
    }
    // the values' factor S_enc (with the RHT's 1/4 when it is folded)
    const float s_mult = fold ? __fmul_rn(ts.s_enc, 0.25f) : ts.s_enc;
    float local_max = 0.0f;
    const PhiloxKeys& keys = a.keys;   // SR round keys, formed by the host
    // block b = r * bpr + j; (r, j) advance by the grid stride without a division
    const uint32_t stride = gridDim.x * kThreads;
    const uint32_t stride_r = stride / a.bpr, stride_j = stride - stride_r * a.bpr;
    uint32_t b = blockIdx.x * kThreads + threadIdx.x;
    uint32_t r = b / a.bpr, j = b - r * a.bpr;
    // the main loop, instantiated with and without the multiplier-overflow
    // test (encode_values); the tested form only when S_enc makes it possible
    auto main_loop = [&](auto guard) {
        constexpr bool G = decltype(guard)::value;
        for (; b < a.total; b += stride) {
            const uint16_t* src = a.x + (int64_t)r * a.ld_x + (int64_t)j * 16;
            uint4 u0 = ld_nc_v4(src), u1 = ld_nc_v4(src + 8);
            if constexpr (kRHT) {
                u0.x ^= a.sg.row[0], u0.y ^= a.sg.row[1], u0.z ^= a.sg.row[2], u0.w ^= a.sg.row[3];
                u1.x ^= a.sg.row[4], u1.y ^= a.sg.row[5], u1.z ^= a.sg.row[6], u1.w ^= a.sg.row[7];
            }
            float t[16] = {bf16lo(u0.x), bf16hi(u0.x), bf16lo(u0.y), bf16hi(u0.y), bf16lo(u0.z), bf16hi(u0.z),
                           bf16lo(u0.w), bf16hi(u0.w), bf16lo(u1.x), bf16hi(u1.x), bf16lo(u1.y), bf16hi(u1.y),
                           bf16lo(u1.z), bf16hi(u1.z), bf16lo(u1.w), bf16hi(u1.w)};
            if constexpr (kRHT) {
                rht16_unscaled_packed(t, 0u);   // signs flipped above; the 1/4 comes below
                if (P == Pass::kEncode && !fold) scale16(t, 0.25f);
            }
            float amax_b = 0.0f;
    #pragma unroll
            for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(t[i]));
            if constexpr (P == Pass::kAmax) {
                local_max = fmaxf(local_max, amax_b);
            } else {
                if (fold) amax_b = __fmul_rn(amax_b, 0.25f);
                float r_b;
                uint2 q;   // with 4/6 scales and RNE, the chosen candidate's codes
                const uint32_t sc =
                    kS46 ? block_scale_46<G>(t, amax_b, ts.s_enc, s_mult, rb_table, &r_b, kSR ? nullptr : &q)
                          : block_scale_tab(amax_b, ts.s_enc, rb_table, &r_b);
                const uint64_t idx = (uint64_t)r * ((uint64_t)a.bpr * 16u) + (uint64_t)j * 16u;
                if (kSR || !kS46) q = encode16<kSR, G>(t, r_b, sc, s_mult, keys, a.stream, idx);
                put_codes(a.out, (int64_t)r, (int64_t)j * 8, q);
                put_scales(a.out, scale_offset(r, j, a.out.s4), (uint8_t)sc);
            }
            j += stride_j;
            r += stride_r;
            if (j >= a.bpr) {
                j -= a.bpr;
                ++r;
            }
        }
    };
    if (P == Pass::kEncode && multiplier_may_overflow(ts.s_enc))
        main_loop(std::true_type{});
    else
        main_loop(std::false_type{});
    if constexpr (P == Pass::kAmax) {
        if constexpr (kRHT) local_max = __fmul_rn(local_max, 0.25f);
        block_max_store(local_max, a.partials_out, red);
    }
}

// ----------------------------------------------------------- col-wise -----
struct ColArgs {
    const uint16_t* x;
    int64_t ld_x;
    uint32_t rows, cols;
    uint32_t tiles_r, tiles_c;   // tiles of 128 rows x 64 columns
    Target out;                  // logical [cols][rows]
    Target out2;                 // 16x16 only: the row-wise orientation
    bool emit_col, emit_row;     // 16x16 only
    const float* partials_in;
    int n_partials;
    float* partials_out;
    float* partials_out_plain;   // kAmax with kDual: max |x| before the RHT
    uint32_t mask;
    RhtSigns sg;                 // the mask's sign flips as XOR words
    PhiloxKeys keys;             // SR round keys of the seed
    uint64_t stream;
};

// One warp covers 16 rows x 64 columns (lane = 2 adjacent columns, so each
// load instruction reads 128 contiguous bytes); a CTA of 8 warps covers a
// 128 x 64 tile.  Each thread owns two column blocks of 16 rows.  kDual (amax
// pass with RHT only) also takes the plain max |x| for a row-wise operand
// quantized without RHT from the same input, so one read serves both.
template <Pass P, bool kRHT, bool kSR, bool kDual = false>
__global__ void __launch_bounds__(kThreads) colwise_kernel(const ColArgs a) {
    __shared__ float red[32];
    __shared__ float rb_table[128];
    TensorScale ts{1.0f, 1.0f};
    bool fold = false;   // the RHT's 1/4 lives in the multipliers (rht_quarter_foldable)
    if constexpr (P == Pass::kEncode) {
        ts = load_tensor_scale(a.partials_in, a.n_partials, red, a.out, nullptr);
        if constexpr (kRHT) fold = rht_quarter_foldable(ts.s_enc);
        fill_rb_table(rb_table, ts.s_enc, fold ? 0.25f : 1.0f);
        __syncthreads();
    }
    const float s_mult = fold ? __fmul_rn(ts.s_enc, 0.25f) : ts.s_enc;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t ntiles = a.tiles_r * a.tiles_c;
    float local_max = 0.0f, plain_max = 0.0f;
    const PhiloxKeys& keys = a.keys;   // SR round keys, formed by the host
    // the main loop, instantiated with and without the multiplier-overflow
    // test (encode_values); the tested form only when S_enc makes it possible
    auto main_loop = [&](auto guard) {
        constexpr bool G = decltype(guard)::value;
        for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const uint32_t tr = tile % a.tiles_r, tc = tile / a.tiles_r;
            const uint32_t r0 = tr * 128u + warp * 16u, c = tc * 64u + lane * 2u;
            if (r0 >= a.rows || c >= a.cols) continue;
            const uint16_t* src = a.x + (int64_t)r0 * a.ld_x + c;
            float t0[16], t1[16];
    #pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t w = ld_nc_u32(src + (int64_t)i * a.ld_x) ^ (kRHT ? a.sg.col[i] : 0u);
                t0[i] = bf16lo(w);
                t1[i] = bf16hi(w);
            }
            if constexpr (kDual) {
    #pragma unroll
                for (int i = 0; i < 16; ++i) plain_max = fmaxf(plain_max, fmaxf(fabsf(t0[i]), fabsf(t1[i])));
            }
            if constexpr (kRHT) {
                rht16_unscaled_x2(t0, t1, 0u);   // signs flipped at the load; the 1/4 comes below
                if (P == Pass::kEncode && !fold) {
                    scale16(t0, 0.25f);
                    scale16(t1, 0.25f);
                }
            }
            float m0 = 0.0f, m1 = 0.0f;
    #pragma unroll
            for (int i = 0; i < 16; ++i) {
                m0 = fmaxf(m0, fabsf(t0[i]));
                m1 = fmaxf(m1, fabsf(t1[i]));
            }
            if constexpr (P == Pass::kAmax) {
                local_max = fmaxf(local_max, fmaxf(m0, m1));
            } else {
                if (fold) {
                    m0 = __fmul_rn(m0, 0.25f);
                    m1 = __fmul_rn(m1, 0.25f);
                }
                float rb0, rb1;
                const uint32_t sc0 = block_scale_tab(m0, ts.s_enc, rb_table, &rb0);
                const uint32_t sc1 = block_scale_tab(m1, ts.s_enc, rb_table, &rb1);
                const uint2 q0 = encode16<kSR, G>(t0, rb0, sc0, s_mult, keys, a.stream, (uint64_t)c * a.rows + r0);
                const uint2 q1 = encode16<kSR, G>(t1, rb1, sc1, s_mult, keys, a.stream, (uint64_t)(c + 1) * a.rows + r0);
                put_codes(a.out, (int64_t)c, (int64_t)(r0 / 2), q0);
                put_codes(a.out, (int64_t)(c + 1), (int64_t)(r0 / 2), q1);
                put_scales(a.out, scale_offset(c, r0 / 16, a.out.s4), (uint8_t)sc0);
                put_scales(a.out, scale_offset(c + 1, r0 / 16, a.out.s4), (uint8_t)sc1);
            }
        }
    };
    if (P == Pass::kEncode && multiplier_may_overflow(ts.s_enc))
        main_loop(std::true_type{});
    else
        main_loop(std::false_type{});
    if constexpr (P == Pass::kAmax) {
        if constexpr (kRHT) local_max = __fmul_rn(local_max, 0.25f);
        block_max_store(local_max, a.partials_out, red);
        if constexpr (kDual) {
            __syncthreads();
            block_max_store(plain_max, a.partials_out_plain, red);
        }
    }
}

// --------------------------------------------- Wgrad re-quantization -----
// Q_16x1(H^T Q_1x16(X)) ("Full-Stack FP4", Sec. 3.2 Eq. (2)): the forward's
// row-wise operand of X is dequantized (RN(RN(e2m1 * s_b) * s_g); the first
// product is exact), rotated along its rows and quantized col-wise, so Wgrad
// sees the same quantized activations as Fprop.  Thread layout of
// colwise_kernel: lane = 2 columns x 16 rows (one code byte per row), a warp
// 16 rows x 64 columns, a CTA 128 x 64.
struct RequantArgs {
    const uint8_t* in_codes;     // [rows][in_ld] bytes
    int64_t in_ld;
    const uint8_t* in_scales;    // tile layout of a [rows][cols] operand
    uint32_t in_s4;
    const float* in_sg;
    uint32_t rows, cols;
    uint32_t tiles_r, tiles_c;   // tiles of 128 rows x 64 columns
    Target out;                  // logical [cols][rows]
    const float* partials_in;
    int n_partials;
    float* partials_out;
    uint32_t mask;
    uint32_t sgf[16];            // row i's sign flip of D as an XOR word on a binary32 (bit i of the mask)
    PhiloxKeys keys;             // SR round keys of the seed
    uint64_t stream;
};

template <Pass P, bool kSR>
__global__ void __launch_bounds__(kThreads) requant_kernel(const RequantArgs a) {
    __shared__ float red[32];
    __shared__ float rb_table[128];
    __shared__ float sb_tab[128];     // E4M3 scale code -> value
    __shared__ float2 g_tab[256];     // code byte -> its two E2M1 values (low nibble first)
    static_assert(kThreads >= 256, "one table entry per thread");
    {
        float lo, hi;
        e2m1_decode_byte(threadIdx.x, lo, hi);
        g_tab[threadIdx.x] = make_float2(lo, hi);
        if (threadIdx.x < 128) sb_tab[threadIdx.x] = e4m3_decode(threadIdx.x);
    }
    const float sg = *a.in_sg;
    // The RHT's 1/4 may go into the multipliers (as in the bf16 quantizers)
    // when every value t / 4 is exact: with s_g >= 2^-114 every nonzero input
    // RN(RN(e2m1 s_b) s_g) is at least 2^-10 s_g >= 2^-124, so the inputs and
    // every butterfly value are multiples of 2^-147.
    const bool fold_in = sg >= 0x1p-114f;
    TensorScale ts{1.0f, 1.0f};
    bool fold = false;
    if constexpr (P == Pass::kEncode) {
        ts = load_tensor_scale(a.partials_in, a.n_partials, red, a.out, nullptr);
        fold = fold_in && rht_quarter_foldable(ts.s_enc);
        fill_rb_table(rb_table, ts.s_enc, fold ? 0.25f : 1.0f);
    } else {
        fold = fold_in;
    }
    __syncthreads();
    // the values' factor S_enc (with the RHT's 1/4 when it is folded)
    const float s_mult = fold ? __fmul_rn(ts.s_enc, 0.25f) : ts.s_enc;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t ntiles = a.tiles_r * a.tiles_c;
    float local_max = 0.0f;
    const PhiloxKeys& keys = a.keys;
    // the main loop, instantiated with and without the multiplier-overflow
    // test (encode_values); the tested form only when S_enc makes it possible
    auto main_loop = [&](auto guard) {
        constexpr bool G = decltype(guard)::value;
        for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const uint32_t tr = tile % a.tiles_r, tc = tile / a.tiles_r;
            const uint32_t r0 = tr * 128u + warp * 16u, c = tc * 64u + lane * 2u;
            if (r0 >= a.rows || c >= a.cols) continue;
            // rows r0 .. r0+15 of one 32-row quadrant: their scales are 16 bytes apart
            const uint8_t* srow = a.in_scales + scale_offset(r0, c / 16, a.in_s4);
            const uint8_t* crow = a.in_codes + (int64_t)r0 * a.in_ld + c / 2;
            float t0[16], t1[16];
    #pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 g = g_tab[__ldg(crow + (int64_t)i * a.in_ld)];
                // D's sign flip of row i on its scale: RN(RN(g (-s_b)) s_g) = -RN(RN(g s_b) s_g)
                const float sb = __uint_as_float(__float_as_uint(sb_tab[__ldg(srow + 16 * i) & 0x7Fu]) ^ a.sgf[i]);
                t0[i] = __fmul_rn(__fmul_rn(g.x, sb), sg);
                t1[i] = __fmul_rn(__fmul_rn(g.y, sb), sg);
            }
            rht16_unscaled_x2(t0, t1, 0u);   // signs flipped above
            if (!fold) {
                scale16(t0, 0.25f);
                scale16(t1, 0.25f);
            }
            float m0 = 0.0f, m1 = 0.0f;
    #pragma unroll
            for (int i = 0; i < 16; ++i) {
                m0 = fmaxf(m0, fabsf(t0[i]));
                m1 = fmaxf(m1, fabsf(t1[i]));
            }
            if (P == Pass::kEncode && fold) {
                m0 = __fmul_rn(m0, 0.25f);
                m1 = __fmul_rn(m1, 0.25f);
            }
            if constexpr (P == Pass::kAmax) {
                local_max = fmaxf(local_max, fmaxf(m0, m1));
            } else {
                float rb0, rb1;
                const uint32_t sc0 = block_scale_tab(m0, ts.s_enc, rb_table, &rb0);
                const uint32_t sc1 = block_scale_tab(m1, ts.s_enc, rb_table, &rb1);
                const uint2 q0 = encode16<kSR, G>(t0, rb0, sc0, s_mult, keys, a.stream, (uint64_t)c * a.rows + r0);
                const uint2 q1 = encode16<kSR, G>(t1, rb1, sc1, s_mult, keys, a.stream, (uint64_t)(c + 1) * a.rows + r0);
                put_codes(a.out, (int64_t)c, (int64_t)(r0 / 2), q0);
                put_codes(a.out, (int64_t)(c + 1), (int64_t)(r0 / 2), q1);
                put_scales(a.out, scale_offset(c, r0 / 16, a.out.s4), (uint8_t)sc0);
                put_scales(a.out, scale_offset(c + 1, r0 / 16, a.out.s4), (uint8_t)sc1);
            }
        }
    };
    if (P == Pass::kEncode && multiplier_may_overflow(ts.s_enc))
        main_loop(std::true_type{});
    else
        main_loop(std::false_type{});
    if constexpr (P == Pass::kAmax) {
        if (fold) local_max = __fmul_rn(local_max, 0.25f);
        block_max_store(local_max, a.partials_out, red);
    }
}

// -------------------------------------------------------------- 16x16 -----
__device__ __forceinline__ uint32_t nibble(uint2 q, int i) {
    return ((i < 8 ? q.x : q.y) >> (4 * (i & 7))) & 0xFu;
}

// Same thread layout as colwise_kernel; the 8 lanes that share a 16x16 tile
// reduce its amax by shuffles.  Emits the row-wise codes (out2), the
// transposed codes (out), or both; both come from the same encode of each
// element, so the col-wise codes are the exact transpose of the row-wise ones.
template <bool kSR>
__global__ void __launch_bounds__(kThreads) tile2d_kernel(const ColArgs a) {
    __shared__ float red[32];
    __shared__ float rb_table[128];
    const TensorScale ts =
        load_tensor_scale(a.partials_in, a.n_partials, red, a.emit_col ? a.out : a.out2,
                          (a.emit_col && a.emit_row) ? &a.out2 : nullptr);
    fill_rb_table(rb_table, ts.s_enc);
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t ntiles = a.tiles_r * a.tiles_c;
    const PhiloxKeys& keys = a.keys;   // SR round keys, formed by the host
    // the main loop, instantiated with and without the multiplier-overflow
    // test (encode_values); the tested form only when S_enc makes it possible
    auto main_loop = [&](auto guard) {
        constexpr bool G = decltype(guard)::value;
        for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const uint32_t tr = tile % a.tiles_r, tc = tile / a.tiles_r;
            const uint32_t r0 = tr * 128u + warp * 16u, c = tc * 64u + lane * 2u;
            // rows % 16 == 0 and cols % 16 == 0: the 8 lanes of a tile agree on this
            const bool valid = (r0 < a.rows) && (c < a.cols);
            float t0[16], t1[16];
            float m = 0.0f;
            if (valid) {
                const uint16_t* src = a.x + (int64_t)r0 * a.ld_x + c;
    #pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t w = ld_nc_u32(src + (int64_t)i * a.ld_x);
                    t0[i] = bf16lo(w);
                    t1[i] = bf16hi(w);
                    m = fmaxf(m, fmaxf(fabsf(t0[i]), fabsf(t1[i])));
                }
            }
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            if (!valid) continue;
            float r_b;
            const uint32_t sc = block_scale_tab(m, ts.s_enc, rb_table, &r_b);
            uint2 q0, q1;
            encode_values<16, G>(t0, r_b, sc, ts.s_enc, t0);
            encode_values<16, G>(t1, r_b, sc, ts.s_enc, t1);
            if constexpr (!kSR) {
                q0 = make_uint2(e2m1_rne_x8(t0), e2m1_rne_x8(t0 + 8));
                q1 = make_uint2(e2m1_rne_x8(t1), e2m1_rne_x8(t1 + 8));
            } else {
                float g0[16], g1[16];
    #pragma unroll
                for (int i = 0; i < 16; ++i) {
                    // SR index: the row-wise index of x, shared by both orientations
                    const uint64_t idx = (uint64_t)(r0 + i) * a.cols + c;     // even: c and c+1 share a word
                    const uint4 w = sr_words4(keys, a.stream, idx >> 3);
                    const uint32_t sel = (uint32_t)(idx >> 1) & 3u;
                    const uint32_t word = sel == 0 ? w.x : (sel == 1 ? w.y : (sel == 2 ? w.z : w.w));
                    g0[i] = e2m1_sr_grid(t0[i], sr_addend_lo(word));
                    g1[i] = e2m1_sr_grid(t1[i], sr_addend_hi(word));
                }
                q0 = make_uint2(e2m1_rne_x8(g0), e2m1_rne_x8(g0 + 8));
                q1 = make_uint2(e2m1_rne_x8(g1), e2m1_rne_x8(g1 + 8));
            }
            if (a.emit_col) {
                put_codes(a.out, (int64_t)c, (int64_t)(r0 / 2), q0);
                put_codes(a.out, (int64_t)(c + 1), (int64_t)(r0 / 2), q1);
                put_scales(a.out, scale_offset(c, r0 / 16, a.out.s4), (uint8_t)sc);
                put_scales(a.out, scale_offset(c + 1, r0 / 16, a.out.s4), (uint8_t)sc);
            }
            if (a.emit_row) {
    #pragma unroll
                for (int i = 0; i < 16; ++i) {
                    put_codes(a.out2, (int64_t)(r0 + i), (int64_t)(c / 2),
                              (uint8_t)(nibble(q0, i) | (nibble(q1, i) << 4)));
                    if ((lane & 7u) == 0) put_scales(a.out2, scale_offset(r0 + i, c / 16, a.out2.s4), (uint8_t)sc);
                }
            }
        }
    };
    if (multiplier_may_overflow(ts.s_enc))
        main_loop(std::true_type{});
    else
        main_loop(std::false_type{});
}

// ------------------------------------------- row + col-RHT pair encode -----
// The encode pass of nvfp4_quantize_row_col_rht in one read of x: each warp
// takes 16-row x 64-column slices of x by TMA (128-byte swizzle, two slots per
// warp so the next slice is in flight while this one is encoded), four of them
// down its 64 rows of a 512-row CTA tile, and encodes every element twice from
// shared memory:
//   col-wise with RHT: lane = 2 columns x 16 rows (as colwise_kernel); the
//   four slices' codes of a column (32 bytes) and scales (4 bytes) are kept
//   in registers and stored together after the fourth;
//   row-wise without RHT: lane = 2 row blocks of 16 (row = lane / 2), 16
//   bytes of codes and 2 scale bytes per lane.
struct PairArgs {
    uint32_t rows, cols;
    uint32_t tiles_r, tiles_c;   // kTileRows-row x 64-column CTA tiles
    Target row, col;
    const float* part_plain;
    const float* part_rht;       // the col-wise operand's partials (with or without RHT)
    int n_partials;              // partials of part_plain
    int n_partials_col;          // partials of part_rht
    bool emit_row, emit_col;
    uint32_t mask;
    RhtSigns sg;                 // the mask's sign flips as XOR words
    PhiloxKeys keys;             // SR round keys of the seed
    uint64_t stream_row, stream_col;
    float* part_out_row;         // amax only: one partial per CTA of each orientation
    float* part_out_col;
};

constexpr int kPairSlots = 2;
constexpr uint32_t kSliceBytes = 16 * 128;   // 16 rows x 64 bf16
// Each warp takes 64 rows (four 16-row slices) of a 512-row x 64-column CTA
// tile, so that the col-wise codes of a column (32 bytes) and its four block
// scales (4 bytes) leave in one store each, whole sectors, instead of 8-byte
// pieces that four warps would each write at different times.
constexpr uint32_t kWarpRows = 64;
constexpr uint32_t kTileRows = (kThreads / 32) * kWarpRows;

// Col-wise codes and scales of columns c, c + 1 over the warp's 64 rows from
// row rb: q0[s], q1[s] the codes of 16-row slice s, sc0, sc1 the four scale
// bytes (slice s in byte s).  Only the slices below `rows` are written.
__device__ __forceinline__ void store_col64(const Target& t, uint32_t c, uint32_t rb, uint32_t rows,
                                            const uint2* q0, const uint2* q1, uint32_t sc0, uint32_t sc1) {
    const int64_t off = rb / 2;
    const uint32_t nv = (rows - rb) / 16u;
    if (nv >= 4u) {
        put_codes(t, (int64_t)c, off, make_uint4(q0[0].x, q0[0].y, q0[1].x, q0[1].y));
        put_codes(t, (int64_t)c, off + 16, make_uint4(q0[2].x, q0[2].y, q0[3].x, q0[3].y));
        put_codes(t, (int64_t)(c + 1), off, make_uint4(q1[0].x, q1[0].y, q1[1].x, q1[1].y));
        put_codes(t, (int64_t)(c + 1), off + 16, make_uint4(q1[2].x, q1[2].y, q1[3].x, q1[3].y));
        put_scales(t, scale_offset(c, rb / 16u, t.s4), sc0);
        put_scales(t, scale_offset(c + 1, rb / 16u, t.s4), sc1);
    } else {
#pragma unroll
        for (uint32_t s = 0; s < 3u; ++s) {
            if (s < nv) {
                put_codes(t, (int64_t)c, off + 8 * s, q0[s]);
                put_codes(t, (int64_t)(c + 1), off + 8 * s, q1[s]);
                put_scales(t, scale_offset(c, rb / 16u + s, t.s4), (uint8_t)(sc0 >> (8 * s)));
                put_scales(t, scale_offset(c + 1, rb / 16u + s, t.s4), (uint8_t)(sc1 >> (8 * s)));
            }
        }
    }
}

// kColRHT: the col-wise operand gets the RHT (else none); kRowRHT: the
// row-wise operand gets it too (along its rows; both orientations of an RHT
// quantize call).  Either orientation may be left out (emit_*).
// kS46: 4/6 adaptive block scales (block_scale_46) in both orientations.
// kAmaxOnly: the amax pass of an RHT call emitting both orientations: no
// encode; each CTA writes the max |value| of each orientation (after its
// transform, the 1/4 included) to part_out_row and part_out_col, from one
// read of x instead of one per orientation.
template <bool kSR, bool kColRHT, bool kS46 = false, bool kRowRHT = false, bool kAmaxOnly = false>
__global__ void __launch_bounds__(kThreads) pair_encode_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                               const PairArgs a) {
    __shared__ float red[32];
    __shared__ float rb_row[128], rb_col[128];
    __shared__ __align__(1024) uint8_t ring[kThreads / 32][kPairSlots][kSliceBytes];
    __shared__ uint64_t full[kThreads / 32][kPairSlots];
    TensorScale ts_row{1.0f, 1.0f}, ts_col{1.0f, 1.0f};
    if (!kAmaxOnly && a.emit_row) ts_row = load_tensor_scale(a.part_plain, a.n_partials, red, a.row, nullptr);
    if (!kAmaxOnly && a.emit_col) ts_col = load_tensor_scale(a.part_rht, a.n_partials_col, red, a.col, nullptr);
    // with S_enc = 1 (amax only) both quarters count as folded: the block
    // maxima below are those of the scaled transform, exactly
    float row_max = 0.0f, col_max = 0.0f;
    // the col-wise RHT's 1/4 lives in its multipliers (rht_quarter_foldable)
    const bool fold = kColRHT && rht_quarter_foldable(ts_col.s_enc);
    const bool fold_row = kRowRHT && rht_quarter_foldable(ts_row.s_enc);
    // the values' factor S_enc per orientation (with the RHT's 1/4 when folded)
    const float s_mult_col = fold ? __fmul_rn(ts_col.s_enc, 0.25f) : ts_col.s_enc;
    const float s_mult_row = fold_row ? __fmul_rn(ts_row.s_enc, 0.25f) : ts_row.s_enc;
    fill_rb_table_at(rb_row, ts_row.s_enc, 0, fold_row ? 0.25f : 1.0f);
    fill_rb_table_at(rb_col, ts_col.s_enc, 128, fold ? 0.25f : 1.0f);
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    if (lane == 0) {
        for (int sl = 0; sl < kPairSlots; ++sl) mbar_init(&full[warp][sl], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const PhiloxKeys& keys = a.keys;   // SR round keys, formed by the host
    const uint32_t ntiles = a.tiles_r * a.tiles_c;
    // this warp's 16-row slice j of the CTA's tiles: tile j / 4, slice j % 4
    // of the warp's 64 rows, if it holds rows
    auto slice_of = [&](uint32_t j, uint32_t& r0, uint32_t& c0) -> bool {
        const uint32_t tile = blockIdx.x + (j >> 2) * gridDim.x;
        if (tile >= ntiles) return false;
        r0 = (tile % a.tiles_r) * kTileRows + warp * kWarpRows + (j & 3u) * 16u;
        c0 = (tile / a.tiles_r) * 64u;
        return r0 < a.rows;
    };
    auto issue = [&](uint32_t j) {
        uint32_t r0, c0;
        if (lane == 0 && slice_of(j, r0, c0)) {
            uint64_t* bar = &full[warp][j % kPairSlots];
            mbar_arrive_expect_tx(bar, kSliceBytes);
            tma_load_2d(ring[warp][j % kPairSlots], &tmap_x, bar, (int32_t)c0, (int32_t)r0);
        }
    };
    const uint32_t kcount = (ntiles > blockIdx.x) ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    uint32_t parity = 0;   // bit s: parity of the next wait on slot s
    // the col-wise codes and scales of the warp's four slices of a tile, slice
    // s in element / byte s, stored once the fourth slice is encoded
    uint2 cq0[4], cq1[4];
    uint32_t cs0 = 0, cs1 = 0;
    for (uint32_t k = 0; k + 1 < (uint32_t)kPairSlots; ++k) issue(k);   // kPairSlots - 1 slices ahead
    // the main loop, instantiated with and without the multiplier-overflow
    // test (encode_values); the tested form only when S_enc makes it possible
    auto main_loop = [&](auto guard) {
        constexpr bool G = decltype(guard)::value;
        for (uint32_t j = 0; j < 4u * kcount; ++j) {
            __syncwarp();   // every lane is done with the slot the next copy fills
            issue(j + kPairSlots - 1);
            uint32_t r0, c0;
            uint2 q0 = make_uint2(0u, 0u), q1 = make_uint2(0u, 0u);
            uint32_t sc0 = 0, sc1 = 0;
            if (slice_of(j, r0, c0)) {
            const uint32_t sl = j % kPairSlots;
            if (!mbar_wait(&full[warp][sl], (parity >> sl) & 1u, 2000000000ull)) {
                // a copy that never landed: let the ones issued after it land
                // before this CTA can exit, then stop
                for (uint32_t k = 1; k < (uint32_t)kPairSlots; ++k) {
                    uint32_t r1, c1;
                    const uint32_t s2 = (j + k) % kPairSlots;
                    if (slice_of(j + k, r1, c1))
                        (void)mbar_wait(&full[warp][s2], (parity >> s2) & 1u, 2000000000ull);
                }
                break;
            }
            parity ^= 1u << sl;
            const uint8_t* src = ring[warp][sl];

            // ---- col-wise with RHT: lane = columns c0 + 2 lane, c0 + 2 lane + 1
            {
                const uint32_t c = c0 + lane * 2u;
                float t0[16], t1[16];
    #pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t off = (uint32_t)i * 128u + (((lane >> 2) ^ (uint32_t)(i & 7)) << 4) + (lane & 3u) * 4u;
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(src + off) ^ (kColRHT ? a.sg.col[i] : 0u);
                    t0[i] = bf16lo(w);
                    t1[i] = bf16hi(w);
                }
                if (a.emit_col && c < a.cols) {
                    if constexpr (kColRHT) {
                        rht16_unscaled_x2(t0, t1, 0u);   // signs flipped at the load; the 1/4 comes below
                        if (!fold) {
                            scale16(t0, 0.25f);
                            scale16(t1, 0.25f);
                        }
                    }
                    float m0 = 0.0f, m1 = 0.0f;
    #pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        m0 = fmaxf(m0, fabsf(t0[i]));
                        m1 = fmaxf(m1, fabsf(t1[i]));
                    }
                    if (fold) {
                        m0 = __fmul_rn(m0, 0.25f);
                        m1 = __fmul_rn(m1, 0.25f);
                    }
                    if constexpr (kAmaxOnly) {
                        col_max = fmaxf(col_max, fmaxf(m0, m1));
                    } else {
                    float rb0, rb1;
                    if constexpr (kS46) {
                        // with RNE the chosen candidates' codes are the block's codes
                        sc0 = block_scale_46<G>(t0, m0, ts_col.s_enc, s_mult_col, rb_col, &rb0, kSR ? nullptr : &q0);
                        sc1 = block_scale_46<G>(t1, m1, ts_col.s_enc, s_mult_col, rb_col, &rb1, kSR ? nullptr : &q1);
                    } else {
                        sc0 = block_scale_tab(m0, ts_col.s_enc, rb_col, &rb0);
                        sc1 = block_scale_tab(m1, ts_col.s_enc, rb_col, &rb1);
                    }
                    if (kSR || !kS46) {
                        q0 = encode16<kSR, G>(t0, rb0, sc0, s_mult_col, keys, a.stream_col, (uint64_t)c * a.rows + r0);
                        q1 = encode16<kSR, G>(t1, rb1, sc1, s_mult_col, keys, a.stream_col,
                                              (uint64_t)(c + 1) * a.rows + r0);
                    }
                    }
                }
            }
            // ---- row-wise without RHT: lane = row r0 + lane / 2, 32 columns
            {
                const uint32_t i = lane >> 1, h = lane & 1u;
                const uint32_t r = r0 + i, cb = c0 + 32u * h;
                if (a.emit_row && cb < a.cols) {
                    float v[32];
    #pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t off = i * 128u + (((4u * h + (uint32_t)kk) ^ (i & 7u)) << 4);
                        uint4 u = *reinterpret_cast<const uint4*>(src + off);
                        if constexpr (kRowRHT) {
                            const uint32_t s0 = 4u * ((uint32_t)kk & 1u);
                            u.x ^= a.sg.row[s0], u.y ^= a.sg.row[s0 + 1], u.z ^= a.sg.row[s0 + 2], u.w ^= a.sg.row[s0 + 3];
                        }
                        v[8 * kk + 0] = bf16lo(u.x);
                        v[8 * kk + 1] = bf16hi(u.x);
                        v[8 * kk + 2] = bf16lo(u.y);
                        v[8 * kk + 3] = bf16hi(u.y);
                        v[8 * kk + 4] = bf16lo(u.z);
                        v[8 * kk + 5] = bf16hi(u.z);
                        v[8 * kk + 6] = bf16lo(u.w);
                        v[8 * kk + 7] = bf16hi(u.w);
                    }
                    if constexpr (kRowRHT) {
                        rht16_unscaled_x2(v, v + 16, 0u);   // signs flipped at the load; the 1/4 comes below
                        if (!fold_row) {
                            scale16(v, 0.25f);
                            scale16(v + 16, 0.25f);
                        }
                    }
                    const bool two = cb + 16u < a.cols;
                    uint2 q[2];
                    uint32_t sc[2];
    #pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        float m = 0.0f;
    #pragma unroll
                        for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(v[16 * jj + e]));
                        if (fold_row) m = __fmul_rn(m, 0.25f);
                        if constexpr (kAmaxOnly) {
                            row_max = fmaxf(row_max, m);
                            continue;
                        }
                        float rb;
                        sc[jj] = kS46 ? block_scale_46<G>(v + 16 * jj, m, ts_row.s_enc, s_mult_row, rb_row, &rb,
                                                          kSR ? nullptr : &q[jj])
                                       : block_scale_tab(m, ts_row.s_enc, rb_row, &rb);
                        if (kSR || !kS46)
                            q[jj] = encode16<kSR, G>(v + 16 * jj, rb, sc[jj], s_mult_row, keys, a.stream_row,
                                                  (uint64_t)r * a.cols + cb + 16u * (uint32_t)jj);
                    }
                    const uint32_t j0 = cb / 16u;
                    if (kAmaxOnly) {
                    } else if (two) {
                        put_codes(a.row, (int64_t)r, (int64_t)(cb / 2), make_uint4(q[0].x, q[0].y, q[1].x, q[1].y));
                        put_scales(a.row, scale_offset(r, j0, a.row.s4), (uint16_t)(sc[0] | (sc[1] << 8)));
                    } else {
                        put_codes(a.row, (int64_t)r, (int64_t)(cb / 2), q[0]);
                        put_scales(a.row, scale_offset(r, j0, a.row.s4), (uint8_t)sc[0]);
                    }
                }
            }
            }
            if constexpr (kAmaxOnly) continue;
            // slice j % 4 joins the warp's col-wise codes; after the fourth, they
            // go out as whole sectors
            cq0[0] = cq0[1], cq0[1] = cq0[2], cq0[2] = cq0[3], cq0[3] = q0;
            cq1[0] = cq1[1], cq1[1] = cq1[2], cq1[2] = cq1[3], cq1[3] = q1;
            cs0 = (cs0 >> 8) | (sc0 << 24);
            cs1 = (cs1 >> 8) | (sc1 << 24);
            if ((j & 3u) == 3u && a.emit_col) {
                const uint32_t tile = blockIdx.x + (j >> 2) * gridDim.x;
                const uint32_t rb = (tile % a.tiles_r) * kTileRows + warp * kWarpRows;
                const uint32_t c = (tile / a.tiles_r) * 64u + lane * 2u;
                if (tile < ntiles && rb < a.rows && c < a.cols) store_col64(a.col, c, rb, a.rows, cq0, cq1, cs0, cs1);
            }
        }
    };
    if (multiplier_may_overflow(ts_row.s_enc) || multiplier_may_overflow(ts_col.s_enc))
        main_loop(std::true_type{});
    else
        main_loop(std::false_type{});
    if constexpr (kAmaxOnly) {
        block_max_store(row_max, a.part_out_row, red);
        __syncthreads();
        block_max_store(col_max, a.part_out_col, red);
    }
}

// ------------------------------------------------ 16x16, RNE, via TMA -----
// The RNE 16x16 encode from TMA-staged 16-row x 64-column slices (as
// pair_kernel): the col-wise codes come from the col layout (lane = 2 columns
// x 16 rows, tile amax by three shuffles), the row-wise codes from the row
// layout (lane = half a row), each with 16-byte code stores; both encode
// every element with the tile's r_b, so the two are exact transposes.
struct Tile2dArgs {
    uint32_t rows, cols;
    uint32_t tiles_r, tiles_c;   // kTileRows-row x 64-column CTA tiles
    Target row, col;
    bool emit_row, emit_col;
    const float* partials;
    int n_partials;
};

__global__ void __launch_bounds__(kThreads) tile2d_rne_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                              const Tile2dArgs a) {
    __shared__ float red[32];
    __shared__ float rb_tab[128];
    __shared__ __align__(1024) uint8_t ring[kThreads / 32][kPairSlots][kSliceBytes];
    __shared__ uint64_t full[kThreads / 32][kPairSlots];
    const TensorScale ts = load_tensor_scale(a.partials, a.n_partials, red, a.emit_col ? a.col : a.row,
                                             (a.emit_col && a.emit_row) ? &a.row : nullptr);
    fill_rb_table(rb_tab, ts.s_enc);
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    if (lane == 0) {
        for (int sl = 0; sl < kPairSlots; ++sl) mbar_init(&full[warp][sl], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const uint32_t ntiles = a.tiles_r * a.tiles_c;
    // this warp's 16-row slice j of the CTA's tiles: tile j / 4, slice j % 4
    // of the warp's 64 rows, if it holds rows
    auto slice_of = [&](uint32_t j, uint32_t& r0, uint32_t& c0) -> bool {
        const uint32_t tile = blockIdx.x + (j >> 2) * gridDim.x;
        if (tile >= ntiles) return false;
        r0 = (tile % a.tiles_r) * kTileRows + warp * kWarpRows + (j & 3u) * 16u;
        c0 = (tile / a.tiles_r) * 64u;
        return r0 < a.rows;
    };
    auto issue = [&](uint32_t j) {
        uint32_t r0, c0;
        if (lane == 0 && slice_of(j, r0, c0)) {
            uint64_t* bar = &full[warp][j % kPairSlots];
            mbar_arrive_expect_tx(bar, kSliceBytes);
            tma_load_2d(ring[warp][j % kPairSlots], &tmap_x, bar, (int32_t)c0, (int32_t)r0);
        }
    };
    const uint32_t kcount = (ntiles > blockIdx.x) ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    uint32_t parity = 0;
    // the col-wise codes and scales of the warp's four slices of a tile
    uint2 cq0[4], cq1[4];
    uint32_t cs = 0;
    for (uint32_t k = 0; k + 1 < (uint32_t)kPairSlots; ++k) issue(k);   // kPairSlots - 1 slices ahead
    // the main loop, instantiated with and without the multiplier-overflow
    // test (encode_values); the tested form only when S_enc makes it possible
    auto main_loop = [&](auto guard) {
        constexpr bool G = decltype(guard)::value;
        for (uint32_t j = 0; j < 4u * kcount; ++j) {
            __syncwarp();
            issue(j + kPairSlots - 1);
            uint32_t r0, c0;
            uint2 q0 = make_uint2(0u, 0u), q1 = make_uint2(0u, 0u);
            uint32_t sc = 0;
            if (slice_of(j, r0, c0)) {
            const uint32_t sl = j % kPairSlots;
            if (!mbar_wait(&full[warp][sl], (parity >> sl) & 1u, 2000000000ull)) {
                for (uint32_t k = 1; k < (uint32_t)kPairSlots; ++k) {
                    uint32_t r1, c1;
                    const uint32_t s2 = (j + k) % kPairSlots;
                    if (slice_of(j + k, r1, c1))
                        (void)mbar_wait(&full[warp][s2], (parity >> s2) & 1u, 2000000000ull);
                }
                break;
            }
            parity ^= 1u << sl;
            const uint8_t* src = ring[warp][sl];
            // col layout: tile amax and scale; col-wise codes
            const uint32_t c = c0 + lane * 2u;
            float t0[16], t1[16];
    #pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(
                    src + (uint32_t)i * 128u + (((lane >> 2) ^ (uint32_t)(i & 7)) << 4) + (lane & 3u) * 4u);
                t0[i] = bf16lo(w);
                t1[i] = bf16hi(w);
            }
            float m = 0.0f;
    #pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(fabsf(t0[i]), fabsf(t1[i])));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            float rb;
            sc = block_scale_tab(m, ts.s_enc, rb_tab, &rb);
            if (a.emit_col && c < a.cols) {
                float v0[16], v1[16];
                encode_values<16, G>(t0, rb, sc, ts.s_enc, v0);
                encode_values<16, G>(t1, rb, sc, ts.s_enc, v1);
                q0 = make_uint2(e2m1_rne_x8(v0), e2m1_rne_x8(v0 + 8));
                q1 = make_uint2(e2m1_rne_x8(v1), e2m1_rne_x8(v1 + 8));
            }
            if (a.emit_row) {
                // row layout: row r0 + lane / 2, columns c0 + 32 (lane & 1) .. + 31
                // = tiles 2h and 2h+1 of the slice, whose scales lanes 16h and
                // 16h + 8 hold
                const uint32_t i = lane >> 1, h = lane & 1u;
                const uint32_t r = r0 + i, cb = c0 + 32u * h;
                const float rbt0 = __shfl_sync(0xFFFFFFFFu, rb, 16 * h), rbt1 = __shfl_sync(0xFFFFFFFFu, rb, 16 * h + 8);
                const uint32_t sct0 = __shfl_sync(0xFFFFFFFFu, sc, 16 * h),
                               sct1 = __shfl_sync(0xFFFFFFFFu, sc, 16 * h + 8);
                if (cb < a.cols) {
                    float v[32];
    #pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t off = i * 128u + (((4u * h + (uint32_t)kk) ^ (i & 7u)) << 4);
                        const uint4 u = *reinterpret_cast<const uint4*>(src + off);
                        const float x8[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                                             bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
                        encode_values<8, G>(x8, kk < 2 ? rbt0 : rbt1, kk < 2 ? sct0 : sct1, ts.s_enc, v + 8 * kk);
                    }
                    const uint32_t j0 = cb / 16u;
                    if (cb + 16u < a.cols) {
                        put_codes(a.row, (int64_t)r, (int64_t)(cb / 2),
                                  make_uint4(e2m1_rne_x8(v), e2m1_rne_x8(v + 8), e2m1_rne_x8(v + 16),
                                             e2m1_rne_x8(v + 24)));
                        put_scales(a.row, scale_offset(r, j0, a.row.s4), (uint16_t)(sct0 | (sct1 << 8)));
                    } else {
                        put_codes(a.row, (int64_t)r, (int64_t)(cb / 2), make_uint2(e2m1_rne_x8(v), e2m1_rne_x8(v + 8)));
                        put_scales(a.row, scale_offset(r, j0, a.row.s4), (uint8_t)sct0);
                    }
                }
            }
            }
            // slice j % 4 joins the warp's col-wise codes; after the fourth, they
            // go out as whole sectors (both columns share the tile's scale)
            cq0[0] = cq0[1], cq0[1] = cq0[2], cq0[2] = cq0[3], cq0[3] = q0;
            cq1[0] = cq1[1], cq1[1] = cq1[2], cq1[2] = cq1[3], cq1[3] = q1;
            cs = (cs >> 8) | (sc << 24);
            if ((j & 3u) == 3u && a.emit_col) {
                const uint32_t tile = blockIdx.x + (j >> 2) * gridDim.x;
                const uint32_t rb = (tile % a.tiles_r) * kTileRows + warp * kWarpRows;
                const uint32_t c = (tile / a.tiles_r) * 64u + lane * 2u;
                if (tile < ntiles && rb < a.rows && c < a.cols) store_col64(a.col, c, rb, a.rows, cq0, cq1, cs, cs);
            }
        }
    };
    if (multiplier_may_overflow(ts.s_enc))
        main_loop(std::true_type{});
    else
        main_loop(std::false_type{});
}

// ------------------------------------------------------------- launch -----
template <typename K>
int persistent_grid(K kernel, int64_t work) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t g = (int64_t)per_sm * device_sm_count();
    if (work < g) g = work;
    return g < 1 ? 1 : (int)g;
}

Target make_target(const QuantTarget* q) {
    Target t{};
    if (!q) return t;
    t.codes = q->codes;
    t.ld_codes = q->ld_codes;
    t.scales = q->scales;
    t.s4 = (uint32_t)((q->lcols + 63) / 64);
    t.amax = q->amax;
    t.sg = q->sg;
    t.xc = extent_rows(q->codes, q->lrows, q->ld_codes, (q->lcols + 1) / 2);
    t.xs = extent_of(q->scales, ((q->lrows + 127) / 128) * (int64_t)t.s4 * 512);
    return t;
}

// Zero the padding bytes of a scale buffer (rows past the last 128-row tile
// boundary or scale columns past cols / 16).
cudaError_t clear_scale_padding(const QuantTarget* q, cudaStream_t st) {
    if (!q) return cudaSuccess;
    const int64_t s4 = (q->lcols + 63) / 64, rt = (q->lrows + 127) / 128;
    if ((q->lcols / 16) % 4 != 0) return cudaMemsetAsync(q->scales, 0, (size_t)(rt * s4 * 512), st);
    if (q->lrows % 128 != 0)
        return cudaMemsetAsync(q->scales + (rt - 1) * s4 * 512, 0, (size_t)(s4 * 512), st);
    return cudaSuccess;
}

// Amax pass over x along rows (plain or RHT): returns the grid it used.
template <bool kRHT>
int row_amax(const RowArgs& base, float* partials, cudaStream_t st) {
    RowArgs a = base;
    a.partials_out = partials;
    auto k = rowwise_kernel<Pass::kAmax, kRHT, false>;
    int g = persistent_grid(k, ((int64_t)a.total + kThreads - 1) / kThreads);
    if (g > kMaxAmaxPartials) g = kMaxAmaxPartials;
    k<<<g, kThreads, 0, st>>>(a);
    return g;
}

// Tensor map of x's 16-row x 64-column slices (128-byte swizzle) for the
// slice-staged kernels; no L2 sector promotion (a 256-byte promotion fetched
// the neighbouring 128 bytes again later: 25 % more DRAM reads on a 16x16
// encode).
bool make_slice_map(CUtensorMap* tmap, const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_x * 2u};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t elem[2] = {1, 1};
    return fn(tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The amax pass of an RHT call emitting both orientations, from one read of
// x (pair_encode_kernel<..., kAmaxOnly>): partials of the row-wise operand's
// transform in part_row, of the col-wise one's in part_col.  Returns the
// number of partials of each (the grid), or -1 when the tensor map cannot be
// made.
int launch_pair_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, uint32_t sign_mask,
                     float* part_row, float* part_col, cudaStream_t st) {
    CUtensorMap tmap;
    if (!make_slice_map(&tmap, x, rows, cols, ld_x)) return -1;
    PairArgs pa{};
    pa.rows = (uint32_t)rows;
    pa.cols = (uint32_t)cols;
    pa.tiles_r = (uint32_t)((rows + kTileRows - 1) / kTileRows);
    pa.tiles_c = (uint32_t)((cols + 63) / 64);
    pa.emit_row = pa.emit_col = true;
    pa.mask = sign_mask;
    pa.sg = rht_signs(sign_mask);
    pa.part_out_row = part_row;
    pa.part_out_col = part_col;
    auto k = pair_encode_kernel<false, true, false, true, true>;
    int g = persistent_grid(k, (int64_t)pa.tiles_r * pa.tiles_c);
    if (g > kMaxAmaxPartials) g = kMaxAmaxPartials;
    k<<<g, kThreads, 0, st>>>(tmap, pa);
    return g;
}

// The slice-staged encode (pair_encode_kernel): optional row-wise operand
// without RHT and optional col-wise operand with or without RHT.
cudaError_t launch_pair_encode(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool sr, bool col_rht,
                               uint32_t sign_mask, uint64_t seed, uint64_t stream_row, uint64_t stream_col,
                               const QuantTarget* row, const QuantTarget* col, const float* part_row,
                               const float* part_col, int n_partials, bool s46, cudaStream_t st,
                               bool row_rht = false, int n_partials_col = -1) {
    CUtensorMap tmap;
    if (!make_slice_map(&tmap, x, rows, cols, ld_x)) return cudaErrorInvalidValue;
    PairArgs pa{};
    pa.rows = (uint32_t)rows;
    pa.cols = (uint32_t)cols;
    pa.tiles_r = (uint32_t)((rows + kTileRows - 1) / kTileRows);
    pa.tiles_c = (uint32_t)((cols + 63) / 64);
    pa.row = make_target(row);
    pa.col = make_target(col);
    pa.emit_row = row != nullptr;
    pa.emit_col = col != nullptr;
    pa.part_plain = part_row;
    pa.part_rht = part_col;
    pa.n_partials = n_partials;
    pa.n_partials_col = n_partials_col < 0 ? n_partials : n_partials_col;
    pa.mask = sign_mask;
    pa.sg = rht_signs(sign_mask);
    pa.keys = philox_keys(seed);
    pa.stream_row = stream_row;
    pa.stream_col = stream_col;
    const int64_t ntiles = (int64_t)pa.tiles_r * pa.tiles_c;
    auto launch = [&](auto k) { k<<<persistent_grid(k, ntiles), kThreads, 0, st>>>(tmap, pa); };
    if (row_rht) {   // both orientations with the RHT (col_rht is set too)
        if (s46 && sr) launch(pair_encode_kernel<true, true, true, true>);
        else if (s46) launch(pair_encode_kernel<false, true, true, true>);
        else if (sr) launch(pair_encode_kernel<true, true, false, true>);
        else launch(pair_encode_kernel<false, true, false, true>);
        return cudaGetLastError();
    }
    if (s46) {
        if (sr && col_rht) launch(pair_encode_kernel<true, true, true>);
        else if (col_rht) launch(pair_encode_kernel<false, true, true>);
        else if (sr) launch(pair_encode_kernel<true, false, true>);
        else launch(pair_encode_kernel<false, false, true>);
    } else {
        if (sr && col_rht) launch(pair_encode_kernel<true, true>);
        else if (col_rht) launch(pair_encode_kernel<false, true>);
        else if (sr) launch(pair_encode_kernel<true, false>);
        else launch(pair_encode_kernel<false, false>);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool scale_2d, bool scale_46,
                            bool sr,
                            bool rht, uint32_t sign_mask, uint64_t seed, uint64_t stream_id,
                            const QuantTarget* row, const QuantTarget* col, float* workspace,
                            cudaStream_t st) {
    cudaError_t err;
    if ((err = clear_scale_padding(row, st)) != cudaSuccess) return err;
    if ((err = clear_scale_padding(col, st)) != cudaSuccess) return err;

    RowArgs ra{};
    ra.x = x;
    ra.ld_x = ld_x;
    ra.bpr = (uint32_t)(cols / 16);
    ra.total = (uint32_t)(rows * (cols / 16));
    ra.mask = sign_mask;
    ra.sg = rht_signs(sign_mask);
    ra.keys = philox_keys(seed);
    ra.stream = stream_id;

    ColArgs ca{};
    ca.x = x;
    ca.ld_x = ld_x;
    ca.rows = (uint32_t)rows;
    ca.cols = (uint32_t)cols;
    ca.tiles_r = (uint32_t)((rows + 127) / 128);
    ca.tiles_c = (uint32_t)((cols + 63) / 64);
    ca.mask = sign_mask;
    ca.sg = rht_signs(sign_mask);
    ca.keys = philox_keys(seed);
    ca.stream = stream_id;
    const int64_t ntiles = (int64_t)ca.tiles_r * ca.tiles_c;

    float* part_a = workspace;
    float* part_b = workspace + kMaxAmaxPartials;

    if (scale_2d) {
        ca.partials_in = part_a;
        ca.n_partials = row_amax<false>(ra, part_a, st);
        ca.out = make_target(col);
        ca.out2 = make_target(row);
        ca.emit_col = col != nullptr;
        ca.emit_row = row != nullptr;
        if (sr) {
            auto k = tile2d_kernel<true>;
            k<<<persistent_grid(k, ntiles), kThreads, 0, st>>>(ca);
            return cudaGetLastError();
        }
        EncodeTiledFn fn = encode_fn();
        CUtensorMap tmap;
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)ld_x * 2u};
        const cuuint32_t box[2] = {64, 16};
        const cuuint32_t elem[2] = {1, 1};
        if (!fn || fn(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, elem,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        Tile2dArgs ta{};
        ta.rows = (uint32_t)rows;
        ta.cols = (uint32_t)cols;
        ta.tiles_r = (uint32_t)((rows + kTileRows - 1) / kTileRows);
        ta.tiles_c = ca.tiles_c;
        ta.row = make_target(row);
        ta.col = make_target(col);
        ta.emit_row = row != nullptr;
        ta.emit_col = col != nullptr;
        ta.partials = part_a;
        ta.n_partials = ca.n_partials;
        auto k = tile2d_rne_kernel;
        k<<<persistent_grid(k, (int64_t)ta.tiles_r * ta.tiles_c), kThreads, 0, st>>>(tmap, ta);
        return cudaGetLastError();
    }

    int n_row = 0, n_col = 0;
    if (!rht) {
        n_row = n_col = row_amax<false>(ra, part_a, st);
        part_b = part_a;
    } else if (row && col) {
        // both orientations' transforms from one read
        n_row = n_col = launch_pair_amax(x, rows, cols, ld_x, sign_mask, part_a, part_b, st);
        if (n_row < 0) return cudaErrorInvalidValue;
    } else {
        if (row) n_row = row_amax<true>(ra, part_a, st);
        if (col) {
            ColArgs c = ca;
            c.partials_out = part_b;
            auto k = colwise_kernel<Pass::kAmax, true, false>;
            int g = persistent_grid(k, ntiles);
            if (g > kMaxAmaxPartials) g = kMaxAmaxPartials;
            k<<<g, kThreads, 0, st>>>(c);
            n_col = g;
        }
    }

    // row-wise: the thread-per-block kernel, unless a col-wise operand is
    // emitted too (then one slice-staged pass emits both, each orientation
    // with its own tensor scale when the RHT is on)
    const bool joint = row && col;
    if (row && !joint) {
        RowArgs r = ra;
        r.out = make_target(row);
        r.partials_in = part_a;
        r.n_partials = n_row;
        auto launch = [&](auto k) {
            k<<<persistent_grid(k, ((int64_t)r.total + kThreads - 1) / kThreads), kThreads, 0, st>>>(r);
        };
        if (scale_46) {
            if (rht && sr) launch(rowwise_kernel<Pass::kEncode, true, true, true>);
            else if (rht) launch(rowwise_kernel<Pass::kEncode, true, false, true>);
            else if (sr) launch(rowwise_kernel<Pass::kEncode, false, true, true>);
            else launch(rowwise_kernel<Pass::kEncode, false, false, true>);
        } else {
            if (rht && sr) launch(rowwise_kernel<Pass::kEncode, true, true>);
            else if (rht) launch(rowwise_kernel<Pass::kEncode, true, false>);
            else if (sr) launch(rowwise_kernel<Pass::kEncode, false, true>);
            else launch(rowwise_kernel<Pass::kEncode, false, false>);
        }
    }
    if (col)
        return launch_pair_encode(x, rows, cols, ld_x, sr, rht, sign_mask, seed, stream_id, stream_id,
                                  joint ? row : nullptr, col, part_a, part_b, n_row, scale_46, st, joint && rht,
                                  rht ? n_col : n_row);
    return cudaGetLastError();
}

cudaError_t launch_quantize_row_col_rht(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool sr,
                                       uint32_t sign_mask, uint64_t seed, uint64_t stream_row, uint64_t stream_col,
                                       const QuantTarget* row, const QuantTarget* col, float* workspace,
                                       cudaStream_t st) {
    cudaError_t err;
    if ((err = clear_scale_padding(row, st)) != cudaSuccess) return err;
    if ((err = clear_scale_padding(col, st)) != cudaSuccess) return err;
    float* part_plain = workspace;
    float* part_rht = workspace + kMaxAmaxPartials;

    ColArgs ca{};
    ca.x = x;
    ca.ld_x = ld_x;
    ca.rows = (uint32_t)rows;
    ca.cols = (uint32_t)cols;
    ca.tiles_r = (uint32_t)((rows + 127) / 128);
    ca.tiles_c = (uint32_t)((cols + 63) / 64);
    ca.mask = sign_mask;
    ca.sg = rht_signs(sign_mask);
    ca.keys = philox_keys(seed);
    const int64_t ntiles = (int64_t)ca.tiles_r * ca.tiles_c;

    // one amax pass: the RHT amax for the col-wise operand and the plain
    // amax for the row-wise one
    int n = 0;
    {
        ColArgs c = ca;
        c.partials_out = part_rht;
        c.partials_out_plain = part_plain;
        auto k = colwise_kernel<Pass::kAmax, true, false, true>;
        n = persistent_grid(k, ntiles);
        if (n > kMaxAmaxPartials) n = kMaxAmaxPartials;
        k<<<n, kThreads, 0, st>>>(c);
    }
    // one encode pass for both orientations, x staged through TMA
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_x * 2u};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t elem[2] = {1, 1};
    if (fn(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    PairArgs pa{};
    pa.rows = (uint32_t)rows;
    pa.cols = (uint32_t)cols;
    pa.tiles_r = (uint32_t)((rows + kTileRows - 1) / kTileRows);
    pa.tiles_c = ca.tiles_c;
    pa.row = make_target(row);
    pa.col = make_target(col);
    pa.part_plain = part_plain;
    pa.part_rht = part_rht;
    pa.n_partials = n;
    pa.n_partials_col = n;
    pa.emit_row = pa.emit_col = true;
    pa.mask = sign_mask;
    pa.sg = rht_signs(sign_mask);
    pa.keys = philox_keys(seed);
    pa.stream_row = stream_row;
    pa.stream_col = stream_col;
    const int64_t pair_tiles = (int64_t)pa.tiles_r * pa.tiles_c;
    auto launch = [&](auto k) { k<<<persistent_grid(k, pair_tiles), kThreads, 0, st>>>(tmap, pa); };
    if (sr) launch(pair_encode_kernel<true, true>);
    else launch(pair_encode_kernel<false, true>);
    return cudaGetLastError();
}

cudaError_t launch_quantize_row_col_rht_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool sr,
                                             uint32_t sign_mask, uint64_t seed, uint64_t stream_row,
                                             uint64_t stream_col, const float* amax_in, const QuantTarget* row,
                                             const QuantTarget* col, cudaStream_t st) {
    cudaError_t err;
    if ((err = clear_scale_padding(row, st)) != cudaSuccess) return err;
    if ((err = clear_scale_padding(col, st)) != cudaSuccess) return err;
    // the encode pass reduces "partials": here one value each
    return launch_pair_encode(x, rows, cols, ld_x, sr, true, sign_mask, seed, stream_row, stream_col, row, col,
                              amax_in, amax_in + 1, 1, false, st);
}

cudaError_t launch_requantize_col_rht(const QuantTarget* in, bool sr, uint32_t sign_mask, uint64_t seed,
                                      uint64_t stream_id, const QuantTarget* out, float* workspace, cudaStream_t st) {
    cudaError_t err;
    if ((err = clear_scale_padding(out, st)) != cudaSuccess) return err;
    RequantArgs ra{};
    ra.in_codes = in->codes;
    ra.in_ld = in->ld_codes;
    ra.in_scales = in->scales;
    ra.in_s4 = (uint32_t)((in->lcols + 63) / 64);
    ra.in_sg = in->sg;
    ra.rows = (uint32_t)in->lrows;
    ra.cols = (uint32_t)in->lcols;
    ra.tiles_r = (uint32_t)((in->lrows + 127) / 128);
    ra.tiles_c = (uint32_t)((in->lcols + 63) / 64);
    ra.out = make_target(out);
    ra.mask = sign_mask;
    for (int i = 0; i < 16; ++i) ra.sgf[i] = ((sign_mask >> i) & 1u) ? 0x80000000u : 0u;
    ra.keys = philox_keys(seed);
    ra.stream = stream_id;
    const int64_t ntiles = (int64_t)ra.tiles_r * ra.tiles_c;
    {
        RequantArgs a = ra;
        a.partials_out = workspace;
        auto k = requant_kernel<Pass::kAmax, false>;
        int g = persistent_grid(k, ntiles);
        if (g > kMaxAmaxPartials) g = kMaxAmaxPartials;
        k<<<g, kThreads, 0, st>>>(a);
        ra.n_partials = g;
    }
    ra.partials_in = workspace;
    auto launch = [&](auto k) { k<<<persistent_grid(k, ntiles), kThreads, 0, st>>>(ra); };
    if (sr) launch(requant_kernel<Pass::kEncode, true>);
    else launch(requant_kernel<Pass::kEncode, false>);
    return cudaGetLastError();
}

cudaError_t quantize_bounds_read_and_clear(uint64_t* n) { return bounds_read_and_clear_local(n); }

}  // namespace nvfp4

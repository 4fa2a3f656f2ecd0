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

#include "device_common.cuh"
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
};

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
    uint64_t seed, stream;
};

// One thread = one 1x16 block: two 16-byte loads, RHT in registers (optional),
// block amax, E4M3 scale, 8 bytes of codes.
template <Pass P, bool kRHT, bool kSR>
__global__ void __launch_bounds__(kThreads) rowwise_kernel(const RowArgs a) {
    __shared__ float red[32];
    __shared__ float rb_table[128];
    TensorScale ts{1.0f, 1.0f};
    if constexpr (P == Pass::kEncode) {
        ts = load_tensor_scale(a.partials_in, a.n_partials, red, a.out, nullptr);
        fill_rb_table(rb_table, ts.s_enc);
        __syncthreads();
    }
    float local_max = 0.0f;
    PhiloxKeys keys;
    if constexpr (kSR) keys = philox_keys(a.seed);
    // block b = r * bpr + j; (r, j) advance by the grid stride without a division
    const uint32_t stride = gridDim.x * kThreads;
    const uint32_t stride_r = stride / a.bpr, stride_j = stride - stride_r * a.bpr;
    uint32_t b = blockIdx.x * kThreads + threadIdx.x;
    uint32_t r = b / a.bpr, j = b - r * a.bpr;
    for (; b < a.total; b += stride) {
        const uint16_t* src = a.x + (int64_t)r * a.ld_x + (int64_t)j * 16;
        const uint4 u0 = ld_nc_v4(src), u1 = ld_nc_v4(src + 8);
        float t[16] = {bf16lo(u0.x), bf16hi(u0.x), bf16lo(u0.y), bf16hi(u0.y), bf16lo(u0.z), bf16hi(u0.z),
                       bf16lo(u0.w), bf16hi(u0.w), bf16lo(u1.x), bf16hi(u1.x), bf16lo(u1.y), bf16hi(u1.y),
                       bf16lo(u1.z), bf16hi(u1.z), bf16lo(u1.w), bf16hi(u1.w)};
        if constexpr (kRHT) rht16(t, a.mask);
        float amax_b = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(t[i]));
        if constexpr (P == Pass::kAmax) {
            local_max = fmaxf(local_max, amax_b);
        } else {
            float r_b;
            const uint32_t sc = block_scale_tab(amax_b, ts.s_enc, rb_table, &r_b);
            const uint64_t idx = (uint64_t)r * ((uint64_t)a.bpr * 16u) + (uint64_t)j * 16u;
            const uint2 q = encode16<kSR>(t, r_b, keys, a.stream, idx);
            *reinterpret_cast<uint2*>(a.out.codes + (int64_t)r * a.out.ld_codes + (int64_t)j * 8) = q;
            a.out.scales[scale_offset(r, j, a.out.s4)] = (uint8_t)sc;
        }
        j += stride_j;
        r += stride_r;
        if (j >= a.bpr) {
            j -= a.bpr;
            ++r;
        }
    }
    if constexpr (P == Pass::kAmax) block_max_store(local_max, a.partials_out, red);
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
    uint64_t seed, stream;
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
    if constexpr (P == Pass::kEncode) {
        ts = load_tensor_scale(a.partials_in, a.n_partials, red, a.out, nullptr);
        fill_rb_table(rb_table, ts.s_enc);
        __syncthreads();
    }
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t ntiles = a.tiles_r * a.tiles_c;
    float local_max = 0.0f, plain_max = 0.0f;
    PhiloxKeys keys;
    if constexpr (kSR) keys = philox_keys(a.seed);
    for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const uint32_t tr = tile % a.tiles_r, tc = tile / a.tiles_r;
        const uint32_t r0 = tr * 128u + warp * 16u, c = tc * 64u + lane * 2u;
        if (r0 >= a.rows || c >= a.cols) continue;
        const uint16_t* src = a.x + (int64_t)r0 * a.ld_x + c;
        float t0[16], t1[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t w = ld_nc_u32(src + (int64_t)i * a.ld_x);
            t0[i] = bf16lo(w);
            t1[i] = bf16hi(w);
        }
        if constexpr (kDual) {
#pragma unroll
            for (int i = 0; i < 16; ++i) plain_max = fmaxf(plain_max, fmaxf(fabsf(t0[i]), fabsf(t1[i])));
        }
        if constexpr (kRHT) {
            rht16(t0, a.mask);
            rht16(t1, a.mask);
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
            float rb0, rb1;
            const uint32_t sc0 = block_scale_tab(m0, ts.s_enc, rb_table, &rb0);
            const uint32_t sc1 = block_scale_tab(m1, ts.s_enc, rb_table, &rb1);
            const uint2 q0 = encode16<kSR>(t0, rb0, keys, a.stream, (uint64_t)c * a.rows + r0);
            const uint2 q1 = encode16<kSR>(t1, rb1, keys, a.stream, (uint64_t)(c + 1) * a.rows + r0);
            *reinterpret_cast<uint2*>(a.out.codes + (int64_t)c * a.out.ld_codes + r0 / 2) = q0;
            *reinterpret_cast<uint2*>(a.out.codes + (int64_t)(c + 1) * a.out.ld_codes + r0 / 2) = q1;
            a.out.scales[scale_offset(c, r0 / 16, a.out.s4)] = (uint8_t)sc0;
            a.out.scales[scale_offset(c + 1, r0 / 16, a.out.s4)] = (uint8_t)sc1;
        }
    }
    if constexpr (P == Pass::kAmax) {
        block_max_store(local_max, a.partials_out, red);
        if constexpr (kDual) {
            __syncthreads();
            block_max_store(plain_max, a.partials_out_plain, red);
        }
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
    PhiloxKeys keys;
    if constexpr (kSR) keys = philox_keys(a.seed);
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
        if constexpr (!kSR) {
            float v0[16], v1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                v0[i] = __fmul_rn(t0[i], r_b);
                v1[i] = __fmul_rn(t1[i], r_b);
            }
            q0 = make_uint2(e2m1_rne_x8(v0), e2m1_rne_x8(v0 + 8));
            q1 = make_uint2(e2m1_rne_x8(v1), e2m1_rne_x8(v1 + 8));
        } else {
            q0 = make_uint2(0u, 0u);
            q1 = make_uint2(0u, 0u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                // SR index: the row-wise index of x, shared by both orientations
                const uint64_t idx = (uint64_t)(r0 + i) * a.cols + c;     // even: c and c+1 share a word
                const uint4 w = sr_words4(keys, a.stream, idx >> 3);
                const uint32_t sel = (uint32_t)(idx >> 1) & 3u;
                const uint32_t word = sel == 0 ? w.x : (sel == 1 ? w.y : (sel == 2 ? w.z : w.w));
                const uint32_t c0 = e2m1_sr_add(__fmul_rn(t0[i], r_b), sr_addend_lo(word));
                const uint32_t c1 = e2m1_sr_add(__fmul_rn(t1[i], r_b), sr_addend_hi(word));
                if (i < 8) {
                    q0.x |= c0 << (4 * i);
                    q1.x |= c1 << (4 * i);
                } else {
                    q0.y |= c0 << (4 * (i - 8));
                    q1.y |= c1 << (4 * (i - 8));
                }
            }
        }
        if (a.emit_col) {
            *reinterpret_cast<uint2*>(a.out.codes + (int64_t)c * a.out.ld_codes + r0 / 2) = q0;
            *reinterpret_cast<uint2*>(a.out.codes + (int64_t)(c + 1) * a.out.ld_codes + r0 / 2) = q1;
            a.out.scales[scale_offset(c, r0 / 16, a.out.s4)] = (uint8_t)sc;
            a.out.scales[scale_offset(c + 1, r0 / 16, a.out.s4)] = (uint8_t)sc;
        }
        if (a.emit_row) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                a.out2.codes[(int64_t)(r0 + i) * a.out2.ld_codes + c / 2] =
                    (uint8_t)(nibble(q0, i) | (nibble(q1, i) << 4));
                if ((lane & 7u) == 0) a.out2.scales[scale_offset(r0 + i, c / 16, a.out2.s4)] = (uint8_t)sc;
            }
        }
    }
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

}  // namespace

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool scale_2d, bool sr,
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
    ra.seed = seed;
    ra.stream = stream_id;

    ColArgs ca{};
    ca.x = x;
    ca.ld_x = ld_x;
    ca.rows = (uint32_t)rows;
    ca.cols = (uint32_t)cols;
    ca.tiles_r = (uint32_t)((rows + 127) / 128);
    ca.tiles_c = (uint32_t)((cols + 63) / 64);
    ca.mask = sign_mask;
    ca.seed = seed;
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
        } else {
            auto k = tile2d_kernel<false>;
            k<<<persistent_grid(k, ntiles), kThreads, 0, st>>>(ca);
        }
        return cudaGetLastError();
    }

    int n_row = 0, n_col = 0;
    if (!rht) {
        n_row = n_col = row_amax<false>(ra, part_a, st);
        part_b = part_a;
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

    if (row) {
        RowArgs r = ra;
        r.out = make_target(row);
        r.partials_in = part_a;
        r.n_partials = n_row;
        auto launch = [&](auto k) {
            k<<<persistent_grid(k, ((int64_t)r.total + kThreads - 1) / kThreads), kThreads, 0, st>>>(r);
        };
        if (rht && sr) launch(rowwise_kernel<Pass::kEncode, true, true>);
        else if (rht) launch(rowwise_kernel<Pass::kEncode, true, false>);
        else if (sr) launch(rowwise_kernel<Pass::kEncode, false, true>);
        else launch(rowwise_kernel<Pass::kEncode, false, false>);
    }
    if (col) {
        ColArgs c = ca;
        c.out = make_target(col);
        c.partials_in = part_b;
        c.n_partials = n_col;
        auto launch = [&](auto k) { k<<<persistent_grid(k, ntiles), kThreads, 0, st>>>(c); };
        if (rht && sr) launch(colwise_kernel<Pass::kEncode, true, true>);
        else if (rht) launch(colwise_kernel<Pass::kEncode, true, false>);
        else if (sr) launch(colwise_kernel<Pass::kEncode, false, true>);
        else launch(colwise_kernel<Pass::kEncode, false, false>);
    }
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
    ca.seed = seed;
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
    {
        RowArgs r{};
        r.x = x;
        r.ld_x = ld_x;
        r.bpr = (uint32_t)(cols / 16);
        r.total = (uint32_t)(rows * (cols / 16));
        r.seed = seed;
        r.stream = stream_row;
        r.out = make_target(row);
        r.partials_in = part_plain;
        r.n_partials = n;
        auto launch = [&](auto k) {
            k<<<persistent_grid(k, ((int64_t)r.total + kThreads - 1) / kThreads), kThreads, 0, st>>>(r);
        };
        if (sr) launch(rowwise_kernel<Pass::kEncode, false, true>);
        else launch(rowwise_kernel<Pass::kEncode, false, false>);
    }
    {
        ColArgs c = ca;
        c.stream = stream_col;
        c.out = make_target(col);
        c.partials_in = part_rht;
        c.n_partials = n;
        auto launch = [&](auto k) { k<<<persistent_grid(k, ntiles), kThreads, 0, st>>>(c); };
        if (sr) launch(colwise_kernel<Pass::kEncode, true, true>);
        else launch(colwise_kernel<Pass::kEncode, true, false>);
    }
    return cudaGetLastError();
}

}  // namespace nvfp4

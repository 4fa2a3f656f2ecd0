// dequantize.cu -- x^ = x_E2M1 * s * s_g for an NVFP4 operand ("Full-Stack
// FP4", Sec. 2), rounded once to BF16 or FP32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "device_common.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

// E2M1 code -> value (sign, 2 exponent bits with bias 1, 1 mantissa bit).
__device__ __forceinline__ float e2m1_decode(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float mag = (e == 0) ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
    return (c & 8u) ? -mag : mag;
}

struct DeqArgs {
    const uint8_t* codes;
    int64_t ld_codes;
    const uint8_t* scales;
    uint32_t s4;
    const float* sg;
    uint32_t bpr, total;
    void* y;
    int64_t ldy;
    Extent xy;   // the bytes of y the call may write
};

// One thread = one block of 16 elements.  e2m1 * s_b is exact in binary32; the
// product with s_g is formed exactly in binary64 and rounded once.
template <bool kFP32>
__global__ void __launch_bounds__(kThreads) dequantize_kernel(const DeqArgs a) {
    const float s_g = *a.sg;
    const uint32_t stride = gridDim.x * kThreads;
    for (uint32_t b = blockIdx.x * kThreads + threadIdx.x; b < a.total; b += stride) {
        const uint32_t r = b / a.bpr, j = b - r * a.bpr;
        const uint2 q = *reinterpret_cast<const uint2*>(a.codes + (int64_t)r * a.ld_codes + (int64_t)j * 8);
        const float sb = e4m3_decode(a.scales[scale_offset(r, j, a.s4)]);
        float p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) p[i] = __fmul_rn(e2m1_decode(((i < 8 ? q.x : q.y) >> (4 * (i & 7))) & 0xFu), sb);
        if constexpr (kFP32) {
            float* dst = reinterpret_cast<float*>(a.y) + (int64_t)r * a.ldy + (int64_t)j * 16;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                store_out(reinterpret_cast<float4*>(dst + i),
                          make_float4(__fmul_rn(p[i], s_g), __fmul_rn(p[i + 1], s_g), __fmul_rn(p[i + 2], s_g),
                                      __fmul_rn(p[i + 3], s_g)),
                          a.xy);
        } else {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __nv_bfloat16 lo = __double2bfloat16((double)p[2 * i] * (double)s_g);
                const __nv_bfloat16 hi = __double2bfloat16((double)p[2 * i + 1] * (double)s_g);
                w[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
            }
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.y) + (int64_t)r * a.ldy + (int64_t)j * 16;
            store_out(reinterpret_cast<uint4*>(dst), make_uint4(w[0], w[1], w[2], w[3]), a.xy);
            store_out(reinterpret_cast<uint4*>(dst + 8), make_uint4(w[4], w[5], w[6], w[7]), a.xy);
        }
    }
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* codes, int64_t ld_codes, const uint8_t* scales, const float* sg,
                              int64_t rows, int64_t cols, void* y, int64_t ldy, bool out_fp32, cudaStream_t st) {
    const int64_t esz = out_fp32 ? 4 : 2;
    DeqArgs a{codes, ld_codes, scales, (uint32_t)((cols + 63) / 64), sg, (uint32_t)(cols / 16),
              (uint32_t)(rows * (cols / 16)), y, ldy, extent_rows(y, rows, ldy * esz, cols * esz)};
    if (a.total == 0) return cudaSuccess;
    int64_t grid = ((int64_t)a.total + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    if (out_fp32) dequantize_kernel<true><<<(int)grid, kThreads, 0, st>>>(a);
    else dequantize_kernel<false><<<(int)grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t dequantize_bounds_read_and_clear(uint64_t* n) { return bounds_read_and_clear_local(n); }

}  // namespace nvfp4

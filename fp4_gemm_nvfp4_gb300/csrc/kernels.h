// kernels.h -- host-side launchers of the NVFP4 kernels (internal to the
// library; the public interface is include/nvfp4.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

// Bit the kernels set in their device status word when a bounded wait runs out.
constexpr unsigned int kStatusTimeoutBit = 1u;

// One emitted orientation of a quantize call: logical [lrows][lcols].
struct QuantTarget {
    uint8_t* codes;
    int64_t ld_codes;
    uint8_t* scales;
    float* amax;      // may be null
    float* sg;
    int64_t lrows, lcols;
};

// Device workspace floats the amax passes of one quantize call use.
constexpr int kMaxAmaxPartials = 4096;
constexpr size_t kQuantizeWorkspaceBytes = 2 * kMaxAmaxPartials * sizeof(float);

// Wgrad's second operand from a row-wise operand (in: [lrows][lcols]; out:
// [lcols][lrows]): dequantize, RHT along the rows, col-wise 1x16.
cudaError_t launch_requantize_col_rht(const QuantTarget* in, bool sr, uint32_t sign_mask, uint64_t seed,
                                      uint64_t stream_id, const QuantTarget* out, float* workspace,
                                      cudaStream_t stream);

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool scale_2d,
                            bool scale_46, bool sr, bool rht, uint32_t sign_mask, uint64_t seed, uint64_t stream_id,
                            const QuantTarget* row, const QuantTarget* col, float* workspace,
                            cudaStream_t stream);

// Row-wise 1x16 without RHT and col-wise 1x16 with RHT of one input, sharing
// one amax pass (workspace as for launch_quantize).
// As launch_quantize_row_col_rht with the two tensor amaxes given (amax_in[0]
// plain, amax_in[1] rotated; e.g. from the producing GEMM): no amax pass.
cudaError_t launch_quantize_row_col_rht_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool sr,
                                             uint32_t sign_mask, uint64_t seed, uint64_t stream_row,
                                             uint64_t stream_col, const float* amax_in, const QuantTarget* row,
                                             const QuantTarget* col, cudaStream_t stream);

cudaError_t launch_quantize_row_col_rht(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, bool sr,
                                       uint32_t sign_mask, uint64_t seed, uint64_t stream_row, uint64_t stream_col,
                                       const QuantTarget* row, const QuantTarget* col, float* workspace,
                                       cudaStream_t stream);

struct GemmOperand {
    const uint8_t* codes;
    int64_t ld_codes;
    const uint8_t* scales;
    const float* sg;
    int64_t rows, cols;
};

// The low-rank term of a LoRA-SVD projection, D += beta * U V^T: U [M][r]
// and V [N][r] row-major BF16, r a multiple of 64; u_scaled is scratch for
// U * beta / (s_gA s_gB) ([M][r] BF16, 16-byte aligned).
struct LowRank {
    const void* u;
    int64_t ldu;
    const void* v;
    int64_t ldv;
    int64_t r;
    float beta;
    void* u_scaled;
};

// D = alpha * (s_gA s_gB A B^T) + beta * C with C [M][ldc] of D's dtype
// (C may be D itself: each element is read before it is written).
struct Axpby {
    float alpha;
    const void* c;
    int64_t ldc;
    float beta;
};

// amax_out (BF16 output only): [0] = max |D|, [1] = max |U d| over the 16-row
// blocks of each column (the RHT U = H16 diag(rht_mask) / 4 along D's rows),
// the two tensor amaxes nvfp4_quantize_row_col_rht takes of D.
cudaError_t launch_gemm(const GemmOperand& a, const GemmOperand& b, void* d, int64_t ldd, bool out_fp32,
                        cudaStream_t stream, const LowRank* lora = nullptr, float* amax_out = nullptr,
                        uint32_t rht_mask = 0, const Axpby* axpby = nullptr);

// Read and clear the GEMM kernels' device status word (synchronous).
cudaError_t gemm_read_and_clear_status(unsigned int* status);

// Add the stores that the debug build's bounds check skipped in one source
// file's kernels to *n and clear that count (synchronous; in the regular
// build they add nothing).
cudaError_t quantize_bounds_read_and_clear(uint64_t* n);
cudaError_t gemm_bounds_read_and_clear(uint64_t* n);
cudaError_t dequantize_bounds_read_and_clear(uint64_t* n);

// Test support: the next GEMM launch waits at most timeout_ns per barrier and
// its leader CTA leaves out one scale-warp arrival, so one wait runs out.
void arm_gemm_fault(uint64_t timeout_ns);

cudaError_t launch_dequantize(const uint8_t* codes, int64_t ld_codes, const uint8_t* scales, const float* sg,
                              int64_t rows, int64_t cols, void* y, int64_t ldy, bool out_fp32,
                              cudaStream_t stream);

// cuTensorMapEncodeTiled from the driver (null if unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace nvfp4

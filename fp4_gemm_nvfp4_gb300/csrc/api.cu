// api.cu -- the C ABI of include/nvfp4.h: argument validation and dispatch.
//
// Every check runs on the host before anything is enqueued, so an error
// status means no kernel was launched (except NVFP4_ERR_CUDA from a launch).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/nvfp4.h"
#include "../../include/nvfp4_testing.h"
#include "bounds.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace {
// Bytes taken off the end of every declared output range (test support of
// the debug build; always 0 in the regular build).
std::atomic<int64_t> g_extent_shrink{0};
}  // namespace

Extent extent_of(const void* p, int64_t bytes) {
    const int64_t shrink = g_extent_shrink.load(std::memory_order_relaxed);
    const int64_t n = bytes > shrink ? bytes - shrink : 0;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Extent{lo, lo + (uintptr_t)n};
}
}  // namespace nvfp4

namespace {

using nvfp4::QuantTarget;

// An NVTX range around one C-ABI call (host side only: a profiler's timeline
// then attributes each kernel launch to the entry point that enqueued it; with
// no tool attached a push/pop costs a null check).
struct ApiRange {
    explicit ApiRange(const char* name) { nvtxRangePushA(name); }
    ~ApiRange() { nvtxRangePop(); }
    ApiRange(const ApiRange&) = delete;
    ApiRange& operator=(const ApiRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Validate one emitted orientation (logical [lrows][lcols]).
nvfp4_status check_target(const nvfp4_tensor* t, int64_t lrows, int64_t lcols) {
    if (!t) return NVFP4_ERR_INVALID_ARG;
    if (t->rows != lrows || t->cols != lcols) return NVFP4_ERR_INVALID_ARG;
    if (!t->global_scale) return NVFP4_ERR_INVALID_ARG;
    if (lrows > 0 && lcols > 0) {
        if (!t->codes || !t->scales) return NVFP4_ERR_INVALID_ARG;
        if (t->ld_codes < lcols / 2) return NVFP4_ERR_SHAPE;
        if (t->ld_codes % 16 != 0 || !aligned16(t->codes) || !aligned16(t->scales)) return NVFP4_ERR_ALIGNMENT;
    }
    return NVFP4_OK;
}

QuantTarget to_target(const nvfp4_tensor* t) {
    return QuantTarget{t->codes, t->ld_codes, t->scales, t->amax, t->global_scale, t->rows, t->cols};
}

nvfp4_status quantize_impl(const void* x, int64_t rows, int64_t cols, int64_t ld_x, nvfp4_scaling scaling,
                           nvfp4_rounding rounding, uint64_t seed, uint64_t stream_id, int orientations,
                           const nvfp4_tensor* out_row, const nvfp4_tensor* out_col, bool rht, uint16_t mask,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (scaling != NVFP4_SCALE_1X16 && scaling != NVFP4_SCALE_16X16 && scaling != NVFP4_SCALE_1X16_46)
        return NVFP4_ERR_INVALID_ARG;
    if (rounding != NVFP4_ROUND_RNE && rounding != NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;
    if (orientations < 1 || orientations > 3) return NVFP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return NVFP4_ERR_SHAPE;
    const bool want_row = (orientations & NVFP4_ROWWISE) != 0;
    const bool want_col = (orientations & NVFP4_COLWISE) != 0;
    const bool two_d = scaling == NVFP4_SCALE_16X16;
    if (rht && two_d) return NVFP4_ERR_UNSUPPORTED;
    if (cols % 16 != 0) return NVFP4_ERR_SHAPE;
    if ((two_d || want_col) && rows % 16 != 0) return NVFP4_ERR_SHAPE;
    if (rows > 0 && cols > 0) {
        if (!x) return NVFP4_ERR_INVALID_ARG;
        if (ld_x < cols) return NVFP4_ERR_SHAPE;
        if (ld_x % 8 != 0 || !aligned16(x)) return NVFP4_ERR_ALIGNMENT;
    }
    if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return NVFP4_ERR_UNSUPPORTED;
    if (rows * (cols / 16) >= (int64_t(1) << 32) - 1) return NVFP4_ERR_UNSUPPORTED;
    nvfp4_status s;
    if (want_row && (s = check_target(out_row, rows, cols)) != NVFP4_OK) return s;
    if (want_col && (s = check_target(out_col, cols, rows)) != NVFP4_OK) return s;
    if (!workspace || workspace_bytes < nvfp4::kQuantizeWorkspaceBytes || !aligned16(workspace))
        return NVFP4_ERR_WORKSPACE;

    QuantTarget tr{}, tc{};
    if (want_row) tr = to_target(out_row);
    if (want_col) tc = to_target(out_col);
    const cudaError_t e = nvfp4::launch_quantize(
        static_cast<const uint16_t*>(x), rows, cols, ld_x, two_d, scaling == NVFP4_SCALE_1X16_46,
        rounding == NVFP4_ROUND_SR, rht, mask, seed,
        stream_id, want_row ? &tr : nullptr, want_col ? &tc : nullptr, static_cast<float*>(workspace), stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Shape, pointer and workspace checks shared by the quantize entry points.
nvfp4_status check_quantize_input(const void* x, int64_t rows, int64_t cols, int64_t ld_x) {
    if (rows < 0 || cols < 0) return NVFP4_ERR_SHAPE;
    if (rows > 0 && cols > 0) {
        if (!x) return NVFP4_ERR_INVALID_ARG;
        if (ld_x < cols) return NVFP4_ERR_SHAPE;
        if (ld_x % 8 != 0 || !aligned16(x)) return NVFP4_ERR_ALIGNMENT;
    }
    if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return NVFP4_ERR_UNSUPPORTED;
    if (rows * (cols / 16) >= (int64_t(1) << 32) - 1) return NVFP4_ERR_UNSUPPORTED;
    return NVFP4_OK;
}

nvfp4_status check_operand(const nvfp4_tensor* t) {
    if (!t || !t->codes || !t->scales || !t->global_scale) return NVFP4_ERR_INVALID_ARG;
    if (t->rows < 0 || t->cols < 0) return NVFP4_ERR_SHAPE;
    if (t->cols % 16 != 0) return NVFP4_ERR_SHAPE;
    if (t->ld_codes < t->cols / 2) return NVFP4_ERR_SHAPE;
    if (t->ld_codes % 16 != 0 || !aligned16(t->codes) || !aligned16(t->scales)) return NVFP4_ERR_ALIGNMENT;
    if (t->rows >= (int64_t(1) << 31) || t->cols >= (int64_t(1) << 31)) return NVFP4_ERR_UNSUPPORTED;
    return NVFP4_OK;
}

nvfp4::GemmOperand to_operand(const nvfp4_tensor* t) {
    return nvfp4::GemmOperand{t->codes, t->ld_codes, t->scales, t->global_scale, t->rows, t->cols};
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Carves one [rows][cols] NVFP4 operand (codes with a 16-byte multiple row
// stride, tile-layout scales, s_g, amax) out of a workspace at *off.
nvfp4_tensor carve_operand(uint8_t* base, size_t* off, int64_t rows, int64_t cols) {
    nvfp4_tensor t{};
    t.rows = rows;
    t.cols = cols;
    t.ld_codes = (cols / 2 + 15) / 16 * 16;
    t.codes = base ? base + *off : nullptr;
    *off = align256(*off + (size_t)(rows * t.ld_codes));
    t.scales = base ? base + *off : nullptr;
    *off = align256(*off + nvfp4_scale_bytes(rows, cols));
    t.global_scale = base ? reinterpret_cast<float*>(base + *off) : nullptr;
    t.amax = base ? reinterpret_cast<float*>(base + *off) + 1 : nullptr;
    *off = align256(*off + 2 * sizeof(float));
    return t;
}

// The Newton-Schulz step's workspace: A_k and B_k (bf16 [m][m]) first, then
// the five quantized operands and the quantizer's scratch.
struct NsWorkspace {
    void* a;
    void* b;
    nvfp4_tensor qx, qxc, qa, qac, qb;
    void* qws;
    size_t bytes;
};

NsWorkspace ns_layout(void* workspace, int64_t m, int64_t n) {
    uint8_t* base = static_cast<uint8_t*>(workspace);
    NsWorkspace w{};
    size_t off = 0;
    w.a = base ? base + off : nullptr;
    off = align256(off + (size_t)(m * m * 2));
    w.b = base ? base + off : nullptr;
    off = align256(off + (size_t)(m * m * 2));
    w.qx = carve_operand(base, &off, m, n);
    w.qxc = carve_operand(base, &off, n, m);
    w.qa = carve_operand(base, &off, m, m);
    w.qac = carve_operand(base, &off, m, m);
    w.qb = carve_operand(base, &off, m, m);
    w.qws = base ? base + off : nullptr;
    off = align256(off + nvfp4::kQuantizeWorkspaceBytes);
    w.bytes = off;
    return w;
}

nvfp4_status gemm_axpby_impl(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, int64_t ldd,
                             nvfp4_dtype out_dtype, float alpha, const void* C, int64_t ldc, float beta,
                             cudaStream_t st) {
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
    if (!std::isfinite(alpha) || !std::isfinite(beta)) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s;
    if ((s = check_operand(A)) != NVFP4_OK) return s;
    if ((s = check_operand(B)) != NVFP4_OK) return s;
    if (A->cols != B->cols) return NVFP4_ERR_SHAPE;
    if (!D) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    const int64_t esz = out_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (ldd < N) return NVFP4_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(D) % (uintptr_t)esz) != 0) return NVFP4_ERR_ALIGNMENT;
    const bool with_c = beta != 0.0f;
    if (with_c) {
        if (!C) return NVFP4_ERR_INVALID_ARG;
        if (ldc < N) return NVFP4_ERR_SHAPE;
        if ((reinterpret_cast<uintptr_t>(C) % (uintptr_t)esz) != 0) return NVFP4_ERR_ALIGNMENT;
        if (C == D && ldc != ldd) return NVFP4_ERR_INVALID_ARG;
    }
    if (ceil_div(M, 128) * ceil_div(N, 256) >= (int64_t(1) << 32)) return NVFP4_ERR_UNSUPPORTED;
    if (K == 0) return NVFP4_ERR_UNSUPPORTED;   // no product to carry the C term
    if (M == 0 || N == 0) return NVFP4_OK;
    const nvfp4::Axpby ax{alpha, with_c ? C : nullptr, with_c ? ldc : 0, with_c ? beta : 0.0f};
    const cudaError_t e = nvfp4::launch_gemm(to_operand(A), to_operand(B), D, ldd, out_dtype == NVFP4_OUT_FP32, st,
                                             nullptr, nullptr, 0, &ax);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t nvfp4_scale_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)(ceil_div(rows, 128) * ceil_div(cols, 64) * 512);
}

size_t nvfp4_quantize_workspace_size(int64_t rows, int64_t cols, int orientations) {
    (void)rows;
    (void)cols;
    (void)orientations;
    return nvfp4::kQuantizeWorkspaceBytes;
}

nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, nvfp4_scaling scaling,
                            nvfp4_rounding rounding, uint64_t seed, uint64_t stream_id, int orientations,
                            const nvfp4_tensor* out_row, const nvfp4_tensor* out_col, void* workspace,
                            size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_quantize");
    return quantize_impl(x, rows, cols, ld_x, scaling, rounding, seed, stream_id, orientations, out_row, out_col,
                         false, 0, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_rht_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, nvfp4_scaling scaling,
                                nvfp4_rounding rounding, uint64_t seed, uint64_t stream_id, int orientations,
                                const nvfp4_tensor* out_row, const nvfp4_tensor* out_col, uint16_t rht_sign_mask,
                                void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_rht_quantize");
    return quantize_impl(x, rows, cols, ld_x, scaling, rounding, seed, stream_id, orientations, out_row, out_col,
                         true, rht_sign_mask, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_quantize_row_col_rht(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                        nvfp4_rounding rounding, uint64_t seed, uint64_t stream_row,
                                        uint64_t stream_col, uint16_t rht_sign_mask, const nvfp4_tensor* out_row,
                                        const nvfp4_tensor* out_col, void* workspace, size_t workspace_bytes,
                                        nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_quantize_row_col_rht");
    if (rounding != NVFP4_ROUND_RNE && rounding != NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return NVFP4_ERR_SHAPE;
    if (cols % 16 != 0 || rows % 16 != 0) return NVFP4_ERR_SHAPE;
    nvfp4_status s;
    if ((s = check_quantize_input(x, rows, cols, ld_x)) != NVFP4_OK) return s;
    if ((s = check_target(out_row, rows, cols)) != NVFP4_OK) return s;
    if ((s = check_target(out_col, cols, rows)) != NVFP4_OK) return s;
    if (!workspace || workspace_bytes < nvfp4::kQuantizeWorkspaceBytes || !aligned16(workspace))
        return NVFP4_ERR_WORKSPACE;
    const QuantTarget tr = to_target(out_row), tc = to_target(out_col);
    const cudaError_t e = nvfp4::launch_quantize_row_col_rht(
        static_cast<const uint16_t*>(x), rows, cols, ld_x, rounding == NVFP4_ROUND_SR, rht_sign_mask, seed, stream_row,
        stream_col, &tr, &tc, static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_requantize_col_rht(const nvfp4_tensor* in_row, nvfp4_rounding rounding, uint64_t seed,
                                      uint64_t stream_id, uint16_t rht_sign_mask, const nvfp4_tensor* out_col,
                                      void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_requantize_col_rht");
    if (rounding != NVFP4_ROUND_RNE && rounding != NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;
    if (!in_row || !out_col) return NVFP4_ERR_INVALID_ARG;
    const int64_t rows = in_row->rows, cols = in_row->cols;
    if (rows < 0 || cols < 0) return NVFP4_ERR_SHAPE;
    if (rows % 16 != 0 || cols % 16 != 0) return NVFP4_ERR_SHAPE;
    nvfp4_status s;
    if ((s = check_target(in_row, rows, cols)) != NVFP4_OK) return s;
    if ((s = check_target(out_col, cols, rows)) != NVFP4_OK) return s;
    if (out_col->global_scale == in_row->global_scale ||
        (rows > 0 && cols > 0 && (out_col->codes == in_row->codes || out_col->scales == in_row->scales)))
        return NVFP4_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return NVFP4_ERR_UNSUPPORTED;
    if (cols * (rows / 16) >= (int64_t(1) << 32) - 1) return NVFP4_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < nvfp4::kQuantizeWorkspaceBytes || !aligned16(workspace))
        return NVFP4_ERR_WORKSPACE;
    const QuantTarget ti = to_target(in_row), to = to_target(out_col);
    const cudaError_t e = nvfp4::launch_requantize_col_rht(&ti, rounding == NVFP4_ROUND_SR, rht_sign_mask, seed,
                                                           stream_id, &to, static_cast<float*>(workspace),
                                                           reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, int64_t ldd,
                        nvfp4_dtype out_dtype, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_gemm");
    (void)workspace;
    (void)workspace_bytes;
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s;
    if ((s = check_operand(A)) != NVFP4_OK) return s;
    if ((s = check_operand(B)) != NVFP4_OK) return s;
    if (A->cols != B->cols) return NVFP4_ERR_SHAPE;
    if (!D) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    const int64_t esz = out_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (ldd < N) return NVFP4_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(D) % (uintptr_t)esz) != 0) return NVFP4_ERR_ALIGNMENT;
    if (ceil_div(M, 128) * ceil_div(N, 256) >= (int64_t(1) << 32)) return NVFP4_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0) return NVFP4_OK;
    if (K == 0)   // empty reduction: D = 0
        return cudaMemset2DAsync(D, (size_t)(ldd * esz), 0, (size_t)(N * esz), (size_t)M, st) == cudaSuccess
                   ? NVFP4_OK
                   : NVFP4_ERR_CUDA;
    const cudaError_t e = nvfp4::launch_gemm(to_operand(A), to_operand(B), D, ldd, out_dtype == NVFP4_OUT_FP32, st);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_gemm_amax(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, int64_t ldd, float* amax_out,
                             uint16_t rht_sign_mask, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_gemm_amax");
    (void)workspace;
    (void)workspace_bytes;
    nvfp4_status s;
    if ((s = check_operand(A)) != NVFP4_OK) return s;
    if ((s = check_operand(B)) != NVFP4_OK) return s;
    if (A->cols != B->cols) return NVFP4_ERR_SHAPE;
    if (!D || !amax_out) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    if (ldd < N) return NVFP4_ERR_SHAPE;
    if (M % 16 != 0) return NVFP4_ERR_SHAPE;   // 16-row blocks of the rotated amax
    if (!aligned16(D) || ldd % 8 != 0 || (reinterpret_cast<uintptr_t>(amax_out) & 3u) != 0)
        return NVFP4_ERR_ALIGNMENT;
    if (ceil_div(M, 128) * ceil_div(N, 256) >= (int64_t(1) << 32)) return NVFP4_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0 || K == 0) {
        // D = 0 (or empty): both maxima are 0
        if (M && N &&
            cudaMemset2DAsync(D, (size_t)(ldd * 2), 0, (size_t)(N * 2), (size_t)M, st) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        return cudaMemsetAsync(amax_out, 0, 2 * sizeof(float), st) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
    }
    const cudaError_t e = nvfp4::launch_gemm(to_operand(A), to_operand(B), D, ldd, false, st, nullptr, amax_out,
                                             rht_sign_mask);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_quantize_row_col_rht_amax(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                             nvfp4_rounding rounding, uint64_t seed, uint64_t stream_row,
                                             uint64_t stream_col, uint16_t rht_sign_mask, const float* amax_in,
                                             const nvfp4_tensor* out_row, const nvfp4_tensor* out_col,
                                             nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_quantize_row_col_rht_amax");
    if (rounding != NVFP4_ROUND_RNE && rounding != NVFP4_ROUND_SR) return NVFP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return NVFP4_ERR_SHAPE;
    if (cols % 16 != 0 || rows % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!amax_in || (reinterpret_cast<uintptr_t>(amax_in) & 3u) != 0) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s;
    if ((s = check_quantize_input(x, rows, cols, ld_x)) != NVFP4_OK) return s;
    if ((s = check_target(out_row, rows, cols)) != NVFP4_OK) return s;
    if ((s = check_target(out_col, cols, rows)) != NVFP4_OK) return s;
    const QuantTarget tr = to_target(out_row), tc = to_target(out_col);
    const cudaError_t e = nvfp4::launch_quantize_row_col_rht_amax(
        static_cast<const uint16_t*>(x), rows, cols, ld_x, rounding == NVFP4_ROUND_SR, rht_sign_mask, seed, stream_row,
        stream_col, amax_in, &tr, &tc, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

size_t nvfp4_gemm_lora_workspace_size(int64_t M, int64_t r) {
    if (M < 0 || r < 0) return 0;
    return (size_t)(M * r * 2) + 16;
}

nvfp4_status nvfp4_gemm_lora(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, int64_t ldd,
                             nvfp4_dtype out_dtype, const void* U, int64_t ldu, const void* V, int64_t ldv,
                             int64_t r, float beta, void* workspace, size_t workspace_bytes,
                             nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_gemm_lora");
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s;
    if ((s = check_operand(A)) != NVFP4_OK) return s;
    if ((s = check_operand(B)) != NVFP4_OK) return s;
    if (A->cols != B->cols) return NVFP4_ERR_SHAPE;
    if (!D || !U || !V) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    const int64_t esz = out_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (ldd < N) return NVFP4_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(D) % (uintptr_t)esz) != 0) return NVFP4_ERR_ALIGNMENT;
    if (r <= 0 || r % 64 != 0 || r > 4096) return NVFP4_ERR_UNSUPPORTED;
    if (ldu < r || ldv < r) return NVFP4_ERR_SHAPE;
    if (!aligned16(U) || !aligned16(V) || ldu % 8 != 0 || ldv % 8 != 0) return NVFP4_ERR_ALIGNMENT;
    if (!std::isfinite(beta)) return NVFP4_ERR_INVALID_ARG;
    if (ceil_div(M, 128) * ceil_div(N, 256) >= (int64_t(1) << 32)) return NVFP4_ERR_UNSUPPORTED;
    if (K == 0) return NVFP4_ERR_UNSUPPORTED;   // no FP4 product to carry the low-rank term
    if (!workspace || !aligned16(workspace) || workspace_bytes < nvfp4_gemm_lora_workspace_size(M, r))
        return NVFP4_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0) return NVFP4_OK;
    const nvfp4::LowRank lr{U, ldu, V, ldv, r, beta, workspace};
    const cudaError_t e =
        nvfp4::launch_gemm(to_operand(A), to_operand(B), D, ldd, out_dtype == NVFP4_OUT_FP32, st, &lr);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_gemm_axpby(const nvfp4_tensor* A, const nvfp4_tensor* B, void* D, int64_t ldd,
                              nvfp4_dtype out_dtype, float alpha, const void* C, int64_t ldc, float beta,
                              void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_gemm_axpby");
    (void)workspace;
    (void)workspace_bytes;
    return gemm_axpby_impl(A, B, D, ldd, out_dtype, alpha, C, ldc, beta, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_newton_schulz_workspace_size(int64_t m, int64_t n) {
    if (m <= 0 || n <= 0) return 0;
    return ns_layout(nullptr, m, n).bytes;
}

nvfp4_status nvfp4_newton_schulz_step(const void* X, int64_t m, int64_t n, int64_t ldx, float a, float b, float c,
                                      uint16_t rht_sign_mask, void* X_out, int64_t ld_out, void* workspace,
                                      size_t workspace_bytes, nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_newton_schulz_step");
    if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c)) return NVFP4_ERR_INVALID_ARG;
    if (m <= 0 || n <= 0 || m % 16 != 0 || n % 16 != 0) return NVFP4_ERR_SHAPE;
    nvfp4_status s;
    if ((s = check_quantize_input(X, m, n, ldx)) != NVFP4_OK) return s;
    if ((s = check_quantize_input(X_out, m, n, ld_out)) != NVFP4_OK) return s;
    if (X_out == X && ld_out != ldx) return NVFP4_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < nvfp4_newton_schulz_workspace_size(m, n))
        return NVFP4_ERR_WORKSPACE;
    const NsWorkspace w = ns_layout(workspace, m, n);
    const size_t qb = nvfp4::kQuantizeWorkspaceBytes;
    // qX = Q_1x16(X H) and qX' = Q_16x1(H^T X), one call
    if ((s = nvfp4_rht_quantize(X, m, n, ldx, NVFP4_SCALE_1X16_46, NVFP4_ROUND_RNE, 0, 0,
                                NVFP4_ROWWISE | NVFP4_COLWISE, &w.qx, &w.qxc, rht_sign_mask, w.qws, qb,
                                stream)) != NVFP4_OK)
        return s;
    // A = qX qX^T
    if ((s = nvfp4_gemm(&w.qx, &w.qx, w.a, m, NVFP4_OUT_BF16, nullptr, 0, stream)) != NVFP4_OK) return s;
    // qA = Q_1x16(A H), qA' = Q_16x1(H^T A); B = b A + c qA qA'
    if ((s = nvfp4_rht_quantize(w.a, m, m, m, NVFP4_SCALE_1X16_46, NVFP4_ROUND_RNE, 0, 0,
                                NVFP4_ROWWISE | NVFP4_COLWISE, &w.qa, &w.qac, rht_sign_mask, w.qws, qb,
                                stream)) != NVFP4_OK)
        return s;
    if ((s = nvfp4_gemm_axpby(&w.qa, &w.qac, w.b, m, NVFP4_OUT_BF16, c, w.a, m, b, nullptr, 0, stream)) !=
        NVFP4_OK)
        return s;
    // qB = Q_1x16(B H); X_out = a X + qB qX'
    if ((s = nvfp4_rht_quantize(w.b, m, m, m, NVFP4_SCALE_1X16_46, NVFP4_ROUND_RNE, 0, 0, NVFP4_ROWWISE, &w.qb,
                                nullptr, rht_sign_mask, w.qws, qb, stream)) != NVFP4_OK)
        return s;
    return nvfp4_gemm_axpby(&w.qb, &w.qxc, X_out, ld_out, NVFP4_OUT_BF16, 1.0f, X, ldx, a, nullptr, 0, stream);
}

nvfp4_status nvfp4_dequantize(const nvfp4_tensor* q, void* y, int64_t ldy, nvfp4_dtype out_dtype,
                              nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_dequantize");
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s;
    if ((s = check_operand(q)) != NVFP4_OK) return s;
    if (!y) return NVFP4_ERR_INVALID_ARG;
    const int64_t esz = out_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (ldy < q->cols) return NVFP4_ERR_SHAPE;
    if (!aligned16(y) || (ldy * esz) % 16 != 0) return NVFP4_ERR_ALIGNMENT;
    if (q->rows * (q->cols / 16) >= (int64_t(1) << 32) - 1) return NVFP4_ERR_UNSUPPORTED;
    const cudaError_t e = nvfp4::launch_dequantize(q->codes, q->ld_codes, q->scales, q->global_scale, q->rows,
                                                   q->cols, y, ldy, out_dtype == NVFP4_OUT_FP32,
                                                   reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

const char* nvfp4_status_string(nvfp4_status status) {
    switch (status) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
        case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE";
        case NVFP4_ERR_ALIGNMENT: return "NVFP4_ERR_ALIGNMENT";
        case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
        case NVFP4_ERR_WORKSPACE: return "NVFP4_ERR_WORKSPACE";
    }
    return "NVFP4_ERR_UNKNOWN";
}

nvfp4_status nvfp4_testing_arm_gemm_timeout(uint32_t wait_limit_us) {
    if (wait_limit_us < 1000u || wait_limit_us > 2000000u) return NVFP4_ERR_INVALID_ARG;
    nvfp4::arm_gemm_fault((uint64_t)wait_limit_us * 1000u);
    return NVFP4_OK;
}

nvfp4_status nvfp4_testing_bounds_violations(uint64_t* count) {
#ifdef NVFP4_BOUNDS_CHECK
    if (!count) return NVFP4_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
    uint64_t n = 0;
    if (nvfp4::quantize_bounds_read_and_clear(&n) != cudaSuccess ||
        nvfp4::gemm_bounds_read_and_clear(&n) != cudaSuccess ||
        nvfp4::dequantize_bounds_read_and_clear(&n) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    *count = n;
    return NVFP4_OK;
#else
    (void)count;
    return NVFP4_ERR_UNSUPPORTED;
#endif
}

nvfp4_status nvfp4_testing_bounds_shrink(int64_t bytes) {
#ifdef NVFP4_BOUNDS_CHECK
    if (bytes < 0 || bytes > 4096) return NVFP4_ERR_INVALID_ARG;
    nvfp4::g_extent_shrink.store(bytes, std::memory_order_relaxed);
    return NVFP4_OK;
#else
    (void)bytes;
    return NVFP4_ERR_UNSUPPORTED;
#endif
}

nvfp4_status nvfp4_device_error(nvfp4_stream_t stream) {
    const ApiRange range("nvfp4_device_error");
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return NVFP4_ERR_CUDA;
    unsigned int status = 0;
    if (nvfp4::gemm_read_and_clear_status(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
    return (status & nvfp4::kStatusTimeoutBit) ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
}

}  // extern "C"

"""ctypes binding of include/nvfp4.h (argument marshalling only).

Each function here has the name and argument order of the C entry point and
returns its nvfp4_status as an int.  Pointers are plain integers (device
addresses, or a cudaStream_t handle).  The library must be built in-tree
(``fp4_gemm_nvfp4_gb300/_build/libnvfp4.so``); loading fails loudly otherwise:
there is no fallback implementation.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libnvfp4.so")

# nvfp4_status
NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_SHAPE = 2
NVFP4_ERR_ALIGNMENT = 3
NVFP4_ERR_UNSUPPORTED = 4
NVFP4_ERR_CUDA = 5
NVFP4_ERR_TIMEOUT = 6
NVFP4_ERR_WORKSPACE = 7
# enums
NVFP4_SCALE_1X16 = 0
NVFP4_SCALE_16X16 = 1
NVFP4_SCALE_1X16_46 = 2
NVFP4_ROUND_RNE = 0
NVFP4_ROUND_SR = 1
NVFP4_OUT_BF16 = 0
NVFP4_OUT_FP32 = 1
NVFP4_ROWWISE = 1
NVFP4_COLWISE = 2

EXPORTED = ("nvfp4_scale_bytes", "nvfp4_quantize_workspace_size", "nvfp4_quantize",
            "nvfp4_rht_quantize", "nvfp4_gemm", "nvfp4_dequantize", "nvfp4_status_string",
            "nvfp4_device_error", "nvfp4_quantize_noalloc", "nvfp4_quantize_row_col_rht",
            "nvfp4_requantize_col_rht", "nvfp4_gemm_lora", "nvfp4_gemm_lora_workspace_size",
            "nvfp4_gemm_amax", "nvfp4_quantize_row_col_rht_amax", "nvfp4_gemm_axpby",
            "nvfp4_newton_schulz_workspace_size", "nvfp4_newton_schulz_step",
            "nvfp4_testing_arm_gemm_timeout", "nvfp4_testing_bounds_violations",
            "nvfp4_testing_bounds_shrink")


class nvfp4_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("global_scale", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld_codes", ctypes.c_int64)]


class NVFP4Error(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libnvfp4.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libnvfp4.so is not built ({path}); run __graft_entry__.build() "
                           "or python -m fp4_gemm_nvfp4_gb300.build")
    L = ctypes.CDLL(path)
    i32, i64, u16, u64, sz, vp = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint16, ctypes.c_uint64,
                                  ctypes.c_size_t, ctypes.c_void_p)
    tp = ctypes.POINTER(nvfp4_tensor)
    L.nvfp4_scale_bytes.argtypes, L.nvfp4_scale_bytes.restype = [i64, i64], sz
    L.nvfp4_quantize_workspace_size.argtypes = [i64, i64, i32]
    L.nvfp4_quantize_workspace_size.restype = sz
    qargs = [vp, i64, i64, i64, i32, i32, u64, u64, i32, tp, tp]
    L.nvfp4_quantize.argtypes = qargs + [vp, sz, vp]
    L.nvfp4_quantize.restype = i32
    L.nvfp4_rht_quantize.argtypes = qargs + [u16, vp, sz, vp]
    L.nvfp4_rht_quantize.restype = i32
    L.nvfp4_quantize_noalloc.argtypes = qargs + [vp]
    L.nvfp4_quantize_noalloc.restype = i32
    L.nvfp4_quantize_row_col_rht.argtypes = [vp, i64, i64, i64, i32, u64, u64, u64, u16, tp, tp, vp, sz, vp]
    L.nvfp4_quantize_row_col_rht.restype = i32
    L.nvfp4_requantize_col_rht.argtypes = [tp, i32, u64, u64, u16, tp, vp, sz, vp]
    L.nvfp4_requantize_col_rht.restype = i32
    L.nvfp4_gemm.argtypes = [tp, tp, vp, i64, i32, vp, sz, vp]
    L.nvfp4_gemm_amax.argtypes = [tp, tp, vp, i64, vp, u16, vp, sz, vp]
    L.nvfp4_gemm_amax.restype = i32
    L.nvfp4_quantize_row_col_rht_amax.argtypes = [vp, i64, i64, i64, i32, u64, u64, u64, u16, vp, tp, tp, vp]
    L.nvfp4_quantize_row_col_rht_amax.restype = i32
    L.nvfp4_gemm_lora_workspace_size.argtypes = [i64, i64]
    L.nvfp4_gemm_lora_workspace_size.restype = sz
    L.nvfp4_gemm_lora.argtypes = [tp, tp, vp, i64, i32, vp, i64, vp, i64, i64, ctypes.c_float, vp, sz, vp]
    L.nvfp4_gemm_lora.restype = i32
    L.nvfp4_gemm.restype = i32
    f32 = ctypes.c_float
    L.nvfp4_gemm_axpby.argtypes = [tp, tp, vp, i64, i32, f32, vp, i64, f32, vp, sz, vp]
    L.nvfp4_gemm_axpby.restype = i32
    L.nvfp4_newton_schulz_workspace_size.argtypes = [i64, i64]
    L.nvfp4_newton_schulz_workspace_size.restype = sz
    L.nvfp4_newton_schulz_step.argtypes = [vp, i64, i64, i64, f32, f32, f32, u16, vp, i64, vp, sz, vp]
    L.nvfp4_newton_schulz_step.restype = i32
    L.nvfp4_dequantize.argtypes = [tp, vp, i64, i32, vp]
    L.nvfp4_dequantize.restype = i32
    L.nvfp4_status_string.argtypes, L.nvfp4_status_string.restype = [i32], ctypes.c_char_p
    L.nvfp4_device_error.argtypes, L.nvfp4_device_error.restype = [vp], i32
    L.nvfp4_testing_arm_gemm_timeout.argtypes = [ctypes.c_uint32]
    L.nvfp4_testing_arm_gemm_timeout.restype = i32
    L.nvfp4_testing_bounds_violations.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    L.nvfp4_testing_bounds_violations.restype = i32
    L.nvfp4_testing_bounds_shrink.argtypes, L.nvfp4_testing_bounds_shrink.restype = [i64], i32
    _lib = L
    return L


def _ref(t):
    return None if t is None else ctypes.byref(t)


def nvfp4_scale_bytes(rows, cols):
    return load().nvfp4_scale_bytes(rows, cols)


def nvfp4_quantize_workspace_size(rows, cols, orientations):
    return load().nvfp4_quantize_workspace_size(rows, cols, orientations)


def nvfp4_quantize(x, rows, cols, ld_x, scaling, rounding, seed, stream_id, orientations,
                   out_row, out_col, workspace, workspace_bytes, stream):
    return load().nvfp4_quantize(x, rows, cols, ld_x, scaling, rounding, seed, stream_id,
                                 orientations, _ref(out_row), _ref(out_col), workspace,
                                 workspace_bytes, stream)


def nvfp4_rht_quantize(x, rows, cols, ld_x, scaling, rounding, seed, stream_id, orientations,
                       out_row, out_col, rht_sign_mask, workspace, workspace_bytes, stream):
    return load().nvfp4_rht_quantize(x, rows, cols, ld_x, scaling, rounding, seed, stream_id,
                                     orientations, _ref(out_row), _ref(out_col), rht_sign_mask,
                                     workspace, workspace_bytes, stream)


def nvfp4_quantize_noalloc(x, rows, cols, ld_x, scaling, rounding, seed, stream_id, orientations,
                           out_row, out_col, stream):
    """nvfp4_quantize without a caller-provided workspace (library-held scratch)."""
    return load().nvfp4_quantize_noalloc(x, rows, cols, ld_x, scaling, rounding, seed, stream_id,
                                         orientations, _ref(out_row), _ref(out_col), stream)


def nvfp4_quantize_row_col_rht(x, rows, cols, ld_x, rounding, seed, stream_row, stream_col, rht_sign_mask,
                               out_row, out_col, workspace, workspace_bytes, stream):
    """Row-wise without RHT and col-wise with RHT of one input, one shared amax pass."""
    return load().nvfp4_quantize_row_col_rht(x, rows, cols, ld_x, rounding, seed, stream_row, stream_col,
                                             rht_sign_mask, _ref(out_row), _ref(out_col), workspace,
                                             workspace_bytes, stream)


def nvfp4_requantize_col_rht(in_row, rounding, seed, stream_id, rht_sign_mask, out_col, workspace,
                             workspace_bytes, stream):
    """Wgrad's second operand re-quantized from a row-wise operand (Eq. (2))."""
    return load().nvfp4_requantize_col_rht(_ref(in_row), rounding, seed, stream_id, rht_sign_mask, _ref(out_col),
                                           workspace, workspace_bytes, stream)


def nvfp4_gemm(A, B, D, ldd, out_dtype, workspace, workspace_bytes, stream):
    return load().nvfp4_gemm(_ref(A), _ref(B), D, ldd, out_dtype, workspace, workspace_bytes, stream)


def nvfp4_gemm_amax(A, B, D, ldd, amax_out, rht_sign_mask, workspace, workspace_bytes, stream):
    """nvfp4_gemm (BF16 out) that also writes max |D| and the rotated amax of D."""
    return load().nvfp4_gemm_amax(_ref(A), _ref(B), D, ldd, amax_out, rht_sign_mask, workspace, workspace_bytes,
                                  stream)


def nvfp4_quantize_row_col_rht_amax(x, rows, cols, ld_x, rounding, seed, stream_row, stream_col, rht_sign_mask,
                                    amax_in, out_row, out_col, stream):
    """nvfp4_quantize_row_col_rht with the two tensor amaxes given (no amax pass)."""
    return load().nvfp4_quantize_row_col_rht_amax(x, rows, cols, ld_x, rounding, seed, stream_row, stream_col,
                                                  rht_sign_mask, amax_in, _ref(out_row), _ref(out_col), stream)


def nvfp4_gemm_lora_workspace_size(M, r):
    return load().nvfp4_gemm_lora_workspace_size(M, r)


def nvfp4_gemm_lora(A, B, D, ldd, out_dtype, U, ldu, V, ldv, r, beta, workspace, workspace_bytes, stream):
    """D = s_gA s_gB A B^T + beta U V^T (the LoRA-SVD projection's low-rank branch fused)."""
    return load().nvfp4_gemm_lora(_ref(A), _ref(B), D, ldd, out_dtype, U, ldu, V, ldv, r, beta, workspace,
                                  workspace_bytes, stream)


def nvfp4_gemm_axpby(A, B, D, ldd, out_dtype, alpha, C, ldc, beta, workspace, workspace_bytes, stream):
    """D = alpha s_gA s_gB A B^T + beta C (C of D's dtype, may be D itself)."""
    return load().nvfp4_gemm_axpby(_ref(A), _ref(B), D, ldd, out_dtype, alpha, C, ldc, beta, workspace,
                                   workspace_bytes, stream)


def nvfp4_newton_schulz_workspace_size(m, n):
    return load().nvfp4_newton_schulz_workspace_size(m, n)


def nvfp4_newton_schulz_step(X, m, n, ldx, a, b, c, rht_sign_mask, X_out, ld_out, workspace, workspace_bytes,
                             stream):
    """One NVFP4 Newton-Schulz iteration X_out = a X + b (X X^T) X + c (X X^T)^2 X with NVFP4 products."""
    return load().nvfp4_newton_schulz_step(X, m, n, ldx, a, b, c, rht_sign_mask, X_out, ld_out, workspace,
                                           workspace_bytes, stream)


def nvfp4_dequantize(q, y, ldy, out_dtype, stream):
    return load().nvfp4_dequantize(_ref(q), y, ldy, out_dtype, stream)


def nvfp4_status_string(status):
    return load().nvfp4_status_string(status).decode()


def nvfp4_device_error(stream):
    return load().nvfp4_device_error(stream)


def nvfp4_testing_arm_gemm_timeout(wait_limit_us):
    """Test support (include/nvfp4_testing.h): the next GEMM launch withholds
    one barrier arrival and gives up on its waits after wait_limit_us."""
    return load().nvfp4_testing_arm_gemm_timeout(wait_limit_us)


def nvfp4_testing_bounds_violations():
    """Test support (include/nvfp4_testing.h): (status, count of the stores the
    debug build's bounds check skipped since the last call)."""
    n = ctypes.c_uint64(0)
    st = load().nvfp4_testing_bounds_violations(ctypes.byref(n))
    return st, n.value


def nvfp4_testing_bounds_shrink(nbytes):
    """Test support (debug build): later calls declare each output buffer
    nbytes bytes shorter than it is."""
    return load().nvfp4_testing_bounds_shrink(nbytes)


def status_string(status):
    try:
        return nvfp4_status_string(status)
    except RuntimeError:
        return f"status {status}"


def check(status, what=""):
    if status != NVFP4_OK:
        raise NVFP4Error(status, what)

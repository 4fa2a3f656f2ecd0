"""CPU oracle for the NVFP4 linear-layer pipeline (ctypes front end).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only code allowed to import this module.
The product library never calls it, and it imports nothing from the product
package: the two sides share only the seeded input generators.

Arrays are numpy: bf16 inputs as uint16 bit patterns, codes and scales as
uint8 (row-major scales, one byte per 16 elements of a logical row).

Parity status of each function (see nvfp4_oracle.c for the citations):
  e2m1_rne / e2m1_sr / e2m1_value   pinned (page grid, bins, SR statistics)
  e4m3_rne_satfinite / e4m3_value    pinned (torch float8_e4m3fn casts)
  philox4x32_10 / sr_bits            round function pinned (cuRAND host
                                     generator); the counter/key placement is
                                     a documented convention
  rht16                              pinned (Sylvester recursion, H H^T = 16 I)
  tensor_scale                       pinned by its invariant (max block scale
                                     lands on 448); the formula is a reading
  quantize / amax                    pinned by invariants and special cases
  dequantize / round_bf16            pinned (grid values, torch bf16 casts)
  gemm_f64                           pinned (exact rational brute force)
  gemm_axpby_f64                     pinned (beta = 0 reduces to gemm_f64;
                                     alpha = 0 to beta * C, exactly)
  newton_schulz_step                 pinned (closed form p(s) = a s + b s^3
                                     + c s^5 on scaled partial identities,
                                     b = c = 0 gives RN(a X), distance to the
                                     unquantized polynomial on random X)
"""
import ctypes
import os

import numpy as np

from . import build as _build

ROWWISE = 1
COLWISE = 2

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u8, u16, u32, u64, i32, i64 = (ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint32,
                                       ctypes.c_uint64, ctypes.c_int, ctypes.c_int64)
        f32, f64, vp = ctypes.c_float, ctypes.c_double, ctypes.c_void_p
        L.oracle_e2m1_value.argtypes, L.oracle_e2m1_value.restype = [u8], f64
        L.oracle_e2m1_rne.argtypes, L.oracle_e2m1_rne.restype = [f32], u8
        L.oracle_e2m1_sr.argtypes, L.oracle_e2m1_sr.restype = [f32, u32], u8
        L.oracle_e4m3_value.argtypes, L.oracle_e4m3_value.restype = [u8], f64
        L.oracle_e4m3_rne_satfinite.argtypes, L.oracle_e4m3_rne_satfinite.restype = [f32], u8
        L.oracle_philox4x32_10.argtypes, L.oracle_philox4x32_10.restype = [vp, vp, vp], None
        L.oracle_sr_bits.argtypes, L.oracle_sr_bits.restype = [u64, u64, u64], u32
        L.oracle_rht16.argtypes, L.oracle_rht16.restype = [vp, u16, vp], None
        L.oracle_tensor_scale.argtypes, L.oracle_tensor_scale.restype = [f32, vp, vp], None
        L.oracle_amax.argtypes = [vp, i64, i64, i64, i32, i32, u16]
        L.oracle_amax.restype = f32
        L.oracle_quantize_rows.argtypes = [vp, i64, i64, i64, i32, i32, i32, u16, u64, u64,
                                           i32, f32, i64, i64, vp, vp]
        L.oracle_quantize_rows.restype = i32
        L.oracle_dequantize.argtypes = [vp, vp, f32, i64, i64, vp]
        L.oracle_requantize_col_rht.argtypes = [vp, vp, f32, i64, i64, i32, u16, u64, u64, f32, i64, i64,
                                                vp, vp, vp]
        L.oracle_requantize_col_rht.restype = i32
        L.oracle_dequantize.restype = None
        L.oracle_round_bf16.argtypes, L.oracle_round_bf16.restype = [f64], u16
        L.oracle_round_bf16_array.argtypes, L.oracle_round_bf16_array.restype = [vp, i64, vp], None
        L.oracle_gemm_f64.argtypes = [vp, vp, f32, vp, vp, f32, i64, i64, i64, vp, i64, vp, vp]
        L.oracle_gemm_f64.restype = None
        L.oracle_num_threads.argtypes, L.oracle_num_threads.restype = [], i32
        for name in ("oracle_e2m1_rne_array", "oracle_e4m3_rne_satfinite_array"):
            getattr(L, name).argtypes, getattr(L, name).restype = [vp, i64, vp], None
        L.oracle_e2m1_sr_array.argtypes = [vp, vp, i64, vp]
        L.oracle_e2m1_sr_array.restype = None
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar primitives -------------------------------------------------
def e2m1_value(code):
    return lib().oracle_e2m1_value(int(code))


def e2m1_rne(v):
    return lib().oracle_e2m1_rne(float(v))


def e2m1_sr(v, rand16):
    return lib().oracle_e2m1_sr(float(v), int(rand16))


def e4m3_value(code):
    return lib().oracle_e4m3_value(int(code))


def e4m3_rne_satfinite(x):
    return lib().oracle_e4m3_rne_satfinite(float(x))


def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits(seed, stream_id, idx):
    return lib().oracle_sr_bits(int(seed), int(stream_id), int(idx))


def rht16(x, sign_mask):
    xx = _c(x, np.float32)
    assert xx.shape == (16,)
    y = np.zeros(16, np.float32)
    lib().oracle_rht16(_ptr(xx), int(sign_mask), _ptr(y))
    return y


def tensor_scale(amax):
    s_enc = ctypes.c_float()
    s_g = ctypes.c_float()
    lib().oracle_tensor_scale(float(np.float32(amax)), ctypes.byref(s_enc), ctypes.byref(s_g))
    return np.float32(s_enc.value), np.float32(s_g.value)


def e2m1_rne_array(v):
    vv = _c(v, np.float32).ravel()
    out = np.zeros(vv.shape, np.uint8)
    lib().oracle_e2m1_rne_array(_ptr(vv), vv.size, _ptr(out))
    return out


def e2m1_sr_array(v, words):
    vv = _c(v, np.float32).ravel()
    ww = _c(words, np.uint32).ravel()
    assert vv.shape == ww.shape
    out = np.zeros(vv.shape, np.uint8)
    lib().oracle_e2m1_sr_array(_ptr(vv), _ptr(ww), vv.size, _ptr(out))
    return out


def e4m3_rne_satfinite_array(x):
    xx = _c(x, np.float32).ravel()
    out = np.zeros(xx.shape, np.uint8)
    lib().oracle_e4m3_rne_satfinite_array(_ptr(xx), xx.size, _ptr(out))
    return out


def round_bf16(v):
    return lib().oracle_round_bf16(float(v))


def round_bf16_array(v):
    """float64 array -> bf16 bit patterns (uint16), each rounded once."""
    vv = _c(v, np.float64)
    out = np.zeros(vv.shape, np.uint16)
    lib().oracle_round_bf16_array(_ptr(vv), vv.size, _ptr(out))
    return out


def bf16_to_f64(bits):
    """bf16 bit patterns -> float64 values (exact)."""
    return (_c(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def num_threads():
    return lib().oracle_num_threads()


# ---- tensor operations -------------------------------------------------
def amax(x_bits, orientation=ROWWISE, use_rht=False, sign_mask=0):
    """Tensor amax of the values one orientation encodes (float32)."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    return np.float32(lib().oracle_amax(_ptr(x), rows, cols, cols, orientation,
                                        int(bool(use_rht)), int(sign_mask)))


def quantize(x_bits, orientation=ROWWISE, scaling=0, rounding=0, use_rht=False,
             sign_mask=0, seed=0, stream_id=0, rows_subset=None, amax_value=None):
    """Quantize one orientation of x (bf16 bit patterns, [rows][cols]).

    Returns dict(codes, scales, amax, s_enc, s_g, rows) where codes/scales
    cover the logical rows in ``rows`` (all logical rows by default; a
    contiguous range (lr0, lr1) when ``rows_subset`` is given).  The tensor
    amax is computed by the oracle over the full tensor unless ``amax_value``
    gives it (a shard of a larger tensor quantized with the amax that the
    shards agreed on).
    """
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    lrows, lcols = (rows, cols) if orientation == ROWWISE else (cols, rows)
    if amax_value is None:
        amax_value = amax(x, orientation, use_rht, sign_mask)
    lr0, lr1 = (0, lrows) if rows_subset is None else rows_subset
    n = lr1 - lr0
    codes = np.zeros((n, lcols // 2), np.uint8)
    scales = np.zeros((n, lcols // 16), np.uint8)
    rc = lib().oracle_quantize_rows(_ptr(x), rows, cols, cols, int(scaling), int(rounding),
                                    int(bool(use_rht)), int(sign_mask), int(seed),
                                    int(stream_id), int(orientation), float(amax_value),
                                    lr0, lr1, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError(f"oracle_quantize_rows rejected the arguments (code {rc})")
    s_enc, s_g = tensor_scale(amax_value)
    return dict(codes=codes, scales=scales, amax=np.float32(amax_value), s_enc=s_enc,
                s_g=s_g, rows=(lr0, lr1))


def requantize_col_rht(q_row, sign_mask, rounding=0, seed=0, stream_id=0, rows_subset=None,
                       amax_value=None):
    """Wgrad's second operand from a row-wise operand (a dict from quantize()):
    dequantize, RHT along the rows, col-wise 1x16 quantization ("Full-Stack
    FP4", Sec. 3.2 Eq. (2)).  Returns the same dict as quantize() for the
    [cols][rows] output."""
    codes = _c(q_row["codes"], np.uint8)
    scales = _c(q_row["scales"], np.uint8)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    lr0, lr1 = (0, cols) if rows_subset is None else rows_subset
    n = lr1 - lr0
    out_codes = np.zeros((n, rows // 2), np.uint8)
    out_scales = np.zeros((n, rows // 16), np.uint8)
    amax_out = np.zeros(1, np.float32)
    rc = lib().oracle_requantize_col_rht(_ptr(codes), _ptr(scales), float(q_row["s_g"]), rows, cols,
                                         int(rounding), int(sign_mask), int(seed), int(stream_id),
                                         -1.0 if amax_value is None else float(amax_value), lr0, lr1,
                                         _ptr(out_codes), _ptr(out_scales), _ptr(amax_out))
    if rc != 0:
        raise ValueError(f"oracle_requantize_col_rht rejected the arguments (code {rc})")
    s_enc, s_g = tensor_scale(amax_out[0])
    return dict(codes=out_codes, scales=out_scales, amax=np.float32(amax_out[0]), s_enc=s_enc, s_g=s_g,
                rows=(lr0, lr1))


def dequantize(codes, scales, s_g):
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint8)
    rows = c.shape[0]
    cols = c.shape[1] * 2
    assert s.shape == (rows, cols // 16)
    out = np.zeros((rows, cols), np.float64)
    lib().oracle_dequantize(_ptr(c), _ptr(s), float(s_g), rows, cols, _ptr(out))
    return out


def gemm_lora_f64(a, b, u_bits, v_bits, beta, row_ids=None):
    """The LoRA-SVD projection of "Full-Stack FP4", Sec. 3.2 Eq. (1):
    y = A * B^T (gemm_f64, the NVFP4 GEMM) + beta * U V^T (the BF16 low-rank
    branch, U = [M][r] and V = [N][r] bf16 bit patterns), in float64.
    Returns (y, abs_sum, lora_abs_sum): the sums of |a b| and of |beta u v|
    over the reduction, for tolerances."""
    y, ab = gemm_f64(a, b, row_ids=row_ids)
    u = (np.ascontiguousarray(u_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = (np.ascontiguousarray(v_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if row_ids is not None:
        u = u[np.asarray(row_ids)]
    lora = float(beta) * (u @ v.T)
    lora_abs = abs(float(beta)) * (np.abs(u) @ np.abs(v).T)
    return y + lora, ab, lora_abs


def gemm_f64(a, b, row_ids=None, with_abs=True):
    """y = A * B^T for two oracle-quantized operands (dicts from quantize()).

    Returns (y, abs_sum) in float64 for the listed rows of A (all by default).
    """
    ac, as_ = _c(a["codes"], np.uint8), _c(a["scales"], np.uint8)
    bc, bs = _c(b["codes"], np.uint8), _c(b["scales"], np.uint8)
    M, K = ac.shape[0], ac.shape[1] * 2
    N = bc.shape[0]
    assert bc.shape[1] * 2 == K
    ids = None if row_ids is None else _c(row_ids, np.int64)
    nr = M if ids is None else ids.shape[0]
    y = np.zeros((nr, N), np.float64)
    ab = np.zeros((nr, N), np.float64) if with_abs else None
    lib().oracle_gemm_f64(_ptr(ac), _ptr(as_), float(a["s_g"]), _ptr(bc), _ptr(bs),
                          float(b["s_g"]), M, N, K, _ptr(ids), nr, _ptr(y), _ptr(ab))
    return y, ab


def gemm_axpby_f64(a, b, alpha, c_bits, beta, row_ids=None):
    """y = alpha * A B^T + beta * C in float64: the GEMM of two oracle-quantized
    operands (gemm_f64) combined with a bf16 matrix C ([M][N] bit patterns, or
    None for beta = 0), as the Newton-Schulz iteration of "Full-Stack FP4",
    Sec. 3.4 combines b A_k + c (qA_k qA_k^16x1) and a X_k + qB_k qX_k^16x1.
    Returns (y, abs_sum): abs_sum = |alpha| sum_k |a_k b_k| + |beta c|, the
    magnitude a tolerance scales with."""
    y, ab = gemm_f64(a, b, row_ids=row_ids)
    y = float(alpha) * y
    ab = abs(float(alpha)) * ab
    if c_bits is not None and float(beta) != 0.0:
        c = bf16_to_f64(c_bits)
        if row_ids is not None:
            c = c[np.asarray(row_ids)]
        y = y + float(beta) * c
        ab = ab + abs(float(beta)) * np.abs(c)
    return y, ab


def newton_schulz_step(x_bits, a, b, c, sign_mask):
    """One NVFP4 Newton-Schulz iteration of the Root optimizer ("Full-Stack
    FP4", Sec. 3.4, the quantized NS iteration):

        qX  = Q_1x16(X H),        A  = qX qX^T
        qA  = Q_1x16(A H),        qA' = Q_16x1(H^T A),   B = b A + c qA qA'
        qB  = Q_1x16(B H),        qX' = Q_16x1(H^T X),   X_next = a X + qB qX'

    X is bf16 [m][n] (bit patterns).  Every quantization is RTN with 4/6
    scaling (the page: "all NVFP4 quantizations adopt RTN and 4/6 scaling");
    H = H16 diag(sign_mask) / 4 along each product's reduction dimension, one
    mask for the whole step so that H H^T = I cancels in each product.  The
    page leaves the storage of A, B and X_next open; here each is a bf16
    tensor rounded once from its float64 value, and (a, b, c) are binary32
    inputs (the page's shape-optimised coefficients are not printed).

    Returns a dict of the intermediate and final tensors: qX, A (bf16 bits),
    qA, qAc, B (bf16 bits), qB, qXc, X (bf16 bits of X_next).
    """
    x_bits = _c(x_bits, np.uint16)
    a, b, c = (float(np.float32(v)) for v in (a, b, c))   # binary32, as the library takes them
    q = lambda t, o: quantize(t, o, scaling=2, rounding=0, use_rht=True, sign_mask=sign_mask)
    qX = q(x_bits, ROWWISE)
    A = round_bf16_array(gemm_f64(qX, qX, with_abs=False)[0])
    qA, qAc = q(A, ROWWISE), q(A, COLWISE)
    B = round_bf16_array(gemm_axpby_f64(qA, qAc, c, A, b)[0])
    qB, qXc = q(B, ROWWISE), q(x_bits, COLWISE)
    X = round_bf16_array(gemm_axpby_f64(qB, qXc, 1.0, x_bits, a)[0])
    return dict(qX=qX, A=A, qA=qA, qAc=qAc, B=B, qB=qB, qXc=qXc, X=X)

"""CPU-side checks of the C ABI: the library loads, exports every entry point
include/nvfp4.h declares, and its host-side validation rejects bad arguments
before any CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi
from tests import helpers

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return capi.load()


def declared_functions():
    """Every entry point the headers in include/ declare."""
    names = set()
    for h in HEADERS:
        names |= set(re.findall(r"NVFP4_API\s+[\w\s\*]+?\b(nvfp4_\w+)\s*\(", open(h).read()))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("nvfp4_quantize", "nvfp4_rht_quantize", "nvfp4_gemm", "nvfp4_dequantize"):
        assert required in names
    assert set(names) == set(capi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_testing_arm_rejects_limits_out_of_range(lib):
    # valid limits arm a fault for the next GEMM launch; only the rejections
    # are exercised here (no GEMM runs on the CPU)
    for us in (0, 999, 2000001, 2 ** 32 - 1):
        assert capi.nvfp4_testing_arm_gemm_timeout(us) == capi.NVFP4_ERR_INVALID_ARG


def test_bounds_check_entry_points_are_debug_only(lib):
    """The regular build has no bounds check: both test-support calls say so
    without touching the GPU."""
    st, _ = capi.nvfp4_testing_bounds_violations()
    assert st == capi.NVFP4_ERR_UNSUPPORTED
    assert capi.nvfp4_testing_bounds_shrink(16) == capi.NVFP4_ERR_UNSUPPORTED


def test_quantize_workspace_is_the_documented_32_kib(lib):
    # the no-allocation quantizer's library-held scratch is 32 KiB: the
    # workspace every shape asks for must not outgrow it
    for rows, cols, orient in ((16, 16, 1), (8192, 3072, 3), (65536, 8192, 2)):
        assert capi.nvfp4_quantize_workspace_size(rows, cols, orient) == 32 * 1024


def test_status_strings(lib):
    for code in range(8):
        assert capi.nvfp4_status_string(code).startswith("NVFP4_")
    assert capi.nvfp4_status_string(0) == "NVFP4_OK"
    assert capi.nvfp4_status_string(99) == "NVFP4_ERR_UNKNOWN"


@pytest.mark.parametrize("rows,cols", [(1, 16), (128, 64), (129, 64), (128, 65 * 16), (8192, 3072),
                                       (16384, 9216), (0, 64), (7, 0)])
def test_scale_bytes_match_documented_layout(lib, rows, cols):
    assert capi.nvfp4_scale_bytes(rows, cols) == helpers.scale_bytes(rows, cols)


@pytest.mark.parametrize("rows,cols", [(1, 16), (200, 48), (384, 1024), (130, 80)])
def test_scale_layout_is_a_bijection_into_the_buffer(rows, cols):
    m = helpers.scale_index_map(rows, cols)
    assert m.min() >= 0 and m.max() < helpers.scale_bytes(rows, cols)
    assert np.unique(m).size == m.size


# ---- host-side validation (returns before any CUDA call) -------------------
A16 = 1 << 20      # fake, 16-byte aligned "device" addresses: never dereferenced


def tensor(rows, cols, ld=None, codes=A16, scales=A16 * 2, sg=A16 * 3):
    return capi.nvfp4_tensor(codes, scales, 0, sg, rows, cols,
                             ld if ld is not None else max(16, (cols // 2 + 15) // 16 * 16))


def quantize(**kw):
    args = dict(x=A16 * 4, rows=64, cols=64, ld_x=64, scaling=0, rounding=0, seed=0, stream_id=0,
                orientations=1, out_row=tensor(64, 64), out_col=tensor(64, 64),
                workspace=A16 * 5, workspace_bytes=capi.nvfp4_quantize_workspace_size(64, 64, 3),
                stream=None)
    args.update(kw)
    return capi.nvfp4_quantize(*args.values())


def test_quantize_validation(lib):
    E = capi
    assert quantize(cols=40, out_row=tensor(64, 40)) == E.NVFP4_ERR_SHAPE           # cols % 16
    assert quantize(orientations=2, rows=24, out_col=tensor(64, 24)) == E.NVFP4_ERR_SHAPE
    assert quantize(scaling=1, rows=24, out_row=tensor(24, 64)) == E.NVFP4_ERR_SHAPE
    assert quantize(x=A16 + 8) == E.NVFP4_ERR_ALIGNMENT
    assert quantize(ld_x=68) == E.NVFP4_ERR_ALIGNMENT
    assert quantize(ld_x=48) == E.NVFP4_ERR_SHAPE
    assert quantize(x=None) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(orientations=0) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(orientations=4) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(scaling=3) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(scaling=2, orientations=2, rows=24, out_col=tensor(64, 24)) == E.NVFP4_ERR_SHAPE   # 4/6 is 1x16
    assert quantize(rounding=5) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(out_row=None) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(out_row=tensor(64, 32)) == E.NVFP4_ERR_INVALID_ARG               # wrong shape
    assert quantize(orientations=2, out_col=tensor(32, 64)) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(out_row=tensor(64, 64, sg=0)) == E.NVFP4_ERR_INVALID_ARG
    assert quantize(out_row=tensor(64, 64, ld=24)) == E.NVFP4_ERR_SHAPE               # ld < cols/2
    assert quantize(out_row=tensor(64, 64, ld=40)) == E.NVFP4_ERR_ALIGNMENT
    assert quantize(out_row=tensor(64, 64, codes=A16 + 4)) == E.NVFP4_ERR_ALIGNMENT
    assert quantize(out_row=tensor(64, 64, scales=A16 + 1)) == E.NVFP4_ERR_ALIGNMENT
    assert quantize(workspace=None) == E.NVFP4_ERR_WORKSPACE
    assert quantize(workspace_bytes=16) == E.NVFP4_ERR_WORKSPACE
    assert quantize(rows=-1) == E.NVFP4_ERR_SHAPE


def row_col_rht(**kw):
    args = dict(x=A16 * 4, rows=64, cols=96, ld_x=96, rounding=0, seed=0, stream_row=0, stream_col=1,
                rht_sign_mask=0x1234, out_row=tensor(64, 96), out_col=tensor(96, 64),
                workspace=A16 * 5, workspace_bytes=capi.nvfp4_quantize_workspace_size(64, 96, 3), stream=None)
    args.update(kw)
    return capi.nvfp4_quantize_row_col_rht(*args.values())


def test_row_col_rht_validation(lib):
    E = capi
    assert row_col_rht(rows=24, out_col=tensor(96, 24)) == E.NVFP4_ERR_SHAPE        # rows % 16 (col-wise)
    assert row_col_rht(cols=40, ld_x=40) == E.NVFP4_ERR_SHAPE                        # cols % 16
    assert row_col_rht(rounding=3) == E.NVFP4_ERR_INVALID_ARG
    assert row_col_rht(out_row=None) == E.NVFP4_ERR_INVALID_ARG                      # both outputs required
    assert row_col_rht(out_col=None) == E.NVFP4_ERR_INVALID_ARG
    assert row_col_rht(out_col=tensor(64, 96)) == E.NVFP4_ERR_INVALID_ARG            # transposed shape expected
    assert row_col_rht(x=A16 + 8) == E.NVFP4_ERR_ALIGNMENT
    assert row_col_rht(x=None) == E.NVFP4_ERR_INVALID_ARG
    assert row_col_rht(workspace_bytes=16) == E.NVFP4_ERR_WORKSPACE
    assert row_col_rht(rows=-16) == E.NVFP4_ERR_SHAPE


def requant(**kw):
    args = dict(in_row=tensor(64, 96, codes=A16 * 6, scales=A16 * 7, sg=A16 * 8), rounding=0, seed=0,
                stream_id=0, mask=0x1234, out_col=tensor(96, 64), workspace=A16 * 5,
                workspace_bytes=capi.nvfp4_quantize_workspace_size(64, 96, 3), stream=None)
    args.update(kw)
    return capi.nvfp4_requantize_col_rht(*args.values())


def test_requantize_validation(lib):
    """Every call here is rejected on the host (no kernel ever sees the fake addresses)."""
    E = capi
    assert requant(in_row=None) == E.NVFP4_ERR_INVALID_ARG
    assert requant(out_col=None) == E.NVFP4_ERR_INVALID_ARG
    assert requant(rounding=2) == E.NVFP4_ERR_INVALID_ARG
    assert requant(in_row=tensor(24, 96, codes=A16 * 6, scales=A16 * 7, sg=A16 * 8),
                   out_col=tensor(96, 24)) == E.NVFP4_ERR_SHAPE                      # rows % 16
    assert requant(out_col=tensor(64, 96)) == E.NVFP4_ERR_INVALID_ARG                 # transposed shape expected
    assert requant(out_col=tensor(96, 64, sg=A16 * 8)) == E.NVFP4_ERR_INVALID_ARG     # shares s_g with the input
    assert requant(out_col=tensor(96, 64, codes=A16 * 6)) == E.NVFP4_ERR_INVALID_ARG  # shares codes
    assert requant(in_row=tensor(64, 96, codes=A16 + 8, scales=A16 * 7, sg=A16 * 8)) == E.NVFP4_ERR_ALIGNMENT
    assert requant(workspace_bytes=16) == E.NVFP4_ERR_WORKSPACE


def gemm_lora(**kw):
    args = dict(A=tensor(64, 128), B=tensor(96, 128), D=A16 * 9, ldd=96, out_dtype=0, U=A16 * 10, ldu=64,
                V=A16 * 11, ldv=64, r=64, beta=0.5, workspace=A16 * 12,
                workspace_bytes=capi.nvfp4_gemm_lora_workspace_size(64, 64), stream=None)
    args.update(kw)
    return capi.nvfp4_gemm_lora(*args.values())


def test_gemm_lora_validation(lib):
    """Every call here is rejected on the host (no kernel ever sees the fake addresses)."""
    E = capi
    assert gemm_lora(r=32, ldu=32, ldv=32) == E.NVFP4_ERR_UNSUPPORTED                # r % 64
    assert gemm_lora(r=0) == E.NVFP4_ERR_UNSUPPORTED
    assert gemm_lora(ldu=32) == E.NVFP4_ERR_SHAPE                                     # ldu < r
    assert gemm_lora(U=A16 + 8) == E.NVFP4_ERR_ALIGNMENT
    assert gemm_lora(ldv=68) == E.NVFP4_ERR_ALIGNMENT                                 # ldv % 8
    assert gemm_lora(U=None) == E.NVFP4_ERR_INVALID_ARG
    assert gemm_lora(beta=float("nan")) == E.NVFP4_ERR_INVALID_ARG
    assert gemm_lora(workspace_bytes=16) == E.NVFP4_ERR_WORKSPACE
    assert gemm_lora(A=tensor(64, 0), B=tensor(96, 0)) == E.NVFP4_ERR_UNSUPPORTED     # K = 0
    assert gemm_lora(B=tensor(96, 64)) == E.NVFP4_ERR_SHAPE                           # K mismatch
    assert capi.nvfp4_gemm_lora_workspace_size(100, 64) >= 100 * 64 * 2


def test_fused_amax_validation(lib):
    """Rejected on the host (no kernel ever sees the fake addresses)."""
    E = capi
    ws = None
    assert capi.nvfp4_gemm_amax(tensor(24, 128), tensor(96, 128), A16 * 9, 96, A16 * 13, 0x1234, ws, 0,
                                None) == E.NVFP4_ERR_SHAPE                                      # M % 16
    assert capi.nvfp4_gemm_amax(tensor(64, 128), tensor(96, 128), A16 * 9 + 8, 96, A16 * 13, 0x1234, ws, 0,
                                None) == E.NVFP4_ERR_ALIGNMENT
    assert capi.nvfp4_gemm_amax(tensor(64, 128), tensor(96, 128), A16 * 9, 100, A16 * 13, 0x1234, ws, 0,
                                None) == E.NVFP4_ERR_ALIGNMENT                                  # ldd % 8
    assert capi.nvfp4_gemm_amax(tensor(64, 128), tensor(96, 128), A16 * 9, 96, None, 0x1234, ws, 0,
                                None) == E.NVFP4_ERR_INVALID_ARG
    q = capi.nvfp4_quantize_row_col_rht_amax
    assert q(A16 * 4, 64, 64, 64, 0, 0, 0, 0, 0x1234, None, tensor(64, 64), tensor(64, 64),
             None) == E.NVFP4_ERR_INVALID_ARG                                                   # amax_in
    assert q(A16 * 4, 24, 64, 64, 0, 0, 0, 0, 0x1234, A16 * 13, tensor(24, 64), tensor(64, 24),
             None) == E.NVFP4_ERR_SHAPE
    assert q(A16 * 4, 64, 64, 64, 7, 0, 0, 0, 0x1234, A16 * 13, tensor(64, 64), tensor(64, 64),
             None) == E.NVFP4_ERR_INVALID_ARG


def test_rht_quantize_rejects_2d(lib):
    ws = capi.nvfp4_quantize_workspace_size(64, 64, 3)
    st = capi.nvfp4_rht_quantize(A16 * 4, 64, 64, 64, capi.NVFP4_SCALE_16X16, 0, 0, 0, 1,
                                 tensor(64, 64), None, 0x1234, A16 * 5, ws, None)
    assert st == capi.NVFP4_ERR_UNSUPPORTED


def test_gemm_validation(lib):
    E = capi

    def gemm(A=None, B=None, D=A16 * 6, ldd=128, dt=0):
        A = A if A is not None else tensor(128, 256)
        B = B if B is not None else tensor(128, 256)
        return capi.nvfp4_gemm(A, B, D, ldd, dt, None, 0, None)

    assert gemm(B=tensor(128, 128)) == E.NVFP4_ERR_SHAPE            # K mismatch
    assert gemm(A=tensor(128, 40, ld=32), B=tensor(128, 40, ld=32)) == E.NVFP4_ERR_SHAPE
    assert gemm(D=None) == E.NVFP4_ERR_INVALID_ARG
    assert gemm(D=A16 + 1) == E.NVFP4_ERR_ALIGNMENT                 # bf16 needs 2-byte alignment
    assert gemm(D=A16 + 2, dt=1) == E.NVFP4_ERR_ALIGNMENT           # fp32 needs 4-byte alignment
    assert gemm(ldd=100) == E.NVFP4_ERR_SHAPE                       # ldd < N
    assert gemm(dt=7) == E.NVFP4_ERR_INVALID_ARG
    assert gemm(A=tensor(128, 256, codes=0)) == E.NVFP4_ERR_INVALID_ARG
    assert gemm(A=tensor(128, 256, ld=120)) == E.NVFP4_ERR_SHAPE
    assert gemm(A=tensor(128, 256, ld=136)) == E.NVFP4_ERR_ALIGNMENT
    # empty outputs are a no-op and touch nothing
    assert gemm(A=tensor(0, 256)) == E.NVFP4_OK


def test_gemm_axpby_validation(lib):
    E = capi

    def axpby(A=None, B=None, D=A16 * 6, ldd=128, dt=0, alpha=1.0, C=A16 * 7, ldc=128, beta=0.5):
        A = A or tensor(128, 256)
        B = B or tensor(128, 256)
        return capi.nvfp4_gemm_axpby(A, B, D, ldd, dt, alpha, C, ldc, beta, None, 0, None)
    assert axpby(alpha=float("nan")) == E.NVFP4_ERR_INVALID_ARG
    assert axpby(beta=float("inf")) == E.NVFP4_ERR_INVALID_ARG
    assert axpby(C=None) == E.NVFP4_ERR_INVALID_ARG                  # beta != 0 reads C
    assert axpby(ldc=100) == E.NVFP4_ERR_SHAPE                       # ldc < N
    assert axpby(C=A16 * 7 + 1) == E.NVFP4_ERR_ALIGNMENT
    assert axpby(C=A16 * 6, ldc=136) == E.NVFP4_ERR_INVALID_ARG      # C == D needs the same ld
    assert axpby(B=tensor(128, 128)) == E.NVFP4_ERR_SHAPE            # K mismatch
    assert axpby(A=tensor(128, 0), B=tensor(128, 0)) == E.NVFP4_ERR_UNSUPPORTED   # K = 0
    assert axpby(dt=3) == E.NVFP4_ERR_INVALID_ARG
    assert axpby(A=tensor(0, 256)) == E.NVFP4_OK                     # empty output: nothing enqueued


def test_newton_schulz_validation(lib):
    E = capi
    ws_bytes = capi.nvfp4_newton_schulz_workspace_size(64, 128)
    assert ws_bytes > 2 * (2 * 64 * 64)   # A and B, then the quantized operands
    assert capi.nvfp4_newton_schulz_workspace_size(0, 128) == 0

    def ns(X=A16 * 4, m=64, n=128, ldx=128, a=1.5, b=-0.5, c=0.0, out=A16 * 8, ld_out=128,
           ws=A16 * 9, ws_bytes=ws_bytes):
        return capi.nvfp4_newton_schulz_step(X, m, n, ldx, a, b, c, 0x1234, out, ld_out, ws, ws_bytes, None)
    assert ns(m=40) == E.NVFP4_ERR_SHAPE
    assert ns(n=72, ldx=72, ld_out=72) == E.NVFP4_ERR_SHAPE
    assert ns(m=0) == E.NVFP4_ERR_SHAPE
    assert ns(a=float("nan")) == E.NVFP4_ERR_INVALID_ARG
    assert ns(X=None) == E.NVFP4_ERR_INVALID_ARG
    assert ns(X=A16 * 4 + 8) == E.NVFP4_ERR_ALIGNMENT
    assert ns(ldx=100) == E.NVFP4_ERR_SHAPE
    assert ns(ldx=132) == E.NVFP4_ERR_ALIGNMENT
    assert ns(out=A16 * 4, ld_out=136) == E.NVFP4_ERR_INVALID_ARG    # in place needs the same ld
    assert ns(ws=None) == E.NVFP4_ERR_WORKSPACE
    assert ns(ws_bytes=ws_bytes - 1) == E.NVFP4_ERR_WORKSPACE
    assert ns(ws=A16 * 9 + 8) == E.NVFP4_ERR_WORKSPACE


def test_dequantize_validation(lib):
    E = capi
    q = tensor(64, 64)
    assert capi.nvfp4_dequantize(q, None, 64, 0, None) == E.NVFP4_ERR_INVALID_ARG
    assert capi.nvfp4_dequantize(q, A16 + 2, 64, 0, None) == E.NVFP4_ERR_ALIGNMENT
    assert capi.nvfp4_dequantize(q, A16, 32, 0, None) == E.NVFP4_ERR_SHAPE
    assert capi.nvfp4_dequantize(q, A16, 68, 0, None) == E.NVFP4_ERR_ALIGNMENT
    assert capi.nvfp4_dequantize(q, A16, 64, 3, None) == E.NVFP4_ERR_INVALID_ARG


def test_product_path_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _fresh_load(str(tmp_path / "missing.so"))


def _fresh_load(path):
    saved = capi._lib
    capi._lib = None
    try:
        return capi.load(path)
    finally:
        capi._lib = saved

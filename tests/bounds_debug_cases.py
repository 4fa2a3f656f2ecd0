"""The library's debug build (NVFP4_BOUNDS_CHECK) on a GPU: run by
tests/test_gpu_bounds_debug.py in a process of its own, so that the debug
library is the only one loaded here.

1. Every entry point, on small ragged shapes in every mode, leaves the bounds
   check's count at zero, and the debug build's results equal the oracle's.
2. With every declared output range shortened by 16 bytes (test support,
   nothing outside any allocation is touched), the check fires: the stores
   that reach into the last 16 bytes are skipped and counted, those bytes
   keep their fill, and every other byte equals the full-range result.
Exits 0 when all holds, 1 (with the reason) otherwise.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from fp4_gemm_nvfp4_gb300 import build, capi  # noqa: E402
from fp4_gemm_nvfp4_gb300 import inputs, ops  # noqa: E402
from tests import helpers  # noqa: E402

FILL = 0x5A


def violations():
    st, n = capi.nvfp4_testing_bounds_violations()
    assert st == capi.NVFP4_OK, capi.status_string(st)
    return n


def expect_clean(what):
    n = violations()
    assert n == 0, f"{what}: {n} stores outside the declared ranges"


def filled_operand(rows, cols):
    op = ops.alloc_operand(rows, cols)
    op.codes.fill_(FILL)
    op.scales.fill_(FILL)
    return op


def check_modes():
    rng_shapes = [(272, 336), (560, 96), (48, 64)]
    for rows, cols in rng_shapes:
        bits = inputs.student_t(rows, cols, rows + cols)
        x = helpers.to_device_bf16(bits)
        for kw in (dict(), dict(sr=True, seed=3), dict(rht_mask=0x1F2E), dict(two_d=True), dict(scale46=True),
                   dict(rht_mask=0x0F0F, sr=True, seed=5, scale46=True)):
            for rowwise, colwise in ((True, False), (False, True), (True, True)):
                ops.quantize(x, rowwise=rowwise, colwise=colwise, **kw)
                torch.cuda.synchronize()
                expect_clean(f"quantize {rows}x{cols} {kw} row={rowwise} col={colwise}")
        row, col = ops.quantize_row_col_rht(x, 0x3333, sr=True, seed=1, stream_row=1, stream_col=2)
        amax = torch.stack([row.amax[0], col.amax[0]]).contiguous()
        ops.quantize_row_col_rht_amax(x, 0x3333, amax)
        ops.requantize_col_rht(row, 0x0F0F, sr=True, seed=2)
        torch.cuda.synchronize()
        expect_clean(f"pair / requantize {rows}x{cols}")
        # the debug build computes what the oracle does
        codes, scales, amax_g, sg, _ = helpers.operand_to_host(row)
        ref = oracle.quantize(bits, oracle.ROWWISE, rounding=1, seed=1, stream_id=1)
        assert np.array_equal(codes, ref["codes"]) and np.array_equal(scales, ref["scales"]), "codes differ"
        for dtype in (torch.bfloat16, torch.float32):
            ops.dequantize(row, dtype)
        torch.cuda.synchronize()
        expect_clean(f"dequantize {rows}x{cols}")
    for M, N, K in ((200, 300, 320), (256, 512, 1024), (130, 260, 80), (96, 271, 64)):
        a = ops.alloc_operand(M, K)
        b = ops.alloc_operand(N, K)
        g = torch.Generator(device="cuda")
        g.manual_seed(M + N + K)
        for op in (a, b):
            op.codes.copy_(torch.randint(0, 256, op.codes.shape, generator=g, device="cuda",
                                         dtype=torch.int32).to(torch.uint8))
            op.scales.copy_(torch.randint(0x20, 0x48, op.scales.shape, generator=g, device="cuda",
                                          dtype=torch.int32).to(torch.uint8))
            op.global_scale.fill_(1.0)
        for dtype in (torch.bfloat16, torch.float32):
            for pad in (0, 3, 8):   # 3: rows off 16 bytes, the epilogue's direct stores
                d = torch.empty((M, N + pad), dtype=dtype, device="cuda")[:, :N]
                ops.gemm(a, b, out_dtype=dtype, out=d)
                c = torch.randn((M, N), device="cuda").to(dtype)
                ops.gemm_axpby(a, b, 0.5, c, 2.0, out=d)
        if M % 16 == 0 and N % 8 == 0:
            ops.gemm_amax(a, b, 0x1234)
        # rows on 16 bytes with N off a 16-byte multiple: TMA stores up to the
        # last whole piece, the lanes' stores after it
        ldt = (N + 7) // 8 * 8 + 8
        for dtype in (torch.bfloat16, torch.float32):
            d = torch.empty((M, ldt), dtype=dtype, device="cuda")[:, :N]
            ops.gemm(a, b, out_dtype=dtype, out=d)
            # C on 16-byte rows as well: copied into the epilogue's slices
            c = torch.randn((M, ldt), device="cuda").to(dtype)[:, :N]
            ops.gemm_axpby(a, b, 0.5, c, 2.0, out=d)
        if M % 16 == 0:
            ops.gemm_amax(a, b, 0x1234, out=torch.empty((M, ldt), dtype=torch.bfloat16, device="cuda")[:, :N])
        torch.cuda.synchronize()
        assert ops.device_error() == capi.NVFP4_OK
        expect_clean(f"gemm {M}x{N}x{K}")


def check_the_check():
    rows, cols, shrink = 272, 336, 16
    x = helpers.to_device_bf16(inputs.normal(rows, cols, 7))
    full = filled_operand(rows, cols)
    ops.quantize(x, out_row=full)
    torch.cuda.synchronize()
    expect_clean("full-range quantize")
    assert capi.nvfp4_testing_bounds_shrink(shrink) == capi.NVFP4_OK
    try:
        part = filled_operand(rows, cols)
        ops.quantize(x, out_row=part)
        torch.cuda.synchronize()
        n = violations()
    finally:
        assert capi.nvfp4_testing_bounds_shrink(0) == capi.NVFP4_OK
    # the codes' declared range ends after byte cols / 2 of the last row
    ld = full.codes.shape[1]
    end = (rows - 1) * ld + cols // 2
    a = full.codes.cpu().numpy().reshape(-1)
    b = part.codes.cpu().numpy().reshape(-1)
    assert n > 0, "the shortened range produced no skipped store"
    cut = np.zeros(a.shape, bool)
    cut[end - shrink:end] = True
    assert (b[cut] == FILL).all(), "a store reached into the withdrawn bytes"
    assert np.array_equal(a[~cut], b[~cut]), "bytes outside the withdrawn range differ"
    # the skipped stores are the 8-byte block stores that reach into them
    assert n >= shrink // 8, n


def main():
    lib = build.build(debug=True)
    capi.load(lib)
    st, n = capi.nvfp4_testing_bounds_violations()
    assert st == capi.NVFP4_OK and n == 0, (st, n)
    check_modes()
    check_the_check()
    print("bounds check: clean in every mode, fires on a shortened range")


if __name__ == "__main__":
    try:
        main()
    except AssertionError as e:
        print(f"FAILED: {e}")
        sys.exit(1)

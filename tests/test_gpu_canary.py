"""Canary-guarded outputs: every entry point writes inside its outputs and
nowhere else.  Each output buffer sits inside a larger allocation whose
guard zones (before, after, and the row padding between the written bytes
and the leading dimension) hold a byte pattern, checked after the call."""
import numpy as np
import pytest
import torch

from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
from tests import helpers

pytestmark = pytest.mark.gpu

CANARY = 0xA5
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


class Guarded:
    """A byte buffer of `n` usable bytes (16-byte aligned) between two guard
    zones, all filled with the canary."""

    def __init__(self, n):
        self.n = n
        self.raw = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.body = self.raw[GUARD:GUARD + n]

    def guards_intact(self):
        h = self.raw.cpu().numpy()
        return bool((h[:GUARD] == CANARY).all() and (h[GUARD + self.n:] == CANARY).all())


def guarded_operand(rows, cols, extra_ld=32):
    """An operand whose codes rows carry `extra_ld` spare bytes (canary) and
    whose code, scale and scalar buffers sit between guard zones."""
    ld = (cols // 2 + 15) // 16 * 16 + extra_ld
    codes = Guarded(rows * ld)
    scales = Guarded(max(16, capi.nvfp4_scale_bytes(rows, cols)))
    scalars = Guarded(16)
    op = ops.NVFP4Operand(codes=codes.body.view(rows, ld), scales=scales.body,
                          amax=scalars.body[:4].view(torch.float32), global_scale=scalars.body[4:8].view(torch.float32),
                          rows=rows, cols=cols)
    return op, (codes, scales, scalars)


def check_operand(op, bufs):
    codes, scales, scalars = bufs
    assert codes.guards_intact(), "write outside the codes buffer"
    assert scales.guards_intact(), "write outside the scales buffer"
    assert scalars.guards_intact(), "write outside amax / s_g"
    pad = op.codes.cpu().numpy()[:, op.cols // 2:]
    assert (pad == CANARY).all(), "write into the row padding of the codes"
    assert (scalars.body.cpu().numpy()[8:] == CANARY).all()


SHAPES = [(272, 336), (560, 96)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kw", [dict(), dict(sr=True, seed=3), dict(rht_mask=0x1F2E), dict(two_d=True),
                                dict(scale46=True), dict(rht_mask=0x1F2E, sr=True, seed=5, scale46=True)])
def test_quantize_writes_only_its_outputs(shape, kw):
    rows, cols = shape
    x = helpers.to_device_bf16(inputs.normal(rows, cols, 9, outlier_channels=2))
    for rowwise, colwise in ((True, False), (False, True), (True, True)):
        row, rb = guarded_operand(rows, cols) if rowwise else (None, None)
        col, cb = guarded_operand(cols, rows) if colwise else (None, None)
        ops.quantize(x, rowwise=rowwise, colwise=colwise, out_row=row, out_col=col, **kw)
        torch.cuda.synchronize()
        assert ops.device_error() == capi.NVFP4_OK
        for op, b in ((row, rb), (col, cb)):
            if op is not None:
                check_operand(op, b)


@pytest.mark.parametrize("shape", SHAPES)
def test_pairs_and_requantize_write_only_their_outputs(shape):
    rows, cols = shape
    x = helpers.to_device_bf16(inputs.student_t(rows, cols, 10))
    row, rb = guarded_operand(rows, cols)
    col, cb = guarded_operand(cols, rows)
    ops.quantize_row_col_rht(x, 0x3333, sr=True, seed=1, out_row=row, out_col=col)
    torch.cuda.synchronize()
    check_operand(row, rb)
    check_operand(col, cb)
    amax = torch.stack([row.amax[0], col.amax[0]]).contiguous()
    row2, rb2 = guarded_operand(rows, cols)
    col2, cb2 = guarded_operand(cols, rows)
    ops.quantize_row_col_rht_amax(x, 0x3333, amax, out_row=row2, out_col=col2)
    req, qb = guarded_operand(cols, rows)
    ops.requantize_col_rht(row, 0x0F0F, sr=True, seed=2, out_col=req)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    for op, b in ((row2, rb2), (col2, cb2), (req, qb)):
        check_operand(op, b)


@pytest.mark.parametrize("M,N,K", [(200, 300, 320), (256, 512, 1024), (130, 260, 80)])
@pytest.mark.parametrize("mode", ["bf16", "fp32", "amax", "axpby"])
def test_gemm_writes_only_its_output(M, N, K, mode):
    rng = np.random.default_rng(M + N + K)
    a = ops.alloc_operand(M, K)
    b = ops.alloc_operand(N, K)
    for op in (a, b):
        op.codes.copy_(torch.from_numpy(rng.integers(0, 256, op.codes.shape, dtype=np.uint8)))
        op.scales.copy_(torch.from_numpy(rng.integers(0x20, 0x48, op.scales.shape, dtype=np.uint8)))
        op.global_scale.fill_(1.0)
    fp32 = mode == "fp32"
    esz = 4 if fp32 else 2
    # the fused amax writes through TMA: rows on 16 bytes
    ldd = (N + 7) // 8 * 8 + 8 if mode == "amax" else N + 8
    if mode == "amax" and M % 16:
        pytest.skip("the fused amax takes 16-row blocks")
    buf = Guarded(M * ldd * esz)
    d = buf.body.view(torch.float32 if fp32 else torch.bfloat16).view(M, ldd)[:, :N]
    amax_buf = Guarded(16)
    if mode == "amax":
        ops.gemm_amax(a, b, 0x1234, out=d, amax=amax_buf.body[:8].view(torch.float32))
    elif mode == "axpby":
        c = torch.randn((M, N), device="cuda").to(torch.bfloat16)
        ops.gemm_axpby(a, b, 0.5, c, 2.0, out=d)
    else:
        ops.gemm(a, b, out=d)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert buf.guards_intact(), "write outside the output buffer"
    pad = buf.body.cpu().numpy().reshape(M, ldd * esz)[:, N * esz:]
    assert (pad == CANARY).all(), "write into the output's row padding"
    assert amax_buf.guards_intact() and (amax_buf.body.cpu().numpy()[8:] == CANARY).all()


def test_dequantize_writes_only_its_output():
    rows, cols = 272, 336
    q, _ = ops.quantize(helpers.to_device_bf16(inputs.normal(rows, cols, 11)))
    ldy = cols + 8
    buf = Guarded(rows * ldy * 4)
    y = buf.body.view(torch.float32).view(rows, ldy)
    capi.check(capi.nvfp4_dequantize(q.struct(), y.data_ptr(), ldy, capi.NVFP4_OUT_FP32, ops.stream_handle()))
    torch.cuda.synchronize()
    assert buf.guards_intact()
    assert (buf.body.cpu().numpy().reshape(rows, ldy * 4)[:, cols * 4:] == CANARY).all()


@pytest.mark.parametrize("N", [257, 263, 271, 300, 8, 3])
@pytest.mark.parametrize("mode", ["bf16", "fp32", "amax", "axpby"])
def test_gemm_tma_rows_write_only_their_columns(N, mode):
    """Rows of D on 16-byte boundaries go out by TMA stores, which write whole
    16-byte pieces: with N not a multiple of 8 (BF16) or 4 (FP32) the last
    piece of a row reaches past column N, so it must not be stored by TMA.
    The padding after column N keeps the canary."""
    M, K = 96, 64
    rng = np.random.default_rng(N)
    a = ops.alloc_operand(M, K)
    b = ops.alloc_operand(N, K)
    for op in (a, b):
        op.codes.copy_(torch.from_numpy(rng.integers(0, 256, op.codes.shape, dtype=np.uint8)))
        op.scales.copy_(torch.from_numpy(rng.integers(0x20, 0x48, op.scales.shape, dtype=np.uint8)))
        op.global_scale.fill_(1.0)
    fp32 = mode == "fp32"
    esz = 4 if fp32 else 2
    ldd = (N + 7) // 8 * 8 + 8                     # rows on 16 bytes: the TMA-store path
    buf = Guarded(M * ldd * esz)
    d = buf.body.view(torch.float32 if fp32 else torch.bfloat16).view(M, ldd)[:, :N]
    amax_buf = Guarded(16)
    if mode == "amax":
        ops.gemm_amax(a, b, 0x1234, out=d, amax=amax_buf.body[:8].view(torch.float32))
    elif mode == "axpby":
        # C with rows on 16 bytes too: the epilogue reads it through the staging slices
        c = torch.randn((M, ldd), device="cuda").to(torch.bfloat16)[:, :N]
        ops.gemm_axpby(a, b, 0.5, c, 2.0, out=d)
    else:
        ops.gemm(a, b, out=d)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert buf.guards_intact(), "write outside the output buffer"
    pad = buf.body.cpu().numpy().reshape(M, ldd * esz)[:, N * esz:]
    assert (pad == CANARY).all(), "write into the output's row padding"
    if mode == "axpby":
        ref_c = (0.5 * ops.gemm(a, b, out_dtype=torch.float32) + 2.0 * c.float())
        assert torch.allclose(d.float(), ref_c, rtol=2 ** -7, atol=1e-6)
    # and the columns themselves are the product
    ref = ops.gemm(a, b, out_dtype=torch.float32) if not fp32 else None
    if mode in ("bf16", "amax"):
        assert torch.equal(d.float(), ref.to(torch.bfloat16).float())

"""torch-facing helpers over the C ABI.

PyTorch provides the device memory and the stream; every step of the
quantize / GEMM / dequantize path runs in the library's CUDA kernels.  These
helpers only allocate the caller-owned buffers the ABI expects and marshal
pointers.
"""
from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import capi


@dataclass
class NVFP4Operand:
    """Device buffers of one encoded operand (see nvfp4_tensor)."""
    codes: torch.Tensor      # uint8 [rows, ld_codes]
    scales: torch.Tensor     # uint8 [nvfp4_scale_bytes(rows, cols)]
    amax: torch.Tensor       # float32 [1]
    global_scale: torch.Tensor  # float32 [1]
    rows: int
    cols: int

    @property
    def ld_codes(self) -> int:
        return self.codes.shape[1]

    def struct(self) -> capi.nvfp4_tensor:
        return capi.nvfp4_tensor(self.codes.data_ptr(), self.scales.data_ptr(),
                                 self.amax.data_ptr(), self.global_scale.data_ptr(),
                                 self.rows, self.cols, self.ld_codes)

    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel() + 8


def _round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


def alloc_operand(rows: int, cols: int, device="cuda") -> NVFP4Operand:
    ld = max(16, _round_up(cols // 2, 16))
    nscale = max(16, capi.nvfp4_scale_bytes(rows, cols))
    return NVFP4Operand(
        codes=torch.empty((rows, ld), dtype=torch.uint8, device=device),
        scales=torch.empty(nscale, dtype=torch.uint8, device=device),
        amax=torch.empty(1, dtype=torch.float32, device=device),
        global_scale=torch.empty(1, dtype=torch.float32, device=device),
        rows=rows, cols=cols)


def stream_handle(stream: Optional[torch.cuda.Stream] = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Workspace:
    """Caller-owned scratch for the quantizer (one per stream)."""

    def __init__(self, device="cuda"):
        n = capi.nvfp4_quantize_workspace_size(0, 0, 3)
        self.buf = torch.empty(n, dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


_workspaces = {}


def _workspace(device) -> Workspace:
    key = torch.device(device)
    if key not in _workspaces:
        _workspaces[key] = Workspace(key)
    return _workspaces[key]


def quantize(x: torch.Tensor, *, two_d: bool = False, sr: bool = False, rht_mask: Optional[int] = None,
             seed: int = 0, stream_id: int = 0, rowwise: bool = True, colwise: bool = False,
             out_row: Optional[NVFP4Operand] = None, out_col: Optional[NVFP4Operand] = None,
             workspace: Optional[Workspace] = None, stream=None, scale46: bool = False
             ) -> Tuple[Optional[NVFP4Operand], Optional[NVFP4Operand]]:
    """Quantize a bf16 CUDA matrix (nvfp4_quantize / nvfp4_rht_quantize).
    scale46 selects 1x16 blocks with 4/6 adaptive scales (NVFP4_SCALE_1X16_46)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if rowwise and out_row is None:
        out_row = alloc_operand(rows, cols, x.device)
    if colwise and out_col is None:
        out_col = alloc_operand(cols, rows, x.device)
    ws = workspace or _workspace(x.device)
    orient = (capi.NVFP4_ROWWISE if rowwise else 0) | (capi.NVFP4_COLWISE if colwise else 0)
    sr_ = capi.NVFP4_ROUND_SR if sr else capi.NVFP4_ROUND_RNE
    sc = capi.NVFP4_SCALE_16X16 if two_d else (capi.NVFP4_SCALE_1X16_46 if scale46 else capi.NVFP4_SCALE_1X16)
    trow = out_row.struct() if rowwise else None
    tcol = out_col.struct() if colwise else None
    st = stream_handle(stream)
    if rht_mask is None:
        status = capi.nvfp4_quantize(x.data_ptr(), rows, cols, x.stride(0), sc, sr_, seed, stream_id,
                                     orient, trow, tcol, ws.ptr, ws.nbytes, st)
    else:
        status = capi.nvfp4_rht_quantize(x.data_ptr(), rows, cols, x.stride(0), sc, sr_, seed,
                                         stream_id, orient, trow, tcol, rht_mask, ws.ptr, ws.nbytes, st)
    capi.check(status, "nvfp4_quantize")
    return (out_row if rowwise else None), (out_col if colwise else None)


def requantize_col_rht(q_row: NVFP4Operand, rht_mask: int, *, sr: bool = False, seed: int = 0,
                       stream_id: int = 0, out_col: Optional[NVFP4Operand] = None,
                       workspace: Optional[Workspace] = None, stream=None) -> NVFP4Operand:
    """Wgrad's second operand from a row-wise operand (nvfp4_requantize_col_rht):
    dequantize, RHT along the rows, col-wise 1x16."""
    if out_col is None:
        out_col = alloc_operand(q_row.cols, q_row.rows, q_row.codes.device)
    ws = workspace or _workspace(q_row.codes.device)
    status = capi.nvfp4_requantize_col_rht(q_row.struct(), capi.NVFP4_ROUND_SR if sr else capi.NVFP4_ROUND_RNE,
                                           seed, stream_id, rht_mask, out_col.struct(), ws.ptr, ws.nbytes,
                                           stream_handle(stream))
    capi.check(status, "nvfp4_requantize_col_rht")
    return out_col


def quantize_row_col_rht(x: torch.Tensor, rht_mask: int, *, sr: bool = False, seed: int = 0,
                         stream_row: int = 0, stream_col: int = 0, out_row: Optional[NVFP4Operand] = None,
                         out_col: Optional[NVFP4Operand] = None, workspace: Optional[Workspace] = None,
                         stream=None) -> Tuple[NVFP4Operand, NVFP4Operand]:
    """Row-wise 1x16 (no RHT) and col-wise 1x16 with RHT of one bf16 matrix
    (nvfp4_quantize_row_col_rht): the Fprop/Dgrad and the Wgrad operand."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out_row is None:
        out_row = alloc_operand(rows, cols, x.device)
    if out_col is None:
        out_col = alloc_operand(cols, rows, x.device)
    ws = workspace or _workspace(x.device)
    status = capi.nvfp4_quantize_row_col_rht(x.data_ptr(), rows, cols, x.stride(0),
                                             capi.NVFP4_ROUND_SR if sr else capi.NVFP4_ROUND_RNE, seed,
                                             stream_row, stream_col, rht_mask, out_row.struct(), out_col.struct(),
                                             ws.ptr, ws.nbytes, stream_handle(stream))
    capi.check(status, "nvfp4_quantize_row_col_rht")
    return out_row, out_col


def gemm(a: NVFP4Operand, b: NVFP4Operand, out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None,
         stream=None) -> torch.Tensor:
    """D = A * B^T (nvfp4_gemm)."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    dt = capi.NVFP4_OUT_FP32 if out.dtype == torch.float32 else capi.NVFP4_OUT_BF16
    status = capi.nvfp4_gemm(a.struct(), b.struct(), out.data_ptr(), out.stride(0), dt, None, 0,
                             stream_handle(stream))
    capi.check(status, "nvfp4_gemm")
    return out



def gemm_amax(a: NVFP4Operand, b: NVFP4Operand, rht_mask: int, out: Optional[torch.Tensor] = None,
              amax: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """D = A * B^T in BF16 plus D's two tensor amaxes (nvfp4_gemm_amax): amax[0]
    plain, amax[1] after the RHT along D's rows with rht_mask."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.codes.device)
    if amax is None:
        amax = torch.empty(2, dtype=torch.float32, device=a.codes.device)
    status = capi.nvfp4_gemm_amax(a.struct(), b.struct(), out.data_ptr(), out.stride(0), amax.data_ptr(),
                                  rht_mask, None, 0, stream_handle(stream))
    capi.check(status, "nvfp4_gemm_amax")
    return out, amax


def quantize_row_col_rht_amax(x: torch.Tensor, rht_mask: int, amax: torch.Tensor, *, sr: bool = False,
                              seed: int = 0, stream_row: int = 0, stream_col: int = 0,
                              out_row: Optional[NVFP4Operand] = None, out_col: Optional[NVFP4Operand] = None,
                              stream=None) -> Tuple[NVFP4Operand, NVFP4Operand]:
    """quantize_row_col_rht with the two tensor amaxes given (nvfp4_quantize_row_col_rht_amax)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert amax.dtype == torch.float32 and amax.numel() >= 2
    rows, cols = x.shape
    if out_row is None:
        out_row = alloc_operand(rows, cols, x.device)
    if out_col is None:
        out_col = alloc_operand(cols, rows, x.device)
    status = capi.nvfp4_quantize_row_col_rht_amax(
        x.data_ptr(), rows, cols, x.stride(0), capi.NVFP4_ROUND_SR if sr else capi.NVFP4_ROUND_RNE, seed,
        stream_row, stream_col, rht_mask, amax.data_ptr(), out_row.struct(), out_col.struct(), stream_handle(stream))
    capi.check(status, "nvfp4_quantize_row_col_rht_amax")
    return out_row, out_col


def gemm_lora(a: NVFP4Operand, b: NVFP4Operand, u: torch.Tensor, v: torch.Tensor, beta: float,
              out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None, scratch: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """D = A * B^T + beta * U V^T (nvfp4_gemm_lora): U [M][r], V [N][r] bf16, r a multiple of 64."""
    assert u.dtype == torch.bfloat16 and v.dtype == torch.bfloat16 and u.stride(1) == 1 and v.stride(1) == 1
    r = u.shape[1]
    assert v.shape[1] == r and u.shape[0] == a.rows and v.shape[0] == b.rows
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    nbytes = capi.nvfp4_gemm_lora_workspace_size(a.rows, r)
    if scratch is None or scratch.numel() < nbytes:
        scratch = torch.empty(nbytes, dtype=torch.uint8, device=a.codes.device)
    dt = capi.NVFP4_OUT_FP32 if out.dtype == torch.float32 else capi.NVFP4_OUT_BF16
    status = capi.nvfp4_gemm_lora(a.struct(), b.struct(), out.data_ptr(), out.stride(0), dt, u.data_ptr(),
                                  u.stride(0), v.data_ptr(), v.stride(0), r, float(beta), scratch.data_ptr(),
                                  scratch.numel(), stream_handle(stream))
    capi.check(status, "nvfp4_gemm_lora")
    return out

def gemm_axpby(a: NVFP4Operand, b: NVFP4Operand, alpha: float, c: Optional[torch.Tensor], beta: float,
               out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """D = alpha * A * B^T + beta * C (nvfp4_gemm_axpby); C has D's dtype and may be `out` itself."""
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    dt = capi.NVFP4_OUT_FP32 if out.dtype == torch.float32 else capi.NVFP4_OUT_BF16
    if c is not None:
        assert c.dtype == out.dtype and c.dim() == 2 and c.stride(1) == 1
    status = capi.nvfp4_gemm_axpby(a.struct(), b.struct(), out.data_ptr(), out.stride(0), dt, float(alpha),
                                   None if c is None else c.data_ptr(), 0 if c is None else c.stride(0),
                                   float(beta), None, 0, stream_handle(stream))
    capi.check(status, "nvfp4_gemm_axpby")
    return out


def newton_schulz_step(x: torch.Tensor, a: float, b: float, c: float, rht_mask: int,
                       out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """One NVFP4 Newton-Schulz iteration of a bf16 [m][n] matrix (nvfp4_newton_schulz_step).
    After the call the workspace begins with A_k and then B_k (bf16 [m][m]; see ns_intermediates)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    m, n = x.shape
    if out is None:
        out = torch.empty_like(x)
    nbytes = capi.nvfp4_newton_schulz_workspace_size(m, n)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    status = capi.nvfp4_newton_schulz_step(x.data_ptr(), m, n, x.stride(0), float(a), float(b), float(c),
                                           rht_mask, out.data_ptr(), out.stride(0), workspace.data_ptr(),
                                           workspace.numel(), stream_handle(stream))
    capi.check(status, "nvfp4_newton_schulz_step")
    return out


def ns_intermediates(workspace: torch.Tensor, m: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """Views of A_k and B_k (bf16 [m][m]) at the start of a Newton-Schulz step's workspace."""
    off_b = (2 * m * m + 255) // 256 * 256
    a = workspace[:2 * m * m].view(torch.bfloat16).view(m, m)
    b = workspace[off_b:off_b + 2 * m * m].view(torch.bfloat16).view(m, m)
    return a, b


def dequantize(q: NVFP4Operand, out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """x^ = e2m1 * s_b * s_g (nvfp4_dequantize)."""
    y = torch.empty((q.rows, q.cols), dtype=out_dtype, device=q.codes.device)
    dt = capi.NVFP4_OUT_FP32 if out_dtype == torch.float32 else capi.NVFP4_OUT_BF16
    capi.check(capi.nvfp4_dequantize(q.struct(), y.data_ptr(), y.stride(0), dt, stream_handle(stream)),
               "nvfp4_dequantize")
    return y


def device_error(stream=None) -> int:
    return capi.nvfp4_device_error(stream_handle(stream))

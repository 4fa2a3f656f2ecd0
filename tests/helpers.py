"""Shared test helpers: moving seeded inputs to the device and reading the
library's outputs back in the oracle's plain layouts.

The scale-layout map below is written from include/nvfp4.h's documentation of
the tile layout; it is test code, independent of the CUDA sources.
"""
import numpy as np

GEMM_TOL_REL = 1e-4      # |y - y_ref| <= 1e-4 * sum_k |a_k b_k| + 1e-6
GEMM_TOL_ABS = 1e-6


def scale_index_map(rows: int, cols: int) -> np.ndarray:
    """offset(r, j) of every block scale of a [rows][cols] operand."""
    S = cols // 16
    s4 = (cols + 63) // 64
    r = np.arange(rows, dtype=np.int64)[:, None]
    j = np.arange(S, dtype=np.int64)[None, :]
    return ((r // 128) * s4 + j // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + j % 4


def scale_bytes(rows: int, cols: int) -> int:
    if rows <= 0 or cols <= 0:
        return 0
    return ((rows + 127) // 128) * ((cols + 63) // 64) * 512


def scales_to_rowmajor(tiled: np.ndarray, rows: int, cols: int) -> np.ndarray:
    return tiled[scale_index_map(rows, cols)]


def padding_mask(rows: int, cols: int) -> np.ndarray:
    """True at the bytes of the scale buffer that hold no block scale."""
    m = np.ones(scale_bytes(rows, cols), bool)
    m[scale_index_map(rows, cols).ravel()] = False
    return m


def to_device_bf16(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def operand_to_host(op):
    """(codes [rows][cols/2], row-major scales, amax, s_g) of a device operand."""
    codes = op.codes.cpu().numpy()[:, : op.cols // 2]
    tiled = op.scales.cpu().numpy()
    scales = scales_to_rowmajor(tiled, op.rows, op.cols) if op.rows and op.cols else \
        np.zeros((op.rows, op.cols // 16), np.uint8)
    return codes, scales, np.float32(op.amax.item()), np.float32(op.global_scale.item()), tiled


def as_oracle_operand(op, row_ids=None):
    """A device operand as the dict the oracle's gemm_f64 takes."""
    codes, scales, _, sg, _ = operand_to_host(op)
    if row_ids is not None:
        codes, scales = codes[row_ids], scales[row_ids]
    return dict(codes=np.ascontiguousarray(codes), scales=np.ascontiguousarray(scales), s_g=sg)


def bf16_half_ulp(y: np.ndarray) -> np.ndarray:
    """Half a bfloat16 ulp at |y| (8 significant bits)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 2.0 ** -134)


def gemm_bound(abs_sum: np.ndarray, y_ref: np.ndarray, bf16: bool) -> np.ndarray:
    b = GEMM_TOL_REL * abs_sum + GEMM_TOL_ABS
    if bf16:
        b = b + bf16_half_ulp(y_ref)
    return b

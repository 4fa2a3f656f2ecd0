"""Seeded synthetic inputs for the NVFP4 linear-layer pipeline.

This module holds no quantization or GEMM arithmetic: it draws numbers.  It is
the one module that both the CUDA path's callers and the CPU oracle's callers
use, so that both sides see the same bytes.

Shapes and distributions follow the pages' 3B model: hidden 3072, FFN 9216,
24 query heads and 12 KV heads of head_dim 128, 2048-token sequences
("Full-Stack FP4" summary page, Results and Analysis).  Values are drawn in
float32 with numpy's PCG64 ``default_rng(seed)`` and rounded to bfloat16
(nearest, ties to even).
"""
import os
from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import numpy as np

HIDDEN = 3072
FFN = 9216
N_HEADS = 24
N_KV_HEADS = 12
HEAD_DIM = 128
SEQ = 2048


def to_bf16_bits(x) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), nearest with ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK_ROWS = 512          # fixed chunking: results do not depend on the thread count


def _chunked(rows: int, cols: int, seed: int, draw) -> np.ndarray:
    """Fill a float32 [rows, cols] array chunk by chunk of _CHUNK_ROWS rows;
    chunk c draws from default_rng(SeedSequence([seed, c])).  Chunks run on a
    thread pool (numpy's bulk samplers release the GIL)."""
    out = np.empty((rows, cols), np.float32)
    n_chunks = (rows + _CHUNK_ROWS - 1) // _CHUNK_ROWS

    def work(c):
        r0, r1 = c * _CHUNK_ROWS, min(rows, (c + 1) * _CHUNK_ROWS)
        rng = np.random.default_rng(np.random.SeedSequence([seed, c]))
        draw(rng, out[r0:r1])

    if n_chunks <= 1:
        for c in range(n_chunks):
            work(c)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(n_chunks, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(n_chunks)))
    return out


def normal(rows: int, cols: int, seed: int, std: float = 1.0, outlier_channels: int = 0,
           outlier_scale: float = 50.0) -> np.ndarray:
    """N(0, std^2) bf16 bits; ``outlier_channels`` columns (chosen by
    default_rng(seed)) scaled by ``outlier_scale``."""
    def draw(rng, block):
        rng.standard_normal(block.shape, dtype=np.float32, out=block)
        if std != 1.0:
            block *= np.float32(std)

    x = _chunked(rows, cols, seed, draw)
    if outlier_channels:
        ch = np.random.default_rng(seed).choice(cols, outlier_channels, replace=False)
        x[:, ch] *= np.float32(outlier_scale)
    return to_bf16_bits(x)


def student_t(rows: int, cols: int, seed: int, df: int = 3, scale: float = 1e-3) -> np.ndarray:
    """Student-t(df) * scale bf16 bits (heavy-tailed gradients), drawn as
    Z / sqrt(chi2_df / df) with chi2_df a sum of df squared standard normals."""
    def draw(rng, block):
        rng.standard_normal(block.shape, dtype=np.float32, out=block)
        chi2 = np.zeros(block.shape, np.float32)
        g = np.empty(block.shape, np.float32)
        for _ in range(int(df)):
            rng.standard_normal(block.shape, dtype=np.float32, out=g)
            g *= g
            chi2 += g
        chi2 *= np.float32(1.0 / df)
        np.sqrt(chi2, out=chi2)
        block /= chi2
        block *= np.float32(scale)

    return to_bf16_bits(_chunked(rows, cols, seed, draw))


def extreme_range(rows: int, cols: int, seed: int, amax: float, span_log2: int = 40,
                  zero_tile_frac: float = 1 / 16, zero_block_frac: float = 1 / 32) -> np.ndarray:
    """Edge-case bf16 bits spanning about 2^-span_log2 of the tensor amax.

    N(0, 1) values whose 16x16 tiles are each scaled by 2^-k, k uniform on
    0..span_log2, with some tiles all zero, some 16-element row blocks all
    zero and some zeros negative; everything is scaled so that the largest
    magnitude is just below ``amax`` and element (0, 0) is set to ``amax``
    itself (pass a bfloat16 value).  Values that fall below the smallest
    bfloat16 subnormal become zeros.  rows and cols are multiples of 16.
    """
    assert rows % 16 == 0 and cols % 16 == 0
    rng = np.random.default_rng([seed, 0xE7])
    x = rng.standard_normal((rows, cols), dtype=np.float32).astype(np.float64)
    tiles = x.reshape(rows // 16, 16, cols // 16, 16)
    k = rng.integers(0, span_log2 + 1, (rows // 16, cols // 16))
    tiles *= np.exp2(-k.astype(np.float64))[:, None, :, None]
    tiles *= (rng.random((rows // 16, cols // 16)) >= zero_tile_frac)[:, None, :, None]
    blocks = x.reshape(rows, cols // 16, 16)
    blocks *= (rng.random((rows, cols // 16)) >= zero_block_frac)[:, :, None]
    m = np.abs(x).max()
    if m > 0:
        x *= (float(amax) * 0.99) / m
    x[x == 0] = 0.0
    neg = rng.random((rows, cols)) < 0.5
    x[(x == 0) & neg] = -0.0
    x[0, 0] = amax
    return to_bf16_bits(x.astype(np.float32))


def rht_sign_mask(seed: int) -> int:
    """The 16 random signs of D for one backward pass, as a bit mask."""
    rng = np.random.default_rng([seed, 0xD])
    return int(rng.integers(0, 1 << 16))


def outlier_count(cols: int, fraction: float = 0.001) -> int:
    """0.1% of the channels, at least one."""
    return max(1, int(round(cols * fraction)))


@dataclass
class Operand:
    """One bf16 input tensor of a workload and how it is quantized."""
    name: str
    rows: int
    cols: int
    kind: str            # "normal", "weight", "grad"
    seed: int
    outliers: int = 0


@dataclass
class Workload:
    name: str
    seed: int
    operands: List[Operand] = field(default_factory=list)
    # (name, A operand, A orientation, B operand, B orientation)
    gemms: List[Tuple[str, str, str, str, str]] = field(default_factory=list)

    def make(self, name: str) -> np.ndarray:
        op = next(o for o in self.operands if o.name == name)
        if op.kind == "normal":
            return normal(op.rows, op.cols, op.seed, 1.0, op.outliers)
        if op.kind == "weight":
            return normal(op.rows, op.cols, op.seed, 0.02)
        if op.kind == "grad":
            return student_t(op.rows, op.cols, op.seed)
        raise ValueError(op.kind)


def c1_single_linear() -> Workload:
    """M=128 tokens, K=1024, N=1024; 4 of 1024 X channels x50; seed 0."""
    return Workload("c1_linear_fwd_128x1024x1024", 0, [
        Operand("X", 128, 1024, "normal", 0, outliers=4),
        Operand("W", 1024, 1024, "weight", 1),
    ], [("fprop", "X", "row", "W", "row")])


def c2_attention_projections(tokens: int = 4 * SEQ) -> Workload:
    qkv = (N_HEADS + 2 * N_KV_HEADS) * HEAD_DIM          # 6144
    return Workload(f"c2_attn_proj_{tokens}tok", 2, [
        Operand("X", tokens, HIDDEN, "normal", 20, outliers=outlier_count(HIDDEN)),
        Operand("W_qkv", qkv, HIDDEN, "weight", 21),
        Operand("W_o", HIDDEN, HIDDEN, "weight", 22),
        Operand("dY_qkv", tokens, qkv, "grad", 23),
        Operand("dY_o", tokens, HIDDEN, "grad", 24),
    ], [("fprop_qkv", "X", "row", "W_qkv", "row2d"),
        ("fprop_o", "X", "row", "W_o", "row2d"),
        ("dgrad_qkv", "dY_qkv", "row", "W_qkv", "col2d"),
        ("dgrad_o", "dY_o", "row", "W_o", "col2d")])


def c3_ffn_wgrad(tokens: int = 4 * SEQ) -> Workload:
    return Workload(f"c3_ffn_wgrad_{tokens}tok", 3, [
        Operand("dY", tokens, FFN, "grad", 30),
        Operand("X", tokens, HIDDEN, "normal", 31),
    ], [("wgrad", "dY", "col_rht_sr", "X", "col_rht")])


def c4_ffn_layer_step(tokens: int = 8 * SEQ) -> Workload:
    return Workload(f"c4_ffn_layer_step_{tokens}tok", 4, [
        Operand("X", tokens, HIDDEN, "normal", 40, outliers=outlier_count(HIDDEN)),
        Operand("W_up", FFN, HIDDEN, "weight", 41),
        Operand("H", tokens, FFN, "normal", 42, outliers=outlier_count(FFN)),
        Operand("W_down", HIDDEN, FFN, "weight", 43),
        Operand("dY_down", tokens, HIDDEN, "grad", 44),
        Operand("dY_up", tokens, FFN, "grad", 45),
    ], [("fprop_up", "X", "row", "W_up", "row2d"),
        ("fprop_down", "H", "row", "W_down", "row2d"),
        ("dgrad_down", "dY_down", "row_sr", "W_down", "col2d"),
        ("dgrad_up", "dY_up", "row_sr", "W_up", "col2d"),
        ("wgrad_down", "dY_down", "col_rht_sr", "H", "col_rht"),
        ("wgrad_up", "dY_up", "col_rht_sr", "X", "col_rht")])


def c5_sweep_sizes() -> List[Tuple[int, int]]:
    """(rows, row_length) of the quantizer sweep: 2^20..2^29 elements."""
    out = []
    for n in (1 << 20, 1 << 22, 1 << 24, 1 << 26, 1 << 28, 1 << 29):
        for L in (3072, 9216, 8192):
            rows = (n // L) // 16 * 16
            out.append((rows, L))
    return out


WORKLOADS: Dict[str, callable] = {
    "c1": c1_single_linear,
    "c2": c2_attention_projections,
    "c3": c3_ffn_wgrad,
    "c4": c4_ffn_layer_step,
}

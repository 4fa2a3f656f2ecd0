"""Seeded random parity cases: shapes, modes, input distributions and leading
dimensions drawn per case (each case's draw depends only on its index), so
that combinations no hand-written case names are still compared with the
oracle -- codes, scales, amax and s_g bit for bit, GEMM outputs within the
tolerance."""
import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
from tests import helpers

pytestmark = pytest.mark.gpu

N_QUANT, N_PAIR, N_GEMM = 48, 16, 24


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def _bits(rng, rows, cols, seed, max_log2=60):
    """One of: N(0,1) with outlier channels, Student-t(3) x 1e-3, N(0, 0.02^2),
    or (16-multiple shapes) the extreme-range recipe with a tensor amax of
    2^-max_log2 .. 2^max_log2."""
    kind = rng.integers(0, 4 if rows % 16 == 0 else 3)
    if kind == 0:
        return inputs.normal(rows, cols, seed, outlier_channels=int(rng.integers(0, 3)))
    if kind == 1:
        return inputs.student_t(rows, cols, seed)
    if kind == 2:
        return inputs.normal(rows, cols, seed, std=0.02)
    amax = float(2.0 ** int(rng.integers(-max_log2, max_log2)))
    return inputs.extreme_range(rows, cols, seed, amax=amax, span_log2=24)


def _padded(bits, pad):
    """bf16 device matrix whose rows are `pad` elements longer than the data."""
    rows, cols = bits.shape
    buf = torch.zeros((rows, cols + pad), dtype=torch.bfloat16, device="cuda")
    buf[:, :cols] = helpers.to_device_bf16(bits)
    return buf[:, :cols]


def _check(g, ref):
    codes, scales, amax, sg, tiled = helpers.operand_to_host(g)
    assert amax == ref["amax"] and sg == ref["s_g"], (amax, ref["amax"], sg, ref["s_g"])
    bad = np.argwhere(codes != ref["codes"])
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"
    bad = np.argwhere(scales != ref["scales"])
    assert bad.size == 0, f"{len(bad)} scales differ, first at {bad[:4].tolist()}"
    if g.rows and g.cols:
        assert not tiled[helpers.padding_mask(g.rows, g.cols)].any(), "scale padding not zero"


@pytest.mark.parametrize("case", range(N_QUANT))
def test_fuzz_quantize(case):
    rng = np.random.default_rng(1_000 + case)
    scaling = int(rng.integers(0, 3))              # 1x16, 16x16, 1x16 with 4/6
    rounding = int(rng.integers(0, 2))
    rht = scaling != 1 and bool(rng.integers(0, 2))
    rowwise, colwise = [(True, False), (False, True), (True, True)][int(rng.integers(0, 3))]
    cols = 16 * int(rng.integers(1, 80))
    rows = int(rng.integers(1, 700))
    if colwise or scaling == 1:
        rows = 16 * max(1, rows // 16)
    pad = 8 * int(rng.integers(0, 4))
    mask = int(rng.integers(0, 1 << 16))
    seed, sid = int(rng.integers(0, 2 ** 62)), int(rng.integers(0, 2 ** 62))
    bits = _bits(rng, rows, cols, 2_000 + case)
    row, col = ops.quantize(_padded(bits, pad), two_d=scaling == 1, scale46=scaling == 2, sr=rounding == 1,
                            rht_mask=mask if rht else None, seed=seed, stream_id=sid, rowwise=rowwise,
                            colwise=colwise)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    kw = dict(scaling=scaling, rounding=rounding, use_rht=rht, sign_mask=mask, seed=seed, stream_id=sid)
    if rowwise:
        _check(row, oracle.quantize(bits, oracle.ROWWISE, **kw))
    if colwise:
        _check(col, oracle.quantize(bits, oracle.COLWISE, **kw))


@pytest.mark.parametrize("case", range(N_PAIR))
def test_fuzz_pair(case):
    """nvfp4_quantize_row_col_rht and its amax-given form on random shapes."""
    rng = np.random.default_rng(3_000 + case)
    rows, cols = 16 * int(rng.integers(1, 60)), 16 * int(rng.integers(1, 60))
    sr = bool(rng.integers(0, 2))
    mask = int(rng.integers(0, 1 << 16))
    seed, s_row, s_col = (int(v) for v in rng.integers(0, 2 ** 62, 3))
    bits = _bits(rng, rows, cols, 4_000 + case)
    ref_row = oracle.quantize(bits, oracle.ROWWISE, rounding=int(sr), seed=seed, stream_id=s_row)
    ref_col = oracle.quantize(bits, oracle.COLWISE, rounding=int(sr), use_rht=True, sign_mask=mask, seed=seed,
                              stream_id=s_col)
    x = _padded(bits, 8 * int(rng.integers(0, 3)))
    if rng.integers(0, 2):
        row, col = ops.quantize_row_col_rht(x, mask, sr=sr, seed=seed, stream_row=s_row, stream_col=s_col)
    else:
        amax = torch.tensor([ref_row["amax"], ref_col["amax"]], dtype=torch.float32, device="cuda")
        row, col = ops.quantize_row_col_rht_amax(x, mask, amax, sr=sr, seed=seed, stream_row=s_row,
                                                 stream_col=s_col)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    _check(row, ref_row)
    _check(col, ref_col)


@pytest.mark.parametrize("case", range(N_GEMM))
def test_fuzz_gemm(case):
    """Quantized operands of random shapes (ragged M and N, K a multiple of
    16) and a random output leading dimension and dtype."""
    rng = np.random.default_rng(5_000 + case)
    M, N = int(rng.integers(1, 600)), int(rng.integers(1, 600))
    K = 16 * int(rng.integers(1, 100))
    out_dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    # tensor amaxes within 2^+-20: products and their sums stay inside FP32
    a_bits = _bits(rng, M, K, 6_000 + case, max_log2=20)
    b_bits = _bits(rng, N, K, 7_000 + case, max_log2=20)
    a, _ = ops.quantize(helpers.to_device_bf16(a_bits))
    b, _ = ops.quantize(helpers.to_device_bf16(b_bits))
    pad = int(rng.integers(0, 12))
    out = torch.full((M, N + pad), 7.0, dtype=out_dtype, device="cuda")
    y = ops.gemm(a, b, out=out[:, :N])
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert bool((out[:, N:] == 7.0).all()), "write into the output's row padding"
    ref, abs_sum = oracle.gemm_f64(helpers.as_oracle_operand(a), helpers.as_oracle_operand(b))
    bound = helpers.gemm_bound(abs_sum, ref, out_dtype == torch.bfloat16)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"{int((err > bound).sum())} of {err.size} outside the bound"

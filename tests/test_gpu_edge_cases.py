"""GPU parity of the quantizer on the method's extreme-range edge cases,
bit-exact against the oracle, through the C ABI:

* block amaxes from 1 down to 2^-40 of the tensor amax, so block scales are
  subnormal E4M3 values or round to 0 (r_b = 0), with all-zero tiles and
  blocks and negative zeros inside non-zero tensors;
* a tensor amax at bfloat16's smallest subnormal and at about 1e-36, where
  S_enc saturates at FLT_MAX and S_enc / s_b overflows for small blocks;
* a tensor amax of 3e38 (1e37 where a 16-point butterfly must stay finite);
* block amaxes exactly on an E4M3 rounding boundary (ties to even) and next
  to it, with S_enc = 1;
* the RHT encode with its 1/4 applied to the values rather than folded into
  the multipliers, reached through a given rotated amax above 1.3e38.

Every mode (1x16, 16x16, 1x16 with 4/6; RNE and SR; with and without RHT) in
both orientations, the row + col-RHT pair kernel and the amax-taking pair.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
from tests import helpers
from tests.test_gpu_quantize import MODES, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def _bf16(v):
    return float(inputs.bf16_bits_to_f32(inputs.to_bf16_bits(np.array([v], np.float32)))[0])


# tensor amax of each case; the RHT variants are capped where 16 such values
# would overflow the butterfly
CASES = {
    "s_enc_one": 2688.0,
    "smallest_subnormal": 2.0 ** -133,
    "tiny_1e-36": _bf16(1e-36),
    "huge_3e38": _bf16(3e38),
}
RHT_CAP = _bf16(1e37)


def _case_bits(name, rows, cols, rht, span=40):
    amax = CASES[name]
    if rht:
        amax = min(amax, RHT_CAP)
    seed = sum(map(ord, name)) + rows + cols
    return inputs.extreme_range(rows, cols, seed, amax, span_log2=span)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("scaling,rounding,rht", MODES)
@pytest.mark.parametrize("orientation", [oracle.ROWWISE, oracle.COLWISE])
@pytest.mark.parametrize("shape", [(128, 320), (560, 96)])
def test_extreme_range_parity(shape, orientation, scaling, rounding, rht, name):
    bits = _case_bits(name, *shape, rht)
    assert_parity(bits, orientation, scaling=scaling, rounding=rounding, use_rht=rht, sign_mask=0x5AC3,
                  seed=77, stream_id=9)


def test_smallest_subnormal_dense():
    """A tensor whose non-zero values are all +-2^-133 (span 0) in the modes
    without RHT."""
    bits = inputs.extreme_range(64, 128, 5, 2.0 ** -133, span_log2=0, zero_tile_frac=0.0, zero_block_frac=0.0)
    xf = inputs.bf16_bits_to_f32(bits)
    assert (xf != 0).sum() > 100
    for scaling, rounding, rht in MODES:
        if rht:
            continue
        for orientation in (oracle.ROWWISE, oracle.COLWISE):
            assert_parity(bits, orientation, scaling=scaling, rounding=rounding, seed=3, stream_id=1)


def _check(g, ref):
    codes, scales, amax, sg, tiled = helpers.operand_to_host(g)
    assert amax == ref["amax"] and sg == ref["s_g"]
    bad = np.argwhere(codes != ref["codes"])
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"
    bad = np.argwhere(scales != ref["scales"])
    assert bad.size == 0, f"{len(bad)} scales differ, first at {bad[:4].tolist()}"
    assert not tiled[helpers.padding_mask(g.rows, g.cols)].any(), "scale padding not zero"


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("rounding", [0, 1])
def test_extreme_range_pair(name, rounding):
    """nvfp4_quantize_row_col_rht (row-wise without RHT, col-wise with RHT,
    one amax pass) and the same pair with both amaxes given."""
    bits = _case_bits(name, 256, 320, True)
    mask, seed = 0x2D4B, 12345
    x = helpers.to_device_bf16(bits)
    row, col = ops.quantize_row_col_rht(x, mask, sr=rounding == 1, seed=seed, stream_row=3, stream_col=4)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    ref_row = oracle.quantize(bits, oracle.ROWWISE, rounding=rounding, seed=seed, stream_id=3)
    ref_col = oracle.quantize(bits, oracle.COLWISE, rounding=rounding, use_rht=True, sign_mask=mask, seed=seed,
                              stream_id=4)
    _check(row, ref_row)
    _check(col, ref_col)
    amax = torch.tensor([ref_row["amax"], ref_col["amax"]], dtype=torch.float32, device="cuda")
    row2, col2 = ops.quantize_row_col_rht_amax(x, mask, amax, sr=rounding == 1, seed=seed, stream_row=3,
                                               stream_col=4)
    torch.cuda.synchronize()
    _check(row2, ref_row)
    _check(col2, ref_col)


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("given_rot", [2.0e38, 3.3e38])
def test_rht_quarter_applied_to_the_values(rounding, given_rot):
    """With a rotated amax above about 1.3e38 the multipliers cannot carry the
    RHT's 1/4 exactly (S_enc / 448 < 2^-124), so the encode scales the rotated
    values by 1/4 instead.  No finite input reaches that amax through the amax
    pass; the amax-taking pair does (an amax given by its producer may exceed
    the tensor's own).  Values of about 1e37 keep the codes non-trivial."""
    bits = _case_bits("huge_3e38", 128, 256, True, span=6)
    mask, seed = 0x7E81, 4242
    ref_row = oracle.quantize(bits, oracle.ROWWISE, rounding=rounding, seed=seed, stream_id=1)
    ref_col = oracle.quantize(bits, oracle.COLWISE, rounding=rounding, use_rht=True, sign_mask=mask, seed=seed,
                              stream_id=2, amax_value=np.float32(given_rot))
    assert np.float32(2688.0) / np.float32(given_rot) / np.float32(448.0) < np.float32(2.0 ** -124)
    assert (ref_col["codes"] & 0x77).any(), "the case must produce non-zero codes"
    amax = torch.tensor([ref_row["amax"], given_rot], dtype=torch.float32, device="cuda")
    row, col = ops.quantize_row_col_rht_amax(helpers.to_device_bf16(bits), mask, amax, sr=rounding == 1,
                                             seed=seed, stream_row=1, stream_col=2)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    _check(row, ref_row)
    _check(col, ref_col)


# ---- block amaxes on E4M3 rounding boundaries (S_enc = 1) ----------------
def _e4m3_values():
    """The finite non-negative E4M3 values, from torch's float8 decode."""
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _boundary_amaxes():
    """Block amaxes a with a / 6 on an E4M3 value, on the midpoint of two
    neighbours (a tie) and one bfloat16 step either side of the midpoint,
    keeping those that are bfloat16 values no larger than 2688."""
    vals = _e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2
    cand = np.concatenate([6 * vals[1:], 6 * mids])
    out = []
    for a in cand:
        for f in (1.0, 1 - 2.0 ** -8, 1 + 2.0 ** -7):
            v = a * f
            if 0 < v <= 2688.0 and _bf16(v) == v:
                out.append(v)
    return np.unique(np.array(out))


def _boundary_bits(rows, cols, tile, seed):
    """Each block (1x16 row block, or 16x16 tile when tile=True) gets one of
    the boundary amaxes at a random position with a random sign, the rest
    N(0, 1) * amax / 4 clipped below it; element (0, 0) holds 2688."""
    rng = np.random.default_rng(seed)
    amaxes = _boundary_amaxes()
    x = np.zeros((rows, cols), np.float64)
    bh = 16 if tile else 1
    for r0 in range(0, rows, bh):
        for c0 in range(0, cols, 16):
            a = amaxes[rng.integers(len(amaxes))]
            blk = np.clip(rng.standard_normal((bh, 16)) * a / 4, -a * 0.9, a * 0.9)
            i, j = rng.integers(bh), rng.integers(16)
            blk[i, j] = a if rng.random() < 0.5 else -a
            x[r0:r0 + bh, c0:c0 + 16] = blk
    x[0, 0] = 2688.0
    bits = inputs.to_bf16_bits(x.astype(np.float32))
    xf = inputs.bf16_bits_to_f32(bits)
    assert np.abs(xf).max() == 2688.0
    return bits


def test_boundary_amaxes_cover_ties():
    a = _boundary_amaxes()
    vals = _e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2
    ties = np.isin(a / 6, mids)
    assert ties.sum() > 60 and (~ties).sum() > 100


@pytest.mark.parametrize("scaling,rounding", [(0, 0), (0, 1), (2, 0), (2, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("orientation", [oracle.ROWWISE, oracle.COLWISE])
def test_e4m3_boundary_parity(orientation, scaling, rounding):
    rows, cols = 256, 512
    bits = _boundary_bits(rows, cols, tile=scaling == 1, seed=31 + scaling)
    if orientation == oracle.COLWISE and scaling != 1:
        bits = np.ascontiguousarray(bits.T)   # the col-wise blocks are the boundary blocks
    assert_parity(bits, orientation, scaling=scaling, rounding=rounding, seed=8, stream_id=2)

"""GPU parity of the quantizer against the CPU oracle (bit-exact codes, block
scales, amax and s_g), through the C ABI."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def gpu_quantize(bits, orientation, scaling=0, rounding=0, use_rht=False, sign_mask=0, seed=0,
                 stream_id=0):
    x = helpers.to_device_bf16(bits)
    row, col = ops.quantize(x, two_d=scaling == 1, scale46=scaling == 2, sr=rounding == 1,
                            rht_mask=sign_mask if use_rht else None, seed=seed, stream_id=stream_id,
                            rowwise=orientation == oracle.ROWWISE, colwise=orientation == oracle.COLWISE)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    return row if orientation == oracle.ROWWISE else col


def assert_parity(bits, orientation, rows_subset=None, **kw):
    g = gpu_quantize(bits, orientation, **kw)
    codes, scales, amax, sg, tiled = helpers.operand_to_host(g)
    ref = oracle.quantize(bits, orientation, rows_subset=rows_subset, **kw)
    assert amax == ref["amax"], (amax, ref["amax"])
    assert sg == ref["s_g"]
    lr0, lr1 = ref["rows"]
    bad = np.argwhere(codes[lr0:lr1] != ref["codes"])
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"
    bad = np.argwhere(scales[lr0:lr1] != ref["scales"])
    assert bad.size == 0, f"{len(bad)} scales differ, first at {bad[:4].tolist()}"
    if rows_subset is None and g.rows and g.cols:
        assert not tiled[helpers.padding_mask(g.rows, g.cols)].any(), "scale padding not zero"
    return g


MODES = [
    # (scaling, rounding, rht); scaling 2 = 1x16 with 4/6 adaptive scales
    (0, 0, False), (0, 1, False), (0, 0, True), (0, 1, True), (1, 0, False), (1, 1, False),
    (2, 0, False), (2, 1, False), (2, 0, True), (2, 1, True),
]


@pytest.mark.parametrize("scaling,rounding,rht", MODES)
@pytest.mark.parametrize("orientation", [oracle.ROWWISE, oracle.COLWISE])
# rows 48, 96 and 560 leave a warp's group of 64 rows with 3, 2 and 3 of
# its four 16-row slices (the col-wise stores of a partial group)
@pytest.mark.parametrize("shape", [(16, 16), (272, 336), (128, 1024), (400, 192), (48, 64), (96, 128), (560, 96)])
def test_quantize_parity_small(shape, orientation, scaling, rounding, rht):
    rows, cols = shape
    bits = inputs.normal(rows, cols, seed=rows * 7 + cols, outlier_channels=2)
    assert_parity(bits, orientation, scaling=scaling, rounding=rounding, use_rht=rht,
                  sign_mask=0xA55A, seed=123456789, stream_id=5)


@pytest.mark.parametrize("rounding", [0, 1])
def test_quantize_rowwise_ragged_rows(rounding):
    # rows need not be a multiple of 16 for row-wise 1x16 blocks
    bits = inputs.student_t(1000, 64, seed=3)
    assert_parity(bits, oracle.ROWWISE, rounding=rounding, seed=9)


def test_quantize_zero_tensor():
    bits = np.zeros((64, 128), np.uint16)
    for orientation in (oracle.ROWWISE, oracle.COLWISE):
        g = assert_parity(bits, orientation)
        codes, scales, amax, sg, _ = helpers.operand_to_host(g)
        assert amax == 0 and sg == 1 and not codes.any() and not scales.any()


def test_quantize_ties_and_negative_zero():
    """With amax = 2688 the tensor scale is exactly 1 and a block with amax 6
    gets scale 1, so its values hit the E2M1 ties unchanged."""
    row = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5,
                    -3.5, -5.0, -0.1], np.float32)
    x = np.tile(row, (32, 4))
    x[0, 0] = 2688.0
    bits = inputs.to_bf16_bits(x)
    g = assert_parity(bits, oracle.ROWWISE)
    codes, _, _, _, _ = helpers.operand_to_host(g)
    nib = np.stack([codes & 0xF, codes >> 4], -1).reshape(32, -1)
    assert list(nib[1, :16]) == [7, 0, 2, 2, 4, 4, 6, 6, 8, 10, 10, 12, 12, 14, 14, 8]
    assert_parity(bits, oracle.ROWWISE, rounding=1, seed=1)


@pytest.mark.parametrize("shape", [(256, 320), (560, 96)])
def test_quantize_both_orientations_in_one_call(shape):
    bits = inputs.normal(*shape, seed=44, outlier_channels=3)
    x = helpers.to_device_bf16(bits)
    for kw in (dict(), dict(sr=True, seed=4), dict(rht_mask=0x0F0F), dict(rht_mask=0x0F0F, sr=True, seed=5),
               dict(two_d=True), dict(scale46=True), dict(scale46=True, sr=True, seed=6),
               dict(scale46=True, rht_mask=0x3C3C), dict(scale46=True, rht_mask=0x3C3C, sr=True, seed=7)):
        row, col = ops.quantize(x, rowwise=True, colwise=True, stream_id=2, **kw)
        torch.cuda.synchronize()
        common = dict(scaling=1 if kw.get("two_d") else (2 if kw.get("scale46") else 0),
                      rounding=1 if kw.get("sr") else 0,
                      use_rht="rht_mask" in kw, sign_mask=kw.get("rht_mask", 0),
                      seed=kw.get("seed", 0), stream_id=2)
        for op, orient in ((row, oracle.ROWWISE), (col, oracle.COLWISE)):
            codes, scales, amax, sg, _ = helpers.operand_to_host(op)
            ref = oracle.quantize(bits, orient, **common)
            assert amax == ref["amax"] and sg == ref["s_g"]
            assert np.array_equal(codes, ref["codes"]) and np.array_equal(scales, ref["scales"])


def test_quantize_respects_leading_dimension():
    bits = inputs.normal(96, 256, seed=5)
    x_wide = torch.zeros((96, 320), dtype=torch.bfloat16, device="cuda")
    x_wide[:, :256] = helpers.to_device_bf16(bits)
    row, col = ops.quantize(x_wide[:, :256], rowwise=True, colwise=True, sr=True, seed=3)
    torch.cuda.synchronize()
    for op, orient in ((row, oracle.ROWWISE), (col, oracle.COLWISE)):
        codes, scales, amax, sg, _ = helpers.operand_to_host(op)
        ref = oracle.quantize(bits, orient, rounding=1, seed=3)
        assert np.array_equal(codes, ref["codes"]) and np.array_equal(scales, ref["scales"])


# ---- full-size workloads (sampled logical rows; the oracle takes the amax
# over the whole tensor itself) -------------------------------------------
def _ranges(n, k=48):
    mid = (n // 2) // 16 * 16
    return [(0, k), (mid, mid + k), (n - k, n)]


@pytest.mark.parametrize("name,rows,cols,kind,orientation,scaling,rounding,rht", [
    ("c2_X", 8192, 3072, "normal", oracle.ROWWISE, 0, 0, False),
    ("c2_Wqkv_row", 6144, 3072, "weight", oracle.ROWWISE, 1, 0, False),
    ("c2_Wqkv_col", 6144, 3072, "weight", oracle.COLWISE, 1, 0, False),
    ("c3_dY_col", 8192, 9216, "grad", oracle.COLWISE, 0, 1, True),
    ("c3_X_col", 8192, 3072, "normal", oracle.COLWISE, 0, 0, True),
    ("c4_dY_row", 16384, 3072, "grad", oracle.ROWWISE, 0, 1, False),
    ("c4_H_46_row", 16384, 9216, "normal", oracle.ROWWISE, 2, 0, False),
    ("c3_dY_46_col", 8192, 9216, "grad", oracle.COLWISE, 2, 1, True),
    # the quantizer sweep's largest size, 2^29 elements (1 GiB of bf16)
    ("c5_max_row", 65536, 8192, "grad", oracle.ROWWISE, 0, 0, False),
    ("c5_max_2d_col", 65536, 8192, "grad", oracle.COLWISE, 1, 0, False),
])
def test_quantize_parity_full_size(name, rows, cols, kind, orientation, scaling, rounding, rht):
    seed = zlib.crc32(name.encode()) % 1000
    if kind == "normal":
        bits = inputs.normal(rows, cols, seed, outlier_channels=inputs.outlier_count(cols))
    elif kind == "weight":
        bits = inputs.normal(rows, cols, seed, std=0.02)
    else:
        bits = inputs.student_t(rows, cols, seed)
    g = gpu_quantize(bits, orientation, scaling=scaling, rounding=rounding, use_rht=rht,
                     sign_mask=inputs.rht_sign_mask(seed), seed=seed, stream_id=1)
    codes, scales, amax, sg, _ = helpers.operand_to_host(g)
    lrows = rows if orientation == oracle.ROWWISE else cols
    for lr0, lr1 in _ranges(lrows):
        ref = oracle.quantize(bits, orientation, scaling=scaling, rounding=rounding, use_rht=rht,
                              sign_mask=inputs.rht_sign_mask(seed), seed=seed, stream_id=1,
                              rows_subset=(lr0, lr1))
        assert amax == ref["amax"] and sg == ref["s_g"]
        assert np.array_equal(codes[lr0:lr1], ref["codes"])
        assert np.array_equal(scales[lr0:lr1], ref["scales"])


def _check_against_oracle(g, ref):
    codes, scales, amax, sg, tiled = helpers.operand_to_host(g)
    assert amax == ref["amax"] and sg == ref["s_g"]
    assert np.array_equal(codes, ref["codes"]), "codes differ"
    assert np.array_equal(scales, ref["scales"]), "scales differ"
    assert not tiled[helpers.padding_mask(g.rows, g.cols)].any(), "scale padding not zero"


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("shape", [(16, 16), (272, 336), (128, 1024), (400, 192), (1040, 3072), (48, 64),
                                   (96, 128), (560, 96)])
def test_row_col_rht_matches_oracle_and_separate_calls(shape, rounding):
    """nvfp4_quantize_row_col_rht: row-wise without RHT and col-wise with RHT
    from one shared amax pass, identical to the two separate calls."""
    rows, cols = shape
    bits = inputs.student_t(rows, cols, seed=rows + 3 * cols) if rounding else \
        inputs.normal(rows, cols, seed=rows + 3 * cols, outlier_channels=2)
    mask, seed = 0x6C3A, 987654321
    x = helpers.to_device_bf16(bits)
    row, col = ops.quantize_row_col_rht(x, mask, sr=rounding == 1, seed=seed, stream_row=3, stream_col=4)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    _check_against_oracle(row, oracle.quantize(bits, oracle.ROWWISE, rounding=rounding, seed=seed, stream_id=3))
    _check_against_oracle(col, oracle.quantize(bits, oracle.COLWISE, rounding=rounding, use_rht=True,
                                               sign_mask=mask, seed=seed, stream_id=4))
    r2, _ = ops.quantize(x, sr=rounding == 1, seed=seed, stream_id=3)
    _, c2 = ops.quantize(x, sr=rounding == 1, seed=seed, stream_id=4, rht_mask=mask, rowwise=False, colwise=True)
    torch.cuda.synchronize()
    for a, b in ((row, r2), (col, c2)):
        ha, hb = helpers.operand_to_host(a), helpers.operand_to_host(b)
        assert all(np.array_equal(u, v) for u, v in zip(ha, hb))


def test_row_col_rht_zero_tensor():
    """amax 0 gives s_g = 1 on both outputs; the col-wise codes are the
    oracle's (the sign flips of D turn some zeros into -0, code 0x8)."""
    bits = np.zeros((64, 128), np.uint16)
    x = helpers.to_device_bf16(bits)
    row, col = ops.quantize_row_col_rht(x, 0x1)
    torch.cuda.synchronize()
    _check_against_oracle(row, oracle.quantize(bits, oracle.ROWWISE))
    _check_against_oracle(col, oracle.quantize(bits, oracle.COLWISE, use_rht=True, sign_mask=0x1))
    for g in (row, col):
        codes, scales, amax, sg, _ = helpers.operand_to_host(g)
        assert amax == 0 and sg == 1 and not scales.any()
    assert not helpers.operand_to_host(row)[0].any()


@pytest.mark.parametrize("name,rows,cols,rounding,amax_given", [
    ("c4_X", 16384, 3072, 0, False),
    ("c4_dY_down", 16384, 3072, 1, False),
    ("c4_H", 16384, 9216, 0, True),
    ("c4_dY_up", 16384, 9216, 1, True),
])
def test_row_col_rht_full_size_sampled(name, rows, cols, rounding, amax_given):
    """The 3B FFN layer step's four activation/gradient quantizations at 16384
    tokens, in the launch configuration the layer step uses (one pair pass;
    H and dY_up with their two tensor amaxes given, as the producing GEMM
    supplies them): sampled logical rows of both outputs against the oracle,
    which takes each tensor amax over the whole tensor itself."""
    seed = zlib.crc32(name.encode()) % 1000
    bits = inputs.student_t(rows, cols, seed) if rounding else \
        inputs.normal(rows, cols, seed, outlier_channels=inputs.outlier_count(cols))
    mask = inputs.rht_sign_mask(seed)
    x = helpers.to_device_bf16(bits)
    ref_amax = {oracle.ROWWISE: oracle.amax(bits, oracle.ROWWISE), oracle.COLWISE: oracle.amax(bits, oracle.COLWISE,
                                                                                               True, mask)}
    if amax_given:
        amax = torch.tensor([ref_amax[oracle.ROWWISE], ref_amax[oracle.COLWISE]], dtype=torch.float32, device="cuda")
        row, col = ops.quantize_row_col_rht_amax(x, mask, amax, sr=rounding == 1, seed=seed,
                                                 stream_row=1, stream_col=2)
    else:
        row, col = ops.quantize_row_col_rht(x, mask, sr=rounding == 1, seed=seed, stream_row=1, stream_col=2)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    del x
    for op, orientation, rht, stream in ((row, oracle.ROWWISE, False, 1), (col, oracle.COLWISE, True, 2)):
        codes, scales, amax_g, sg, _ = helpers.operand_to_host(op)
        assert amax_g == ref_amax[orientation]
        for lr0, lr1 in _ranges(op.rows):
            ref = oracle.quantize(bits, orientation, rounding=rounding, use_rht=rht, sign_mask=mask, seed=seed,
                                  stream_id=stream, rows_subset=(lr0, lr1), amax_value=ref_amax[orientation])
            assert sg == ref["s_g"]
            assert np.array_equal(codes[lr0:lr1], ref["codes"]), (name, orientation, lr0)
            assert np.array_equal(scales[lr0:lr1], ref["scales"]), (name, orientation, lr0)


# ---- Wgrad re-quantization from the forward's row-wise operand (Eq. (2)) ----
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("shape", [(16, 16), (272, 336), (128, 1024), (400, 192), (1040, 3072)])
def test_requantize_col_rht_matches_oracle(shape, rounding):
    rows, cols = shape
    bits = inputs.normal(rows, cols, seed=rows + 3 * cols, outlier_channels=2)
    x = helpers.to_device_bf16(bits)
    row, _ = ops.quantize(x)
    col = ops.requantize_col_rht(row, 0x5AA5, sr=rounding == 1, seed=77, stream_id=6)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    ref = oracle.requantize_col_rht(oracle.quantize(bits), 0x5AA5, rounding=rounding, seed=77, stream_id=6)
    _check_against_oracle(col, ref)


def test_requantize_col_rht_full_size_sampled():
    rows, cols = 16384, 3072
    bits = inputs.normal(rows, cols, 8, outlier_channels=inputs.outlier_count(cols))
    row, _ = ops.quantize(helpers.to_device_bf16(bits))
    col = ops.requantize_col_rht(row, inputs.rht_sign_mask(8), sr=True, seed=8, stream_id=2)
    torch.cuda.synchronize()
    codes, scales, amax, sg, _ = helpers.operand_to_host(col)
    q = oracle.quantize(bits)
    for lr0, lr1 in _ranges(cols):
        ref = oracle.requantize_col_rht(q, inputs.rht_sign_mask(8), rounding=1, seed=8, stream_id=2,
                                        rows_subset=(lr0, lr1))
        assert amax == ref["amax"] and sg == ref["s_g"]
        assert np.array_equal(codes[lr0:lr1], ref["codes"])
        assert np.array_equal(scales[lr0:lr1], ref["scales"])


# ---- whole tensors at the layer step's size (every code and scale) -------
def test_whole_tensor_c4_dy_up_pair():
    """The layer step's dY_up pair quantization (16384 x 9216, SR in both
    orientations, RHT on the col-wise operand, both tensor amaxes given as
    the producing GEMM supplies them), compared with the oracle over the
    whole tensor: every code byte and every scale of both outputs."""
    rows, cols, seed = 16384, 9216, 17
    bits = inputs.student_t(rows, cols, seed)
    mask = inputs.rht_sign_mask(seed)
    ref_row = oracle.quantize(bits, oracle.ROWWISE, rounding=1, seed=seed, stream_id=3)
    ref_col = oracle.quantize(bits, oracle.COLWISE, rounding=1, use_rht=True, sign_mask=mask, seed=seed,
                              stream_id=4)
    amax = torch.tensor([ref_row["amax"], ref_col["amax"]], dtype=torch.float32, device="cuda")
    row, col = ops.quantize_row_col_rht_amax(helpers.to_device_bf16(bits), mask, amax, sr=True, seed=seed,
                                             stream_row=3, stream_col=4)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    _check_against_oracle(row, ref_row)
    _check_against_oracle(col, ref_col)


def test_whole_tensor_c4_weight_16x16():
    """W_up (9216 x 3072) with 16x16 scaling, both orientations from one
    call, compared with the oracle over the whole tensor."""
    rows, cols, seed = 9216, 3072, 18
    bits = inputs.normal(rows, cols, seed, std=0.02)
    row, col = ops.quantize(helpers.to_device_bf16(bits), two_d=True, rowwise=True, colwise=True)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    _check_against_oracle(row, oracle.quantize(bits, oracle.ROWWISE, scaling=1))
    _check_against_oracle(col, oracle.quantize(bits, oracle.COLWISE, scaling=1))

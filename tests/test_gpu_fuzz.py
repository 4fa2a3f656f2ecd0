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

N_QUANT, N_PAIR, N_GEMM, N_OTHER = 256, 96, 96, 48


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


def _u64(rng):
    """A seed or stream id over the whole 64-bit range."""
    return int(rng.integers(0, 2 ** 64, dtype=np.uint64))


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
    seed, sid = _u64(rng), _u64(rng)
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
    seed, s_row, s_col = _u64(rng), _u64(rng), _u64(rng)
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


def _gemm_operands(rng, case, M, N, K):
    a_bits = _bits(rng, M, K, 8_000 + case, max_log2=20)
    b_bits = _bits(rng, N, K, 9_000 + case, max_log2=20)
    a, _ = ops.quantize(helpers.to_device_bf16(a_bits))
    b, _ = ops.quantize(helpers.to_device_bf16(b_bits))
    return a, b


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_requantize(case):
    """The Wgrad re-quantization of a row-wise operand on random shapes."""
    rng = np.random.default_rng(11_000 + case)
    rows, cols = 16 * int(rng.integers(1, 50)), 16 * int(rng.integers(1, 50))
    sr = bool(rng.integers(0, 2))
    mask = int(rng.integers(0, 1 << 16))
    seed, sid = _u64(rng), _u64(rng)
    bits = _bits(rng, rows, cols, 12_000 + case)
    row, _ = ops.quantize(helpers.to_device_bf16(bits))
    col = ops.requantize_col_rht(row, mask, sr=sr, seed=seed, stream_id=sid)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    _check(col, oracle.requantize_col_rht(oracle.quantize(bits), mask, rounding=int(sr), seed=seed,
                                          stream_id=sid))


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_dequantize(case):
    """x^ = e2m1 s_b s_g of a random operand, into a padded BF16 or FP32 output."""
    rng = np.random.default_rng(13_000 + case)
    rows, cols = int(rng.integers(1, 500)), 16 * int(rng.integers(1, 60))
    bits = _bits(rng, rows, cols, 14_000 + case)
    q, _ = ops.quantize(helpers.to_device_bf16(bits), sr=bool(rng.integers(0, 2)), seed=case)
    fp32 = bool(rng.integers(0, 2))
    esz = 4 if fp32 else 2
    ldy = cols + (16 // esz) * int(rng.integers(0, 3))
    buf = torch.full((rows, ldy), 7.0, dtype=torch.float32 if fp32 else torch.bfloat16, device="cuda")
    st = capi.nvfp4_dequantize(q.struct(), buf.data_ptr(), ldy, capi.NVFP4_OUT_FP32 if fp32 else capi.NVFP4_OUT_BF16,
                               ops.stream_handle())
    assert st == capi.NVFP4_OK
    torch.cuda.synchronize()
    codes, scales, _, sg, _ = helpers.operand_to_host(q)
    ref = oracle.dequantize(codes, scales, sg)
    y = buf[:, :cols].float().cpu().numpy().astype(np.float64)
    want = ref.astype(np.float32).astype(np.float64) if fp32 else oracle.bf16_to_f64(oracle.round_bf16_array(ref))
    assert np.array_equal(y, want), "dequantized values differ"
    assert bool((buf[:, cols:] == 7.0).all()), "write into the output's row padding"


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_gemm_amax(case):
    """The fused-amax GEMM writes the plain GEMM's output and its two amaxes."""
    rng = np.random.default_rng(15_000 + case)
    M, N, K = 16 * int(rng.integers(1, 40)), int(rng.integers(1, 600)), 16 * int(rng.integers(1, 60))
    a, b = _gemm_operands(rng, case, M, N, K)
    mask = int(rng.integers(0, 1 << 16))
    ldd = (N + 7) // 8 * 8 + 8 * int(rng.integers(0, 3))
    out = torch.full((M, ldd), 7.0, dtype=torch.bfloat16, device="cuda")
    d, amax = ops.gemm_amax(a, b, mask, out=out[:, :N])
    d_plain = ops.gemm(a, b)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert torch.equal(d, d_plain)
    assert bool((out[:, N:] == 7.0).all()), "write into the output's row padding"
    d_bits = d.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    got = amax.cpu().numpy()
    assert got[0] == oracle.amax(d_bits, oracle.ROWWISE)
    assert got[1] == oracle.amax(d_bits, oracle.COLWISE, True, mask)


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_gemm_axpby(case):
    """D = alpha A B^T + beta C with random scalars, dtypes and strides."""
    rng = np.random.default_rng(17_000 + case)
    M, N, K = int(rng.integers(1, 400)), int(rng.integers(1, 400)), 16 * int(rng.integers(1, 60))
    a, b = _gemm_operands(rng, case, M, N, K)
    fp32 = bool(rng.integers(0, 2))
    dtype = torch.float32 if fp32 else torch.bfloat16
    alpha, beta = float(rng.uniform(-2, 2)), float(rng.uniform(-2, 2))
    c_bits = inputs.normal(M, N, 18_000 + case)
    c = helpers.to_device_bf16(c_bits).to(dtype)
    ldd = N + int(rng.integers(0, 9))
    out = torch.full((M, ldd), 7.0, dtype=dtype, device="cuda")
    y = ops.gemm_axpby(a, b, alpha, c, beta, out=out[:, :N])
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert bool((out[:, N:] == 7.0).all()), "write into the output's row padding"
    ref, abs_sum = oracle.gemm_axpby_f64(helpers.as_oracle_operand(a), helpers.as_oracle_operand(b), alpha, c_bits,
                                         beta)
    bound = helpers.gemm_bound(abs_sum, ref, not fp32)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"{int((err > bound).sum())} of {err.size} outside the bound"


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_gemm_axpby_staged_c(case):
    """The C term read through the epilogue's staging slices: C and D rows on
    16-byte boundaries while N is ragged (a row's last 16-byte piece of C
    partly past column N), M off the 32-row rounds, BF16 or FP32, half the
    cases with C and D the same buffer."""
    rng = np.random.default_rng(29_000 + case)
    M, K = int(rng.integers(1, 400)), 16 * int(rng.integers(1, 60))
    N = 8 * int(rng.integers(0, 50)) + int(rng.integers(1, 8))
    a, b = _gemm_operands(rng, case, M, N, K)
    fp32 = bool(rng.integers(0, 2))
    dtype, per = (torch.float32, 4) if fp32 else (torch.bfloat16, 8)
    alpha, beta = float(rng.uniform(-2, 2)), float(rng.uniform(-2, 2))
    c_bits = inputs.normal(M, N, 30_000 + case)
    ld = (N + per - 1) // per * per + per * int(rng.integers(0, 3))
    buf = torch.full((M, ld), 7.0, dtype=dtype, device="cuda")
    d = buf[:, :N]
    if rng.integers(0, 2):
        d.copy_(helpers.to_device_bf16(c_bits).to(dtype))
        c = d
    else:
        c = torch.full((M, ld), -3.0, dtype=dtype, device="cuda")[:, :N]
        c.copy_(helpers.to_device_bf16(c_bits).to(dtype))
    y = ops.gemm_axpby(a, b, alpha, c, beta, out=d)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert bool((buf[:, N:] == 7.0).all()), "write into the output's row padding"
    ref, abs_sum = oracle.gemm_axpby_f64(helpers.as_oracle_operand(a), helpers.as_oracle_operand(b), alpha, c_bits,
                                         beta)
    bound = helpers.gemm_bound(abs_sum, ref, not fp32)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"{int((err > bound).sum())} of {err.size} outside the bound"


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_noalloc_equals_quantize(case):
    """nvfp4_quantize_noalloc gives the regular call's result."""
    rng = np.random.default_rng(19_000 + case)
    rows, cols = 16 * int(rng.integers(1, 40)), 16 * int(rng.integers(1, 40))
    bits = _bits(rng, rows, cols, 20_000 + case)
    x = helpers.to_device_bf16(bits)
    scaling = int(rng.integers(0, 3))
    sr = bool(rng.integers(0, 2))
    seed = _u64(rng)
    r1, c1 = ops.quantize(x, two_d=scaling == 1, scale46=scaling == 2, sr=sr, seed=seed, colwise=True)
    r2, c2 = ops.alloc_operand(rows, cols), ops.alloc_operand(cols, rows)
    st = capi.nvfp4_quantize_noalloc(x.data_ptr(), rows, cols, x.stride(0), scaling, int(sr), seed, 0,
                                     capi.NVFP4_ROWWISE | capi.NVFP4_COLWISE, r2.struct(), c2.struct(),
                                     ops.stream_handle())
    assert st == capi.NVFP4_OK
    torch.cuda.synchronize()
    for g, h in ((r1, r2), (c1, c2)):
        hg, hh = helpers.operand_to_host(g), helpers.operand_to_host(h)
        assert hg[2] == hh[2] and hg[3] == hh[3]
        assert np.array_equal(hg[0], hh[0]) and np.array_equal(hg[1], hh[1])


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_gemm_lora(case):
    """D = A B^T + beta U V^T with a random rank (a multiple of 64), shapes,
    beta and output dtype and leading dimension; tolerance as in the fixed
    cases (the GEMM bound plus 2^-8 of sum |beta u v|, U being rounded to
    BF16 once more on its way into the tensor cores)."""
    rng = np.random.default_rng(21_000 + case)
    M, N, K = int(rng.integers(1, 400)), int(rng.integers(1, 400)), 16 * int(rng.integers(1, 60))
    r = 64 * int(rng.integers(1, 4))
    a, b = _gemm_operands(rng, case, M, N, K)
    beta = float(rng.uniform(-2, 2))
    u_bits = inputs.to_bf16_bits(rng.standard_normal((M, r)).astype(np.float32) * float(rng.uniform(0.1, 4)))
    v_bits = inputs.to_bf16_bits(rng.standard_normal((N, r)).astype(np.float32) * float(rng.uniform(0.1, 4)))
    fp32 = bool(rng.integers(0, 2))
    dtype = torch.float32 if fp32 else torch.bfloat16
    ldd = N + int(rng.integers(0, 9))
    out = torch.full((M, ldd), 7.0, dtype=dtype, device="cuda")
    y = ops.gemm_lora(a, b, helpers.to_device_bf16(u_bits), helpers.to_device_bf16(v_bits), beta, out=out[:, :N])
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert bool((out[:, N:] == 7.0).all()), "write into the output's row padding"
    ref, abs_sum, lora_abs = oracle.gemm_lora_f64(helpers.as_oracle_operand(a), helpers.as_oracle_operand(b), u_bits,
                                                  v_bits, beta)
    bound = helpers.gemm_bound(abs_sum, ref, not fp32) + 2.0 ** -8 * lora_abs
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"{int((err > bound).sum())} of {err.size} outside the bound"


@pytest.mark.parametrize("case", range(8))
def test_fuzz_quantize_large(case):
    """Shapes of several persistent-grid rounds (up to 4096 x 4096), every
    code and scale compared."""
    rng = np.random.default_rng(23_000 + case)
    rows, cols = 16 * int(rng.integers(64, 257)), 16 * int(rng.integers(64, 257))
    scaling = int(rng.integers(0, 3))
    rounding = int(rng.integers(0, 2))
    rht = scaling != 1 and bool(rng.integers(0, 2))
    mask = int(rng.integers(0, 1 << 16))
    seed, sid = _u64(rng), _u64(rng)
    bits = _bits(rng, rows, cols, 24_000 + case)
    row, col = ops.quantize(helpers.to_device_bf16(bits), two_d=scaling == 1, scale46=scaling == 2,
                            sr=rounding == 1, rht_mask=mask if rht else None, seed=seed, stream_id=sid,
                            rowwise=True, colwise=True)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    kw = dict(scaling=scaling, rounding=rounding, use_rht=rht, sign_mask=mask, seed=seed, stream_id=sid)
    _check(row, oracle.quantize(bits, oracle.ROWWISE, **kw))
    _check(col, oracle.quantize(bits, oracle.COLWISE, **kw))


@pytest.mark.parametrize("case", range(8))
def test_fuzz_gemm_large_sampled_rows(case):
    """GEMMs of several tile waves (M, N up to 3000, K up to 4096), compared
    on 32 sampled rows with every column."""
    rng = np.random.default_rng(25_000 + case)
    M, N = int(rng.integers(600, 3000)), int(rng.integers(600, 3000))
    K = 16 * int(rng.integers(16, 257))
    a, b = _gemm_operands(rng, case, M, N, K)
    fp32 = bool(rng.integers(0, 2))
    y = ops.gemm(a, b, out_dtype=torch.float32 if fp32 else torch.bfloat16)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    ids = np.sort(rng.choice(M, 32, replace=False))
    ref, abs_sum = oracle.gemm_f64(helpers.as_oracle_operand(a, ids), helpers.as_oracle_operand(b))
    bound = helpers.gemm_bound(abs_sum, ref, not fp32)
    err = np.abs(y[torch.from_numpy(ids).cuda()].float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"{int((err > bound).sum())} of {err.size} outside the bound"


@pytest.mark.parametrize("case", range(N_OTHER))
def test_fuzz_gemm_axpby_in_place(case):
    """D = alpha A B^T + beta D with C and D the same buffer (each element is
    read before it is written), random ragged N and leading dimension."""
    rng = np.random.default_rng(27_000 + case)
    M, N, K = int(rng.integers(1, 400)), int(rng.integers(1, 400)), 16 * int(rng.integers(1, 60))
    a, b = _gemm_operands(rng, case, M, N, K)
    fp32 = bool(rng.integers(0, 2))
    dtype = torch.float32 if fp32 else torch.bfloat16
    alpha, beta = float(rng.uniform(-2, 2)), float(rng.uniform(-2, 2))
    c_bits = inputs.normal(M, N, 28_000 + case)
    ldd = N + int(rng.integers(0, 9))
    buf = torch.full((M, ldd), 7.0, dtype=dtype, device="cuda")
    d = buf[:, :N]
    d.copy_(helpers.to_device_bf16(c_bits).to(dtype))
    y = ops.gemm_axpby(a, b, alpha, d, beta, out=d)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert bool((buf[:, N:] == 7.0).all()), "write into the output's row padding"
    ref, abs_sum = oracle.gemm_axpby_f64(helpers.as_oracle_operand(a), helpers.as_oracle_operand(b), alpha, c_bits,
                                         beta)
    bound = helpers.gemm_bound(abs_sum, ref, not fp32)
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), f"{int((err > bound).sum())} of {err.size} outside the bound"

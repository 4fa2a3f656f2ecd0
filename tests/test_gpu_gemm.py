"""GPU parity of the NVFP4 GEMM against the oracle's FP64 GEMM, through the C
ABI.  Tolerance: |y - y_ref| <= 1e-4 * sum_k |a_k b_k| + 1e-6 per element,
plus half a bfloat16 ulp of y_ref for BF16 output (the rounding of the output
itself)."""
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


def _random_operand_host(rng, rows, K):
    codes = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (rows, K // 16), dtype=np.uint8)   # finite E4M3 >= 0
    s_g = np.float32(rng.uniform(0.05, 2.0))
    return dict(codes=codes, scales=scales, s_g=s_g)


def _upload(host, rows, K):
    op = ops.alloc_operand(rows, K)
    codes = np.zeros((rows, op.ld_codes), np.uint8)
    codes[:, : K // 2] = host["codes"]
    tiled = np.zeros(op.scales.numel(), np.uint8)
    if rows and K:
        tiled[helpers.scale_index_map(rows, K)] = host["scales"]
    op.codes.copy_(torch.from_numpy(codes))
    op.scales.copy_(torch.from_numpy(tiled))
    op.global_scale.fill_(float(host["s_g"]))
    op.amax.fill_(0.0)
    return op


def _check(y, y_ref, abs_sum, bf16):
    bound = helpers.gemm_bound(abs_sum, y_ref, bf16)
    err = np.abs(y.astype(np.float64) - y_ref)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (f"{int((err > bound).sum())} of {err.size} outside the bound; "
                                  f"worst at {worst}: y={y[worst]} ref={y_ref[worst]} "
                                  f"bound={bound[worst]}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (1, 1, 16), (200, 300, 320), (130, 260, 80),
                                   (384, 512, 1024), (257, 129, 4096), (64, 1000, 192)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_random_operands(M, N, K, out_dtype):
    rng = np.random.default_rng(M * 1_000_003 + N * 1009 + K)
    a_h = _random_operand_host(rng, M, K)
    b_h = _random_operand_host(rng, N, K)
    a, b = _upload(a_h, M, K), _upload(b_h, N, K)
    y = ops.gemm(a, b, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    y_ref, abs_sum = oracle.gemm_f64(a_h, b_h)
    _check(y.float().cpu().numpy(), y_ref, abs_sum, out_dtype == torch.bfloat16)


def test_gemm_output_leading_dimension_and_no_overwrite():
    rng = np.random.default_rng(3)
    M, N, K = 136, 264, 128
    a_h, b_h = _random_operand_host(rng, M, K), _random_operand_host(rng, N, K)
    a, b = _upload(a_h, M, K), _upload(b_h, N, K)
    big = torch.full((M + 3, 320), 7.0, dtype=torch.float32, device="cuda")
    ops.gemm(a, b, out=big[:M, :N])
    torch.cuda.synchronize()
    y_ref, abs_sum = oracle.gemm_f64(a_h, b_h)
    host = big.cpu().numpy()
    _check(host[:M, :N], y_ref, abs_sum, False)
    assert np.all(host[:M, N:] == 7.0) and np.all(host[M:] == 7.0)


def test_gemm_zero_k_gives_zero():
    a = ops.alloc_operand(64, 0)
    b = ops.alloc_operand(32, 0)
    a.global_scale.fill_(1.0)
    b.global_scale.fill_(1.0)
    y = torch.full((64, 32), 5.0, dtype=torch.float32, device="cuda")
    ops.gemm(a, b, out=y)
    assert torch.count_nonzero(y).item() == 0


def _quantized_pair(x_bits, w_bits, a_kw, b_kw):
    """GPU and oracle quantizations of the same seeded inputs."""
    xa = helpers.to_device_bf16(x_bits)
    xb = helpers.to_device_bf16(w_bits)

    def gpu(x, orientation, scaling=0, rounding=0, use_rht=False, sign_mask=0, seed=0, stream_id=0):
        row, col = ops.quantize(x, two_d=scaling == 1, sr=rounding == 1,
                                rht_mask=sign_mask if use_rht else None, seed=seed, stream_id=stream_id,
                                rowwise=orientation == oracle.ROWWISE,
                                colwise=orientation == oracle.COLWISE)
        return row if orientation == oracle.ROWWISE else col

    return gpu(xa, **a_kw), gpu(xb, **b_kw)


def test_gemm_c1_single_linear_forward():
    """128 tokens x 1024 -> 1024, outlier channels, 1x16 RNE on both operands."""
    wl = inputs.c1_single_linear()
    x_bits, w_bits = wl.make("X"), wl.make("W")
    ga, gb = _quantized_pair(x_bits, w_bits, dict(orientation=oracle.ROWWISE),
                             dict(orientation=oracle.ROWWISE))
    qa = oracle.quantize(x_bits)
    qb = oracle.quantize(w_bits)
    y_ref, abs_sum = oracle.gemm_f64(qa, qb)
    for dt in (torch.float32, torch.bfloat16):
        y = ops.gemm(ga, gb, out_dtype=dt)
        torch.cuda.synchronize()
        _check(y.float().cpu().numpy(), y_ref, abs_sum, dt == torch.bfloat16)


# Full-size GEMMs: (A rows, A cols, A kind, A quantizer kw, B rows, B cols, B
# kind, B quantizer kw, fused amax).  A and B are the bf16 tensors the
# operands are quantized from (a col-wise operand is the transpose of its
# tensor); kinds as in the 3B workloads (activations with outlier channels,
# weights N(0, 0.02^2), gradients t(3) * 1e-3), gradients with SR and the
# Wgrad operands with the RHT as in the layer step.
_GRAD_SR_ROW = dict(orientation=oracle.ROWWISE, rounding=1, seed=21, stream_id=1)
_GRAD_SR_COL = dict(orientation=oracle.COLWISE, rounding=1, use_rht=True, sign_mask=0x6B2D, seed=21, stream_id=2)
_ACT_COL = dict(orientation=oracle.COLWISE, use_rht=True, sign_mask=0x6B2D)
_ROW = dict(orientation=oracle.ROWWISE)
_W_ROW = dict(orientation=oracle.ROWWISE, scaling=1)
_W_COL = dict(orientation=oracle.COLWISE, scaling=1)
T4, T2 = 16384, 8192
FULL = {
    # attention projections at 8192 tokens (3072 -> 6144 QKV, 3072 -> 3072 O)
    "c2_fprop_qkv": (T2, 3072, "normal", _ROW, 6144, 3072, "weight", _W_ROW, False),
    "c2_fprop_o": (T2, 3072, "normal", _ROW, 3072, 3072, "weight", _W_ROW, False),
    "c2_dgrad_qkv": (T2, 6144, "grad", _ROW, 6144, 3072, "weight", _W_COL, False),
    "c2_dgrad_o": (T2, 3072, "grad", _ROW, 3072, 3072, "weight", _W_COL, False),
    # FFN Wgrad at 8192 tokens
    "c3_wgrad": (T2, 9216, "grad", _GRAD_SR_COL, T2, 3072, "normal", _ACT_COL, False),
    # the FFN layer step at 16384 tokens: up 3072 -> 9216, down 9216 -> 3072;
    # fprop_up and dgrad_down take their output's two amaxes in the epilogue
    "c4_fprop_up": (T4, 3072, "normal", _ROW, 9216, 3072, "weight", _W_ROW, True),
    "c4_fprop_down": (T4, 9216, "normal", _ROW, 3072, 9216, "weight", _W_ROW, False),
    "c4_dgrad_down": (T4, 3072, "grad", _GRAD_SR_ROW, 3072, 9216, "weight", _W_COL, True),
    "c4_dgrad_up": (T4, 9216, "grad", _GRAD_SR_ROW, 9216, 3072, "weight", _W_COL, False),
    "c4_wgrad_down": (T4, 3072, "grad", _GRAD_SR_COL, T4, 9216, "normal", _ACT_COL, False),
    "c4_wgrad_up": (T4, 9216, "grad", _GRAD_SR_COL, T4, 3072, "normal", _ACT_COL, False),
}


def _make(kind, rows, cols, seed):
    if kind == "normal":
        return inputs.normal(rows, cols, seed, outlier_channels=inputs.outlier_count(cols))
    if kind == "weight":
        return inputs.normal(rows, cols, seed, std=0.02)
    return inputs.student_t(rows, cols, seed)


def _gpu_operand(bits, orientation, scaling=0, rounding=0, use_rht=False, sign_mask=0, seed=0, stream_id=0):
    row, col = ops.quantize(helpers.to_device_bf16(bits), two_d=scaling == 1, sr=rounding == 1,
                            rht_mask=sign_mask if use_rht else None, seed=seed, stream_id=stream_id,
                            rowwise=orientation == oracle.ROWWISE, colwise=orientation == oracle.COLWISE)
    return row if orientation == oracle.ROWWISE else col


def oracle_rows(bits, kw, rows):
    """The oracle's quantization of the listed logical rows of one
    orientation, with the tensor amax taken over the whole tensor."""
    kw = dict(kw)
    orientation = kw.pop("orientation", oracle.ROWWISE)
    amax = oracle.amax(bits, orientation, kw.get("use_rht", False), kw.get("sign_mask", 0))
    parts = [oracle.quantize(bits, orientation, rows_subset=(int(r), int(r) + 1), amax_value=amax, **kw)
             for r in rows]
    return dict(codes=np.concatenate([q["codes"] for q in parts]),
                scales=np.concatenate([q["scales"] for q in parts]), s_g=parts[0]["s_g"])


def sample_rows(M, n=24, seed=7):
    rows = np.sort(np.random.default_rng(seed).choice(M, n, replace=False))
    rows[0], rows[-1] = 0, M - 1
    return rows


@pytest.mark.parametrize("name", sorted(FULL))
def test_gemm_full_size_sampled_rows(name):
    """Sampled rows (each with all N columns) of the full-size GEMM against the
    oracle's FP64 GEMM of the oracle's own quantization of the same inputs;
    the fused-amax GEMMs also write their two tensor amaxes, checked against
    the oracle's amax of the tensor the GEMM wrote."""
    ar, ac, ak, akw, br, bc, bk, bkw, fused = FULL[name]
    a_bits, b_bits = _make(ak, ar, ac, 11), _make(bk, br, bc, 12)
    ga, gb = _gpu_operand(a_bits, **akw), _gpu_operand(b_bits, **bkw)
    mask = 0x39C6
    if fused:
        y, amax = ops.gemm_amax(ga, gb, mask)
    else:
        y = ops.gemm(ga, gb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    M, N = ga.rows, gb.rows
    del ga, gb
    rows = sample_rows(M)
    qa = oracle_rows(a_bits, akw, rows)
    bkw_ = dict(bkw)
    qb = oracle.quantize(b_bits, bkw_.pop("orientation"), **bkw_)
    y_ref, abs_sum = oracle.gemm_f64(qa, qb)
    _check(y[torch.from_numpy(rows).cuda()].float().cpu().numpy(), y_ref, abs_sum, True)
    if fused:
        # the two tensor amaxes the pair quantization of D takes: max |D| and
        # the col-wise RHT amax (16-row blocks of D's columns)
        d_bits = y.view(torch.int16).cpu().numpy().view(np.uint16)
        got = amax.cpu().numpy()
        assert got[0] == oracle.amax(d_bits, oracle.ROWWISE)
        assert got[1] == oracle.amax(d_bits, oracle.COLWISE, True, mask)


def test_wgrad_rht_cancels_in_the_product():
    """(U A)^T (U B) = A^T B: the Wgrad GEMM of RHT-quantized operands tracks the
    un-rotated product within the quantization noise (Full-Stack FP4 Eq. (2))."""
    T, N, K = 2048, 256, 256
    dy = inputs.student_t(T, N, 21)
    x = inputs.normal(T, K, 22)
    ga, gb = _quantized_pair(dy, x, dict(orientation=oracle.COLWISE, rounding=1, use_rht=True,
                                         sign_mask=0x1357, seed=5),
                             dict(orientation=oracle.COLWISE, use_rht=True, sign_mask=0x1357))
    y = ops.gemm(ga, gb, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    exact = inputs.bf16_bits_to_f32(dy).astype(np.float64).T @ inputs.bf16_bits_to_f32(x).astype(np.float64)
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.3          # quantization noise only (about 0.17 here)
    # with different sign diagonals the rotations do not cancel
    ga2, gb2 = _quantized_pair(dy, x, dict(orientation=oracle.COLWISE, use_rht=True, sign_mask=0x1357),
                               dict(orientation=oracle.COLWISE, use_rht=True, sign_mask=0xECA8))
    y2 = ops.gemm(ga2, gb2, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    assert np.linalg.norm(y2 - exact) / np.linalg.norm(exact) > 0.8


# ---- LoRA-SVD projection: the BF16 low-rank branch fused into the GEMM ----
@pytest.mark.parametrize("M,N,K,r,beta", [(128, 256, 256, 64, 0.5), (200, 300, 320, 128, -1.25),
                                          (384, 512, 3072, 64, 2.0), (130, 260, 80, 192, 0.75)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_lora_matches_oracle(M, N, K, r, beta, out_dtype):
    """D = s_gA s_gB A B^T + beta U V^T ("Full-Stack FP4", Sec. 3.2 Eq. (1)).
    Tolerance: the GEMM bound plus 2^-8 of sum |beta u v| (U is scaled and
    rounded to BF16 once more on its way into the tensor cores)."""
    rng = np.random.default_rng(M * 7 + N * 11 + K * 13 + r)
    a_h = _random_operand_host(rng, M, K)
    b_h = _random_operand_host(rng, N, K)
    a, b = _upload(a_h, M, K), _upload(b_h, N, K)
    u_bits = inputs.to_bf16_bits(rng.standard_normal((M, r)).astype(np.float32) * 4.0)
    v_bits = inputs.to_bf16_bits(rng.standard_normal((N, r)).astype(np.float32) * 0.5)
    u = helpers.to_device_bf16(u_bits)
    v = helpers.to_device_bf16(v_bits)
    y = ops.gemm_lora(a, b, u, v, beta, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    y_ref, abs_sum, lora_abs = oracle.gemm_lora_f64(a_h, b_h, u_bits, v_bits, beta)
    bound = helpers.gemm_bound(abs_sum, y_ref, out_dtype == torch.bfloat16) + 2.0 ** -8 * lora_abs
    err = np.abs(y.float().cpu().numpy().astype(np.float64) - y_ref)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (int((err > bound).sum()), worst, y_ref[worst], bound[worst])
    if out_dtype == torch.float32:
        # the low-rank term on its own: the same GEMM without it differs by
        # beta U V^T up to U's BF16 rounding and the roundings of the FP32
        # accumulator as each of the r/16 BF16 MMAs adds onto it
        y_plain = ops.gemm(a, b, out_dtype=torch.float32).cpu().numpy().astype(np.float64)
        y_l = y.cpu().numpy().astype(np.float64)
        lora_ref = y_ref - oracle.gemm_f64(a_h, b_h)[0]
        tight = 2.0 ** -8 * lora_abs + (r / 16 + 2) * 2.0 ** -23 * (np.abs(y_plain) + np.abs(y_l)) + 1e-30
        dev = np.abs((y_l - y_plain) - lora_ref)
        bad = np.argwhere(dev > tight)
        assert bad.size == 0, (len(bad), bad[:6].tolist(), [(float(dev[i, j]), float(tight[i, j]),
                               float(lora_ref[i, j]), float(y_l[i, j] - y_plain[i, j])) for i, j in bad[:4]])


def test_gemm_lora_full_size_fprop_up_sampled():
    """The 16384x9216x3072 Fprop of the up projection with a rank-64 branch
    (U = X L1^T, V = L2 as random BF16), sampled rows."""
    M, N, K, r = 16384, 9216, 3072, 64
    x_bits = inputs.normal(M, K, 3, outlier_channels=inputs.outlier_count(K))
    w_bits = inputs.normal(N, K, 4, std=0.02)
    a, _ = ops.quantize(helpers.to_device_bf16(x_bits))
    b, _ = ops.quantize(helpers.to_device_bf16(w_bits), two_d=True)
    rng = np.random.default_rng(5)
    u_bits = inputs.to_bf16_bits(rng.standard_normal((M, r)).astype(np.float32))
    v_bits = inputs.to_bf16_bits(rng.standard_normal((N, r)).astype(np.float32) * 0.02)
    y = ops.gemm_lora(a, b, helpers.to_device_bf16(u_bits), helpers.to_device_bf16(v_bits), 0.5)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    rows = np.sort(np.random.default_rng(6).choice(M, 96, replace=False))
    qa = oracle.quantize(x_bits, rows_subset=None)
    qb = oracle.quantize(w_bits, scaling=1)
    y_ref, abs_sum, lora_abs = oracle.gemm_lora_f64(qa, qb, u_bits, v_bits, 0.5, row_ids=rows)
    bound = helpers.gemm_bound(abs_sum, y_ref, True) + 2.0 ** -8 * lora_abs
    err = np.abs(y.float().cpu().numpy()[rows].astype(np.float64) - y_ref)
    assert np.all(err <= bound), int((err > bound).sum())

"""GPU parity of the GEMM with a C term (nvfp4_gemm_axpby) and of the NVFP4
Newton-Schulz step (nvfp4_newton_schulz_step, "Full-Stack FP4" Sec. 3.4)
against the oracle, through the C ABI.

The step is checked stage by stage: each of A_k, B_k and X_k+1 is compared
with the oracle's value computed from the GPU's own inputs to that stage (the
quantizations of a stage's input are bit-exact on both sides; the products are
compared within the GEMM tolerance, |y - y_ref| <= 1e-4 * (|alpha| sum_k
|a_k b_k| + |beta c|) + 1e-6 plus half a bf16 ulp of y_ref for the output's
own rounding)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, ops
from tests import helpers

pytestmark = pytest.mark.gpu

MUON = (3.4445, -4.7750, 2.0315)


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def _f32(v):
    return float(np.float32(v))


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check(y, y_ref, abs_sum, bf16):
    bound = helpers.gemm_bound(abs_sum, y_ref, bf16)
    err = np.abs(y.astype(np.float64) - y_ref)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (f"{int((err > bound).sum())} of {err.size} outside the bound; "
                                  f"worst at {worst}: y={y[worst]} ref={y_ref[worst]} bound={bound[worst]}")


def _quantized_pair(rng, M, N, K):
    xa = oracle.round_bf16_array(rng.standard_normal((M, K)))
    xb = oracle.round_bf16_array(rng.standard_normal((N, K)))
    a, _ = ops.quantize(helpers.to_device_bf16(xa))
    b, _ = ops.quantize(helpers.to_device_bf16(xb))
    torch.cuda.synchronize()
    return a, b


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 300, 320), (257, 129, 1024), (64, 1000, 192)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_axpby(M, N, K, out_dtype):
    rng = np.random.default_rng(M * 7919 + N * 31 + K)
    a, b = _quantized_pair(rng, M, N, K)
    c_host = rng.standard_normal((M, N)).astype(np.float32)
    if out_dtype == torch.bfloat16:
        c_bits = oracle.round_bf16_array(c_host)
        c = helpers.to_device_bf16(c_bits)
    else:
        c = torch.from_numpy(c_host).cuda()
        c_bits = None
    alpha, beta = _f32(-1.375), _f32(0.6)
    y = ops.gemm_axpby(a, b, alpha, c, beta, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    qa, qb = helpers.as_oracle_operand(a), helpers.as_oracle_operand(b)
    y_ref, abs_sum = oracle.gemm_axpby_f64(qa, qb, alpha, c_bits, beta) if c_bits is not None else \
        oracle.gemm_axpby_f64(qa, qb, alpha, None, 0.0)
    if c_bits is None:   # FP32 C: add the term here, in float64
        y_ref = y_ref + beta * c_host.astype(np.float64)
        abs_sum = abs_sum + abs(beta) * np.abs(c_host.astype(np.float64))
    _check(y.float().cpu().numpy(), y_ref, abs_sum, out_dtype == torch.bfloat16)


def test_gemm_axpby_in_place_and_beta_zero():
    rng = np.random.default_rng(17)
    M, N, K = 272, 384, 512
    a, b = _quantized_pair(rng, M, N, K)
    qa, qb = helpers.as_oracle_operand(a), helpers.as_oracle_operand(b)
    c_bits = oracle.round_bf16_array(rng.standard_normal((M, N)))
    d = helpers.to_device_bf16(c_bits)
    ops.gemm_axpby(a, b, 0.5, d, -2.0, out=d)          # D = 0.5 A B^T - 2 D, in place
    y_ref, abs_sum = oracle.gemm_axpby_f64(qa, qb, 0.5, c_bits, -2.0)
    _check(d.float().cpu().numpy(), y_ref, abs_sum, True)
    # beta = 0: C is not read (NULL), D = alpha A B^T
    y = ops.gemm_axpby(a, b, 3.0, None, 0.0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    y_ref, abs_sum = oracle.gemm_axpby_f64(qa, qb, 3.0, None, 0.0)
    _check(y.cpu().numpy(), y_ref, abs_sum, False)
    assert ops.device_error() == capi.NVFP4_OK


def _ns_input(m, n, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((m, n))
    return oracle.round_bf16_array(g / np.linalg.norm(g))


def _q(bits, orientation, mask):
    return oracle.quantize(bits, orientation, scaling=2, rounding=0, use_rht=True, sign_mask=mask)


def _check_ns_stages(x_bits, a_bits, b_bits, out_bits, coef, mask, row_ids=None):
    a, b, c = (_f32(v) for v in coef)
    sub = (lambda t: t) if row_ids is None else (lambda t: t[row_ids])
    # stage 1: A = qX qX^T from X
    qx = _q(x_bits, oracle.ROWWISE, mask)
    a_ref, ab = oracle.gemm_f64(qx, qx, row_ids=row_ids)
    _check(sub(oracle.bf16_to_f64(a_bits)), a_ref, ab, True)
    # stage 2: B = b A + c qA qA' from the GPU's A
    qa, qac = _q(a_bits, oracle.ROWWISE, mask), _q(a_bits, oracle.COLWISE, mask)
    b_ref, ab = oracle.gemm_axpby_f64(qa, qac, c, a_bits, b, row_ids=row_ids)
    _check(sub(oracle.bf16_to_f64(b_bits)), b_ref, ab, True)
    # stage 3: X_out = a X + qB qX' from the GPU's B
    qb, qxc = _q(b_bits, oracle.ROWWISE, mask), _q(x_bits, oracle.COLWISE, mask)
    x_ref, ab = oracle.gemm_axpby_f64(qb, qxc, 1.0, x_bits, a, row_ids=row_ids)
    _check(sub(oracle.bf16_to_f64(out_bits)), x_ref, ab, True)


@pytest.mark.parametrize("m,n", [(128, 256), (272, 528), (64, 3072), (512, 512)])
@pytest.mark.parametrize("coef", [MUON, (1.5, -0.5, 0.0)])
def test_newton_schulz_step_stages(m, n, coef):
    mask = 0xC3A5 ^ m
    x_bits = _ns_input(m, n, m + n)
    x = helpers.to_device_bf16(x_bits)
    ws = torch.empty(capi.nvfp4_newton_schulz_workspace_size(m, n), dtype=torch.uint8, device="cuda")
    out = ops.newton_schulz_step(x, *coef, mask, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    a_k, b_k = ops.ns_intermediates(ws, m)
    _check_ns_stages(x_bits, _bits(a_k), _bits(b_k), _bits(out), coef, mask)


def test_newton_schulz_step_in_place_matches_out_of_place():
    m, n = 160, 320
    x_bits = _ns_input(m, n, 5)
    x = helpers.to_device_bf16(x_bits)
    out = ops.newton_schulz_step(x, *MUON, 0x0F1E)
    x2 = x.clone()
    ops.newton_schulz_step(x2, *MUON, 0x0F1E, out=x2)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), x2.view(torch.int16))


def test_newton_schulz_iterations_stay_near_orthogonal():
    # the cubic map (1.5, -0.5, 0) run 12 times on the GPU keeps the singular
    # values near 1, as the oracle's pin shows for the same iteration
    m, n = 256, 768
    rng = np.random.default_rng(9)
    g = rng.standard_normal((m, n))
    x = helpers.to_device_bf16(oracle.round_bf16_array(0.9 * g / np.linalg.norm(g, 2)))
    ws = torch.empty(capi.nvfp4_newton_schulz_workspace_size(m, n), dtype=torch.uint8, device="cuda")
    for k in range(12):
        x = ops.newton_schulz_step(x, 1.5, -0.5, 0.0, (0x1357 + 97 * k) & 0xFFFF, workspace=ws)
    sv = torch.linalg.svdvals(x.float()).cpu().numpy()
    assert 0.8 < sv.min() and sv.max() < 1.2, (sv.min(), sv.max())


def test_newton_schulz_step_ffn_weight_shape_sampled_rows():
    # the 3B model's FFN weight (3072 x 9216): stages checked on sampled rows
    m, n = 3072, 9216
    x_bits = _ns_input(m, n, 21)
    x = helpers.to_device_bf16(x_bits)
    ws = torch.empty(capi.nvfp4_newton_schulz_workspace_size(m, n), dtype=torch.uint8, device="cuda")
    out = ops.newton_schulz_step(x, *MUON, 0x5A5A, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    a_k, b_k = ops.ns_intermediates(ws, m)
    rows = np.sort(np.random.default_rng(2).choice(m, 24, replace=False)).astype(np.int64)
    _check_ns_stages(x_bits, _bits(a_k), _bits(b_k), _bits(out), MUON, 0x5A5A, row_ids=rows)


def test_newton_schulz_step_argument_errors():
    x = torch.zeros((40, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(capi.nvfp4_newton_schulz_workspace_size(48, 64), dtype=torch.uint8, device="cuda")
    st = capi.nvfp4_newton_schulz_step(x.data_ptr(), 40, 64, 64, 1.0, 0.0, 0.0, 0, x.data_ptr(), 64,
                                       ws.data_ptr(), ws.numel(), None)
    assert st == capi.NVFP4_ERR_SHAPE          # m % 16 != 0
    y = torch.zeros((48, 64), dtype=torch.bfloat16, device="cuda")
    st = capi.nvfp4_newton_schulz_step(y.data_ptr(), 48, 64, 64, 1.0, 0.0, 0.0, 0, y.data_ptr(), 64,
                                       ws.data_ptr(), 16, None)
    assert st == capi.NVFP4_ERR_WORKSPACE
    st = capi.nvfp4_newton_schulz_step(y.data_ptr(), 48, 64, 64, float("nan"), 0.0, 0.0, 0, y.data_ptr(), 64,
                                       ws.data_ptr(), ws.numel(), None)
    assert st == capi.NVFP4_ERR_INVALID_ARG

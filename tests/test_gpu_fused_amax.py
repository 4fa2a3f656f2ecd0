"""The output amax fused into the producing GEMM (nvfp4_gemm_amax) and the
quantization that takes it (nvfp4_quantize_row_col_rht_amax): the
quantization's amax pass moves into the GEMM epilogue ("Full-Stack FP4",
Appendix 9, on fusing quantization with the producing operation).

The fused maxima are checked against their definition applied to the GEMM's
own BF16 output (max |D|, and max |H16 D d| / 4 over 16-row blocks in the
quantizer's rounding order, written out below in float32 numpy); the
amax-taking quantization is checked against the oracle on host inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
from tests import helpers
from tests.test_gpu_gemm import _random_operand_host, _upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def _rotated_amax_f32(d, mask):
    """max |H16 diag(mask) d| / 4 over the 16-row blocks of each column of d
    (float32): signs, butterfly stages 0..3 as (a + b, a - b), then 1/4."""
    m, n = d.shape
    t = d.astype(np.float32).reshape(m // 16, 16, n).copy()
    signs = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)], np.float32)
    t *= signs[None, :, None]
    for s in range(4):
        h = 1 << s
        for i in range(16):
            if i & h:
                continue
            a, b = t[:, i, :].copy(), t[:, i | h, :].copy()
            t[:, i, :] = a + b
            t[:, i | h, :] = a - b
    return np.float32(np.abs(t).max() * np.float32(0.25)) if t.size else np.float32(0)


@pytest.mark.parametrize("M,N,K,mask", [(128, 256, 256, 0x1234), (208, 296, 320, 0xFFFF), (384, 512, 1024, 0),
                                        (1040, 3072, 3072, 0xA5C3)])
def test_gemm_amax_equals_definition_on_its_output(M, N, K, mask):
    rng = np.random.default_rng(M + N + K)
    a, b = _upload(_random_operand_host(rng, M, K), M, K), _upload(_random_operand_host(rng, N, K), N, K)
    d, amax = ops.gemm_amax(a, b, mask)
    d_plain = ops.gemm(a, b)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    assert torch.equal(d, d_plain), "the fused-amax GEMM must write the same output"
    df = d.float().cpu().numpy()
    got = amax.cpu().numpy()
    assert got[0] == np.float32(np.abs(df).max())
    assert got[1] == _rotated_amax_f32(df, mask)


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("shape", [(16, 16), (272, 336), (1040, 3072)])
def test_quantize_with_given_amax_matches_oracle(shape, rounding):
    rows, cols = shape
    bits = inputs.normal(rows, cols, seed=rows + cols, outlier_channels=2)
    mask = 0x3C5A
    amax = torch.tensor([oracle.amax(bits, oracle.ROWWISE), oracle.amax(bits, oracle.COLWISE, True, mask)],
                        dtype=torch.float32, device="cuda")
    row, col = ops.quantize_row_col_rht_amax(helpers.to_device_bf16(bits), mask, amax, sr=rounding == 1, seed=11,
                                             stream_row=1, stream_col=2)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK
    for op, ref in ((row, oracle.quantize(bits, oracle.ROWWISE, rounding=rounding, seed=11, stream_id=1)),
                    (col, oracle.quantize(bits, oracle.COLWISE, rounding=rounding, use_rht=True, sign_mask=mask,
                                          seed=11, stream_id=2))):
        codes, scales, am, sg, _ = helpers.operand_to_host(op)
        assert am == ref["amax"] and sg == ref["s_g"]
        assert np.array_equal(codes, ref["codes"]) and np.array_equal(scales, ref["scales"])


def test_fused_chain_equals_unfused_chain():
    """GEMM with fused amax -> amax-taking quantization of its output equals
    the plain GEMM -> nvfp4_quantize_row_col_rht, bit for bit."""
    rng = np.random.default_rng(7)
    M, N, K = 512, 1024, 768
    a, b = _upload(_random_operand_host(rng, M, K), M, K), _upload(_random_operand_host(rng, N, K), N, K)
    mask = 0x9E37
    d, amax = ops.gemm_amax(a, b, mask)
    r1, c1 = ops.quantize_row_col_rht_amax(d, mask, amax, sr=True, seed=5, stream_row=3, stream_col=4)
    r2, c2 = ops.quantize_row_col_rht(ops.gemm(a, b), mask, sr=True, seed=5, stream_row=3, stream_col=4)
    torch.cuda.synchronize()
    for x, y in ((r1, r2), (c1, c2)):
        hx, hy = helpers.operand_to_host(x), helpers.operand_to_host(y)
        assert hx[2] == hy[2] and hx[3] == hy[3]
        assert np.array_equal(hx[0], hy[0]) and np.array_equal(hx[1], hy[1])

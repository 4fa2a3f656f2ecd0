"""GPU parity of nvfp4_dequantize: x^ = e2m1 * s_b * s_g rounded once to the
output type, bit-exact with the oracle's binary64 decode."""
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


@pytest.mark.parametrize("rows,cols,two_d", [(64, 256, False), (272, 336, False), (96, 128, True)])
def test_dequantize_matches_oracle(rows, cols, two_d):
    bits = inputs.student_t(rows, cols, seed=rows + cols)
    row, _ = ops.quantize(helpers.to_device_bf16(bits), two_d=two_d)
    y32 = ops.dequantize(row, torch.float32).cpu().numpy()
    y16 = ops.dequantize(row, torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.quantize(bits, scaling=1 if two_d else 0)
    deq = oracle.dequantize(ref["codes"], ref["scales"], ref["s_g"])
    assert np.array_equal(y32, deq.astype(np.float32))
    want16 = np.array([oracle.round_bf16(v) for v in deq.ravel()], np.uint16).reshape(deq.shape)
    assert np.array_equal(y16, want16)


def test_dequantize_all_codes_and_scales():
    """Every E2M1 code against every finite E4M3 scale, s_g = 1/3."""
    K = 16 * 127
    codes = np.tile(np.arange(16, dtype=np.uint8), (1, K // 16))[0]
    packed = (codes[0::2] | (codes[1::2] << 4)).reshape(1, K // 2)
    scales = np.arange(127, dtype=np.uint8).reshape(1, 127)
    op = ops.alloc_operand(1, K)
    host_codes = np.zeros((1, op.ld_codes), np.uint8)
    host_codes[:, : K // 2] = packed
    tiled = np.zeros(op.scales.numel(), np.uint8)
    tiled[helpers.scale_index_map(1, K)] = scales
    op.codes.copy_(torch.from_numpy(host_codes))
    op.scales.copy_(torch.from_numpy(tiled))
    op.global_scale.fill_(float(np.float32(1 / 3)))
    y = ops.dequantize(op, torch.float32).cpu().numpy()
    deq = oracle.dequantize(packed, scales, np.float32(1 / 3))
    assert np.array_equal(y, deq.astype(np.float32))

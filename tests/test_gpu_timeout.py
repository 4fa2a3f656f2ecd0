"""The GEMM's bounded waits on a real GPU, without a fault: the test support
entry point (include/nvfp4_testing.h) makes the next GEMM launch leave out
one barrier arrival and give up on its waits after a short limit.  The launch
must end by itself, report NVFP4_ERR_TIMEOUT through nvfp4_device_error,
leave its output unwritten, and the next GEMM in the same process must be
correct."""
import time

import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, ops
from tests.test_gpu_gemm import _check, _random_operand_host, _upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


@pytest.mark.parametrize("fused_amax", [False, True])
def test_gemm_wait_runs_out_and_the_next_call_is_correct(fused_amax):
    rng = np.random.default_rng(99)
    M, N, K = 256, 256, 512          # one 256 x 256 tile: one CTA pair
    a_h, b_h = _random_operand_host(rng, M, K), _random_operand_host(rng, N, K)
    a, b = _upload(a_h, M, K), _upload(b_h, N, K)
    y_ref, abs_sum = oracle.gemm_f64(a_h, b_h)
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK

    capi.check(capi.nvfp4_testing_arm_gemm_timeout(20000), "arm")     # 20 ms per wait
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    if fused_amax:
        ops.gemm_amax(a, b, 0x1234, out=y)
    else:
        ops.gemm(a, b, out=y)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert ops.device_error() == capi.NVFP4_ERR_TIMEOUT
    assert ops.device_error() == capi.NVFP4_OK       # read and cleared
    assert elapsed < 1.5, elapsed                     # a few 20 ms limits, not the 2 s default
    assert torch.all(y == 7.0), "a launch that timed out must not write its output"

    # the arm was consumed: the next calls run normally and are correct
    for dt in (torch.float32, torch.bfloat16):
        y2 = ops.gemm(a, b, out_dtype=dt)
        torch.cuda.synchronize()
        assert ops.device_error() == capi.NVFP4_OK
        _check(y2.float().cpu().numpy(), y_ref, abs_sum, dt == torch.bfloat16)

"""nvfp4_quantize_noalloc: the quantizer for callers that cannot provide device
scratch (for example a plugin whose host runtime owns all device memory, or
code that must not allocate once running).  It must produce exactly what
nvfp4_quantize produces with a caller-provided workspace, call after call,
although every call reuses the same library-held scratch.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, inputs, ops
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def _quantize_pair(x, scaling, rounding, seed, stream_id):
    """The same call through nvfp4_quantize (workspace) and nvfp4_quantize_noalloc."""
    rows, cols = x.shape
    st = ops.stream_handle()
    ws = ops.Workspace()
    outs = []
    for noalloc in (False, True):
        row = ops.alloc_operand(rows, cols)
        col = ops.alloc_operand(cols, rows)
        orient = capi.NVFP4_ROWWISE | capi.NVFP4_COLWISE
        if noalloc:
            status = capi.nvfp4_quantize_noalloc(x.data_ptr(), rows, cols, x.stride(0), scaling, rounding, seed,
                                                 stream_id, orient, row.struct(), col.struct(), st)
        else:
            status = capi.nvfp4_quantize(x.data_ptr(), rows, cols, x.stride(0), scaling, rounding, seed, stream_id,
                                         orient, row.struct(), col.struct(), ws.ptr, ws.nbytes, st)
        assert status == capi.NVFP4_OK, capi.status_string(status)
        outs.append((row, col))
    torch.cuda.synchronize()
    return outs


def _same(a, b):
    ca, sa, ama, sga, ta = helpers.operand_to_host(a)
    cb, sb, amb, sgb, tb = helpers.operand_to_host(b)
    assert ama == amb and sga == sgb
    assert np.array_equal(ca, cb) and np.array_equal(ta, tb)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    first = helpers.to_device_bf16(inputs.normal(384, 512, seed=71, outlier_channels=2))
    second = helpers.to_device_bf16(inputs.student_t(256, 768, seed=72))
    calls = [(first, capi.NVFP4_SCALE_1X16, capi.NVFP4_ROUND_RNE, 0, 0),
             (second, capi.NVFP4_SCALE_1X16, capi.NVFP4_ROUND_SR, 99, 3)]
    for x, scaling, rounding, seed, stream_id in calls:
        (ref_row, ref_col), (na_row, na_col) = _quantize_pair(x, scaling, rounding, seed, stream_id)
        _same(ref_row, na_row)
        _same(ref_col, na_col)

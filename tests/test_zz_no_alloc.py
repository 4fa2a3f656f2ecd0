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


BOTH = capi.NVFP4_ROWWISE | capi.NVFP4_COLWISE


def _quantize_pair(x, scaling, rounding, seed, stream_id, orient=BOTH):
    """The same call through nvfp4_quantize (workspace) and nvfp4_quantize_noalloc."""
    rows, cols = x.shape
    st = ops.stream_handle()
    ws = ops.Workspace()
    outs = []
    for noalloc in (False, True):
        row = ops.alloc_operand(rows, cols) if orient & capi.NVFP4_ROWWISE else None
        col = ops.alloc_operand(cols, rows) if orient & capi.NVFP4_COLWISE else None
        rs = row.struct() if row is not None else None
        cs = col.struct() if col is not None else None
        if noalloc:
            status = capi.nvfp4_quantize_noalloc(x.data_ptr(), rows, cols, x.stride(0), scaling, rounding, seed,
                                                 stream_id, orient, rs, cs, st)
        else:
            status = capi.nvfp4_quantize(x.data_ptr(), rows, cols, x.stride(0), scaling, rounding, seed, stream_id,
                                         orient, rs, cs, ws.ptr, ws.nbytes, st)
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


def test_noalloc_matches_in_every_scaling_mode_and_after_a_larger_call():
    """16x16 and 4/6 scaling through the shared scratch, then a row-wise-only
    call on a small tensor right after a large one: the small call's amax
    pass writes fewer partials than the large call left in the scratch, and
    the result must still equal the workspace entry point's (the leftovers
    are not read)."""
    big = helpers.to_device_bf16(inputs.normal(4096, 3072, seed=73, outlier_channels=3))
    small = helpers.to_device_bf16(inputs.student_t(64, 128, seed=74, scale=1e-6))
    calls = [(big, capi.NVFP4_SCALE_16X16, capi.NVFP4_ROUND_RNE, 0, 0, BOTH),
             (big, capi.NVFP4_SCALE_1X16_46, capi.NVFP4_ROUND_SR, 5, 1, BOTH),
             (big, capi.NVFP4_SCALE_1X16, capi.NVFP4_ROUND_RNE, 0, 0, BOTH),
             (small, capi.NVFP4_SCALE_1X16, capi.NVFP4_ROUND_RNE, 0, 0, capi.NVFP4_ROWWISE),
             (small, capi.NVFP4_SCALE_1X16_46, capi.NVFP4_ROUND_RNE, 0, 0, capi.NVFP4_COLWISE)]
    for x, scaling, rounding, seed, stream_id, orient in calls:
        (ref_row, ref_col), (na_row, na_col) = _quantize_pair(x, scaling, rounding, seed, stream_id, orient)
        for a, b in ((ref_row, na_row), (ref_col, na_col)):
            if a is not None:
                _same(a, b)

"""The library under CUDA-graph capture and under concurrent host threads:
the results equal those of plain eager calls."""
import threading

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


def _host(op):
    codes, scales, amax, sg, _ = helpers.operand_to_host(op)
    return codes.copy(), scales.copy(), float(amax), float(sg)


def _same(a, b):
    assert a[2] == b[2] and a[3] == b[3]
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_graph_replay_equals_eager_on_new_inputs():
    """A captured chain (pair quantization of X with SR, 16x16 of W, GEMM with
    the fused amax, amax-given pair quantization of its output, Wgrad-shaped
    GEMM) replayed on inputs copied into the captured buffers gives what the
    eager calls give on the same inputs."""
    M, K, N = 512, 768, 1024
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    mask = 0x6A5C
    xr, xc = ops.alloc_operand(M, K), ops.alloc_operand(K, M)
    wr, wc = ops.alloc_operand(N, K), ops.alloc_operand(K, N)
    h = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    amax = torch.zeros(2, dtype=torch.float32, device="cuda")
    hr, hc = ops.alloc_operand(M, N), ops.alloc_operand(N, M)
    g_out = torch.empty((K, N), dtype=torch.float32, device="cuda")
    ws = ops.Workspace()
    stream = torch.cuda.Stream()

    def chain():
        ops.quantize_row_col_rht(x, mask, sr=True, seed=7, stream_row=1, stream_col=2, out_row=xr, out_col=xc,
                                 workspace=ws)
        ops.quantize(w, two_d=True, rowwise=True, colwise=True, out_row=wr, out_col=wc, workspace=ws)
        ops.gemm_amax(xr, wr, mask, out=h, amax=amax)
        ops.quantize_row_col_rht_amax(h, mask, amax, out_row=hr, out_col=hc)
        ops.gemm(xc, hc, out=g_out)     # [K][N] from two col-wise operands (K-major over the M tokens)

    def snapshot():
        torch.cuda.synchronize()
        return [_host(op) for op in (xr, xc, wr, wc, hr, hc)] + [h.cpu().clone(), g_out.cpu().clone(),
                                                                 amax.cpu().clone()]

    def load(seed):
        x.copy_(helpers.to_device_bf16(inputs.normal(M, K, seed, outlier_channels=2)))
        w.copy_(helpers.to_device_bf16(inputs.normal(N, K, seed + 1, std=0.02)))

    with torch.cuda.stream(stream):
        load(1)
        chain()                      # eager warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain()
    for seed in (11, 12):
        with torch.cuda.stream(stream):
            load(seed)
            chain()
        eager = snapshot()
        with torch.cuda.stream(stream):
            x.zero_()
            w.zero_()
            load(seed)
            g.replay()
        replay = snapshot()
        assert ops.device_error() == capi.NVFP4_OK
        for e, r in zip(eager[:6], replay[:6]):
            _same(e, r)
        for e, r in zip(eager[6:], replay[6:]):
            assert torch.equal(e, r)


def test_concurrent_host_threads_give_the_single_thread_results():
    """Four threads, each with its own stream and buffers, run quantize and
    GEMM calls at once; every result equals the same call made alone."""
    shapes = [(256, 512, 384), (272, 336, 640), (128, 1024, 256), (400, 192, 512)]

    def job(i, results, stream):
        M, K, N = shapes[i]
        xb = inputs.student_t(M, K, 30 + i)
        wb = inputs.normal(N, K, 40 + i, std=0.02)
        with torch.cuda.stream(stream):
            ws = ops.Workspace()    # one quantizer workspace per stream
            for _ in range(10):
                x = helpers.to_device_bf16(xb)
                w = helpers.to_device_bf16(wb)
                xr, xc = ops.quantize_row_col_rht(x, 0x1357 + i, sr=True, seed=i, stream_row=1, stream_col=2,
                                                  workspace=ws, stream=stream)
                wr, _ = ops.quantize(w, workspace=ws, stream=stream)
                y = ops.gemm(xr, wr, stream=stream)
            stream.synchronize()
        results[i] = (_host(xr), _host(xc), _host(wr), y.cpu())

    alone = {}
    for i in range(len(shapes)):
        job(i, alone, torch.cuda.Stream())
    together = {}
    threads = [threading.Thread(target=job, args=(i, together, torch.cuda.Stream())) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert ops.device_error() == capi.NVFP4_OK
    for i in range(len(shapes)):
        for a, b in zip(alone[i][:3], together[i][:3]):
            _same(a, b)
        assert torch.equal(alone[i][3], together[i][3])

"""The benchmarked FFN layer step at 16384 tokens, end to end against the
oracle: the step object bench.py times (the same entry points, launch order
and buffers), run once on the GPU, then every quantized operand and every
GEMM output checked on sampled rows.

The step's dataflow ("Full-Stack FP4", Sec. 2: Fprop, Dgrad and Wgrad of a
linear layer; Appendix 9: quantization fused with the producing operation):
H is written by Fprop-up and dY_up by Dgrad-down, whose epilogues also take
the two tensor amaxes that the pair quantization of H and dY_up then uses
without an amax pass.  The oracle follows the same chain: the inputs X,
W_up, W_down and dY_down come from the seeded generators, and H and dY_up,
after their own check against the oracle's GEMM, are the tensors the GPU
wrote (a GEMM output rounded to BF16 is not unique across summation orders,
so the quantizations downstream are checked on the tensor the step actually
produced).
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from fp4_gemm_nvfp4_gb300 import build as libbuild
from fp4_gemm_nvfp4_gb300 import capi, ops
from tests import helpers
from tests.test_gpu_gemm import _check, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    libbuild.build()
    capi.load()


def _to_host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_kw(name, orient, mask, seed):
    kw = dict(next(k for n, _, k in bench.QUANTS if n == name))
    out = bench._oracle_kw(kw, mask, seed, orient)
    out["orientation"] = oracle.ROWWISE if orient == "row" else oracle.COLWISE
    return out


def test_layer_step_16384_tokens_against_the_oracle_chain():
    assert bench.FUSE_AMAX and bench.TOKENS == 16384
    host, mask = bench.host_inputs()
    seed = 4
    dev = {k: helpers.to_device_bf16(v) for k, v in host.items()}
    step = bench.Step(dev, mask, seed)
    step.run()
    torch.cuda.synchronize()
    assert ops.device_error() == capi.NVFP4_OK

    # the oracle's inputs: generated tensors, and the two the step produced
    src_bits = dict(host)
    for src, gname in bench.PRODUCED.items():
        src_bits[src] = _to_host_bits(step.out[gname])
    src_of = {n: s for n, s, _ in bench.QUANTS}

    # 1. the two produced tensors' amaxes, taken in their GEMM's epilogue
    for src, gname in bench.PRODUCED.items():
        got = step.amax[gname].cpu().numpy()
        assert got[0] == oracle.amax(src_bits[src], oracle.ROWWISE), gname
        assert got[1] == oracle.amax(src_bits[src], oracle.COLWISE, True, mask), gname

    # 2. every quantized operand, sampled logical rows of both orientations
    for name, src, _ in bench.QUANTS:
        for orient, op in zip(("row", "col"), step.q[name]):
            if op is None:
                continue
            kw = _oracle_kw(name, orient, mask, seed)
            rows = sample_rows(op.rows, n=16, seed=len(name) + op.rows)
            ref = oracle_rows(src_bits[src], kw, rows)
            codes, scales, _, sg, _ = helpers.operand_to_host(op)
            assert sg == ref["s_g"], (name, orient)
            assert np.array_equal(codes[rows], ref["codes"]), (name, orient)
            assert np.array_equal(scales[rows], ref["scales"]), (name, orient)

    # 3. every GEMM output on sampled rows against the oracle's FP64 GEMM of
    # the oracle-quantized operands
    for gname, (an, ao), (bn, bo) in bench.GEMMS:
        a_op = step.operand(an, ao)
        rows = sample_rows(a_op.rows, n=12, seed=len(gname))
        qa = oracle_rows(src_bits[src_of[an]], _oracle_kw(an, ao, mask, seed), rows)
        bkw = _oracle_kw(bn, bo, mask, seed)
        qb = oracle.quantize(src_bits[src_of[bn]], bkw.pop("orientation"), **bkw)
        y_ref, abs_sum = oracle.gemm_f64(qa, qb)
        y = step.out[gname][torch.from_numpy(rows).cuda()].float().cpu().numpy()
        _check(y, y_ref, abs_sum, True)

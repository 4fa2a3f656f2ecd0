"""bench.py's accounting of the layer step (CPU only): the launches one step
makes, the GEMM FLOPs and the quantizers' algorithmic bytes that the bench
line's roofline fractions divide by.  The expected launch counts are those
of the library's launchers (one amax pass, one per orientation with the RHT,
and one encode pass emitting every requested orientation; no amax pass when
the producing GEMM took the amax)."""
import pytest

import bench


@pytest.fixture(autouse=True)
def tokens_16384():
    old = bench.TOKENS
    bench.set_tokens(16384)
    yield
    bench.set_tokens(old)


def _step_calls():
    calls = {}
    for name, src, kw in bench.QUANTS:
        kw = dict(kw)
        if bench.produced(src):
            kw["amax_given"] = True
        calls[name] = (src, kw)
    return calls


def _operand_shape(calls, name, orient):
    rows, cols = bench.SHAPES[calls[name][0]]
    return (rows, cols) if orient == "row" else (cols, rows)


def test_quantize_call_launches():
    assert bench.quant_launches(dict(pair=True, rht_mask=1)) == 2
    assert bench.quant_launches(dict(pair=True, rht_mask=1, amax_given=True)) == 1
    assert bench.quant_launches(dict(rowwise=True, colwise=True, two_d=True)) == 2
    assert bench.quant_launches(dict(rowwise=True)) == 2
    assert bench.quant_launches(dict(rowwise=True, colwise=True)) == 2
    assert bench.quant_launches(dict(rowwise=True, rht_mask=1)) == 2
    assert bench.quant_launches(dict(rowwise=True, colwise=True, rht_mask=1)) == 3


def test_quantize_call_bytes_per_element():
    n = 1 << 20
    # amax pass 2 B, encode pass 2 B, 0.5625 B written per orientation
    assert bench.quant_bytes(1024, 1024, dict(rowwise=True)) == n * 4.5625
    assert bench.quant_bytes(1024, 1024, dict(rowwise=True, colwise=True, two_d=True)) == n * 5.125
    assert bench.quant_bytes(1024, 1024, dict(pair=True, rht_mask=1)) == n * 5.125
    assert bench.quant_bytes(1024, 1024, dict(pair=True, rht_mask=1, amax_given=True)) == n * 3.125
    # with the RHT each orientation has its own amax pass
    assert bench.quant_bytes(1024, 1024, dict(rowwise=True, colwise=True, rht_mask=1)) == n * 7.125


def test_step_has_sixteen_launches():
    calls = _step_calls()
    launches = sum(bench.quant_launches(kw) for _, kw in calls.values()) + len(bench.GEMMS)
    assert launches == 16
    assert [k for k, _ in bench.ORDER].count("g") == 6 and [k for k, _ in bench.ORDER].count("q") == 6


def test_step_gemms_share_their_reduction_dim_and_total_5566_gflop():
    calls = _step_calls()
    flops = 0
    for _, (an, ao), (bn, bo) in bench.GEMMS:
        m, k = _operand_shape(calls, an, ao)
        n, kb = _operand_shape(calls, bn, bo)
        assert k == kb
        assert k % 16 == 0
        flops += 2 * m * n * k
    # six GEMMs of 16384 x 9216 x 3072 in some order of their dimensions
    assert flops == 6 * 2 * 16384 * 9216 * 3072
    assert round(flops / 1e9, 1) == 5566.3


def test_step_quantize_bytes():
    calls = _step_calls()
    total = sum(bench.quant_bytes(*bench.SHAPES[src], kw) for src, kw in calls.values())
    x, h, w = 16384 * 3072, 16384 * 9216, 9216 * 3072
    # X and dY_down: amax + pair; H and dY_up: pair with the amax given; two 16x16 weights
    assert total == 2 * x * 5.125 + 2 * h * 3.125 + 2 * w * 5.125
    assert int(total) == 1749811200

"""Pins for the oracle's NVFP4 Newton-Schulz iteration ("Full-Stack FP4",
Sec. 3.4, the quantized NS iteration of the Root optimizer) and the GEMM with
a C term it is built from.

Each check compares the oracle with something other than itself: the
iteration's polynomial p(s) = a s + b s^3 + c s^5 in closed form on inputs
whose quantization is exact, the b = c = 0 special case, the unquantized
iteration in float64, and the fixed point of the cubic Newton-Schulz map.
No expected value comes from the CUDA library.
"""
import numpy as np
import pytest

import oracle

MUON = (3.4445, -4.7750, 2.0315)   # the standard Muon coefficients the page compares against


def _f32(v):
    return float(np.float32(v))


def _scaled_partial_identity(m, n, s_blocks):
    """X = [diag(s) | 0] with s constant on each 16-row block."""
    x = np.zeros((m, n))
    s = np.repeat(np.asarray(s_blocks, np.float64), 16)
    x[np.arange(m), np.arange(m)] = s
    return oracle.round_bf16_array(x), s


@pytest.mark.parametrize("coef", [(1.5, -0.5, 0.0), (2.0, -1.0, -2.0), (0.75, 0.5, 1.0)])
def test_ns_closed_form_on_scaled_partial_identity(coef):
    # X = [diag(s) | 0], s = 1 on rows 0-15 and 1/2 on rows 16-31.  Each
    # quantized tensor then has one magnitude per 16-block (RHT rows are
    # +-value/4) and block maxima a power of two apart (c = 0 or c = 2b makes
    # B's two diagonal values differ by 1/4 or 1/8), so every block scale is
    # exact and the step is the NS polynomial: A = diag(s^2), B = diag(b s^2
    # + c s^4), X_next = diag(a s + b s^3 + c s^5), up to the decode scales'
    # rounding (2^-24) and one bf16 rounding of X_next.
    a, b, c = (_f32(v) for v in coef)
    x_bits, s = _scaled_partial_identity(32, 64, [1.0, 0.5])
    r = oracle.newton_schulz_step(x_bits, *coef, sign_mask=0x6A3C)
    A = oracle.bf16_to_f64(r["A"])
    B = oracle.bf16_to_f64(r["B"])
    X = oracle.bf16_to_f64(r["X"])
    assert np.array_equal(A, np.diag(s ** 2))
    assert np.array_equal(B, np.diag(b * s ** 2 + c * s ** 4))
    p = a * s + b * s ** 3 + c * s ** 5
    assert np.all(np.abs(np.diag(X[:, :32]) - p) <= 2.0 ** -9 * np.abs(p) + 1e-6)
    assert np.count_nonzero(X[:, 32:]) == 0
    assert np.count_nonzero(X[:, :32] - np.diag(np.diag(X[:, :32]))) == 0


def test_ns_muon_coefficients_on_scaled_partial_identity():
    # With the Muon coefficients B's two diagonal values are not a power of
    # two apart: the smaller block's E4M3 scale (and the 4/6 choice) carries
    # up to 1/16 relative error into the c-and-b term, the rest is as above.
    a, b, c = (_f32(v) for v in MUON)
    x_bits, s = _scaled_partial_identity(32, 64, [1.0, 0.5])
    r = oracle.newton_schulz_step(x_bits, *MUON, sign_mask=0x6A3C)
    B = np.diag(oracle.bf16_to_f64(r["B"]))
    X = np.diag(oracle.bf16_to_f64(r["X"])[:, :32])
    b_exact = b * s ** 2 + c * s ** 4
    assert np.all(np.abs(B - b_exact) <= 2.0 ** -8 * np.abs(b_exact))
    tol = 2.0 ** -4 * np.abs(B * s) + 2.0 ** -8 * (np.abs(a * s) + np.abs(B * s))
    assert np.all(np.abs(X - (a * s + B * s)) <= tol)
    # the block holding the tensor amax is exact
    assert np.all(np.abs(X[:16] - (a + B[:16])) <= 2.0 ** -8 * np.abs(a + B[:16]))


def test_ns_without_the_cubic_terms_is_a_scaling():
    # b = c = 0: B = 0 quantizes to zero codes, so X_next = RN_bf16(a X) exactly
    rng = np.random.default_rng(11)
    x_bits = oracle.round_bf16_array(rng.standard_normal((48, 96)) * 0.05)
    r = oracle.newton_schulz_step(x_bits, 1.75, 0.0, 0.0, sign_mask=0x0F0F)
    assert np.count_nonzero(oracle.bf16_to_f64(r["B"])) == 0
    assert np.array_equal(r["X"], oracle.round_bf16_array(_f32(1.75) * oracle.bf16_to_f64(x_bits)))


@pytest.mark.parametrize("m,n", [(64, 128), (96, 288)])
def test_ns_step_close_to_unquantized_polynomial(m, n):
    # Muon-style input G / ||G||_F: one quantized step lands within 2 % of
    # a X + b (X X^T) X + c (X X^T)^2 X computed in float64 (measured 0.2-0.5 %)
    rng = np.random.default_rng(m + n)
    g = rng.standard_normal((m, n))
    x_bits = oracle.round_bf16_array(g / np.linalg.norm(g))
    x = oracle.bf16_to_f64(x_bits)
    a, b, c = (_f32(v) for v in MUON)
    gram = x @ x.T
    p = a * x + b * gram @ x + c * gram @ gram @ x
    r = oracle.newton_schulz_step(x_bits, *MUON, sign_mask=0xB5C3)
    err = np.linalg.norm(oracle.bf16_to_f64(r["X"]) - p) / np.linalg.norm(p)
    assert err < 0.02, err
    # and A is X X^T up to FP4 noise
    assert np.linalg.norm(oracle.bf16_to_f64(r["A"]) - gram) / np.linalg.norm(gram) < 0.15


def test_cubic_ns_iteration_settles_near_orthogonal():
    # (a, b, c) = (1.5, -0.5, 0) has a super-attracting fixed point at s = 1
    # (p'(1) = 0): the quantized iteration keeps every singular value near 1
    # (measured 0.86 .. 1.13 after 12 steps; exact arithmetic reaches 1)
    rng = np.random.default_rng(3)
    g = rng.standard_normal((64, 128))
    xk = oracle.round_bf16_array(0.9 * g / np.linalg.norm(g, 2))
    for k in range(12):
        xk = oracle.newton_schulz_step(xk, 1.5, -0.5, 0.0, sign_mask=0x1357 + 97 * k)["X"]
    sv = np.linalg.svd(oracle.bf16_to_f64(xk), compute_uv=False)
    assert 0.8 < sv.min() and sv.max() < 1.2, (sv.min(), sv.max())


def test_gemm_axpby_reduces_to_its_terms():
    rng = np.random.default_rng(5)
    xa = oracle.round_bf16_array(rng.standard_normal((32, 64)))
    xb = oracle.round_bf16_array(rng.standard_normal((48, 64)))
    cb = oracle.round_bf16_array(rng.standard_normal((32, 48)))
    qa, qb = oracle.quantize(xa), oracle.quantize(xb)
    y0, ab0 = oracle.gemm_f64(qa, qb)
    y, ab = oracle.gemm_axpby_f64(qa, qb, 0.5, cb, 0.0)
    assert np.array_equal(y, 0.5 * y0) and np.array_equal(ab, 0.5 * ab0)
    y, _ = oracle.gemm_axpby_f64(qa, qb, 0.0, cb, -2.0)
    assert np.array_equal(y, -2.0 * oracle.bf16_to_f64(cb))

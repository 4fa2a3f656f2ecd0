"""Pins for the CPU oracle: facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print (tests/golden), a library routine run independently (torch's
float8/bfloat16 casts, cuRAND's host Philox generator), a closed form, an
invariant, or exact brute force.  No expected value here comes from the CUDA
library.
"""
import ctypes
import ctypes.util
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fp4_gemm_nvfp4_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _grid():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_grid.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                code, e, m, val = line.split()
                rows.append((int(code), int(e), int(m), float(val)))
    return rows


def _bins():
    bins, ties = [], []
    with open(os.path.join(GOLDEN, "e2m1_bins.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "tie":
                ties.append((float(parts[1]), float(parts[2])))
            else:
                lo, hi, val, step = parts
                bins.append((float(lo), float(hi), float(val), None if step == "-" else float(step)))
    return bins, ties


GRID = np.array([g[3] for g in _grid()])


def _unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def _e2m1_values(codes4):
    mag = GRID[codes4 & 7]
    return np.where(codes4 & 8, -mag, mag)


def _torch_e4m3_values(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------- E2M1 ----
def test_e2m1_grid_matches_page_enumeration():
    for code, e, m, val in _grid():
        # the page's definition: bias 1, exponent 0 is subnormal (0.m * 2^0)
        by_bits = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert by_bits == val
        assert oracle.e2m1_value(code) == val
        assert oracle.e2m1_value(code | 8) == -val


def test_e2m1_rne_bins_and_ties():
    bins, ties = _bins()
    eps = 1e-6
    for lo, hi, val, _ in bins:
        inside = [lo + eps, (lo + min(hi, 8.0)) / 2, min(hi, 100.0) - eps]
        for v in inside:
            q = oracle.e2m1_value(oracle.e2m1_rne(v))
            assert q == val, (v, q, val)
            assert oracle.e2m1_value(oracle.e2m1_rne(-v)) == -val
    for tie, expect in ties:
        assert oracle.e2m1_value(oracle.e2m1_rne(tie)) == expect, tie
        assert oracle.e2m1_value(oracle.e2m1_rne(-tie)) == -expect, tie
    for big in (6.0, 7.0, 1e9, 3.4e38):
        assert oracle.e2m1_rne(big) == 7 and oracle.e2m1_rne(-big) == 15


def test_e2m1_rne_error_within_half_step():
    """Appendix 7 of "Full-Stack FP4": RTN error |delta| <= step_k / 2."""
    rng = np.random.default_rng(1)
    v = np.concatenate([np.arange(0, 6.0, 1 / 4096, dtype=np.float32),
                        rng.uniform(0, 6, 200000).astype(np.float32)])
    q = _e2m1_values(oracle.e2m1_rne_array(v))
    bins, _ = _bins()
    for lo_grid, hi_grid in zip(GRID[:-1], GRID[1:]):
        sel = (v >= lo_grid) & (v < hi_grid)
        step = hi_grid - lo_grid
        assert np.all(np.abs(q[sel] - v[sel]) <= step / 2)
        assert np.all((q[sel] == lo_grid) | (q[sel] == hi_grid))
    # and the result is the nearest grid point
    nearest = np.min(np.abs(v[:, None] - GRID[None, :]), axis=1)
    assert np.array_equal(np.abs(q - v), nearest)


def test_e2m1_sign_bit_follows_input():
    assert oracle.e2m1_rne(-0.1) == 8       # negative value rounding to zero keeps its sign
    assert oracle.e2m1_rne(-0.0) == 8
    assert oracle.e2m1_rne(0.0) == 0
    assert oracle.e2m1_sr(-0.0, 0) == 8
    assert oracle.e2m1_sr(-0.2, 0xFFFFFFFF) == 8


def test_e2m1_sr_grid_points_never_move():
    words = [0, 1, 0xFF, 0x100, 0x7FFF, 0xFFFF]
    for code in range(8):
        for w in words:
            assert oracle.e2m1_sr(float(GRID[code]), w) == code
            assert oracle.e2m1_sr(-float(GRID[code]), w) == code | 8


def test_e2m1_sr_probability_threshold():
    """P(up) = d / step realised with 16 random bits: up iff u < ceil(frac * 2^16)."""
    for v in (0.1, 0.3, 0.74, 1.2, 1.6, 1.9, 2.2, 2.9, 3.3, 4.5, 5.9, 1e-7):
        k = int(np.searchsorted(GRID, v, side="right") - 1)
        frac = Fraction(float(np.float32(v))) - Fraction(float(GRID[k]))
        frac /= Fraction(float(GRID[k + 1] - GRID[k]))
        thr = math.ceil(frac * 2 ** 16)
        assert oracle.e2m1_sr(v, thr - 1) == k + 1
        assert oracle.e2m1_sr(v, thr) == k
        assert oracle.e2m1_sr(v, 0xFFFF) == k


@pytest.mark.parametrize("v", [0.1, 0.3, 0.74, 1.2, 1.9, 2.2, 2.9, 3.3, 4.5, 5.9])
def test_e2m1_sr_unbiased_with_page_variance(v):
    """Appendix 7: SR is unbiased with variance d (step - d); 10^6 draws, 4 sigma."""
    n = 1_000_000
    rng = np.random.default_rng(int(v * 1000))
    words = rng.integers(0, 2 ** 16, n, dtype=np.uint64).astype(np.uint32)
    q = _e2m1_values(oracle.e2m1_sr_array(np.full(n, v, np.float32), words))
    k = int(np.searchsorted(GRID, v, side="right") - 1)
    step = GRID[k + 1] - GRID[k]
    d = float(np.float32(v)) - GRID[k]
    var = d * (step - d)
    err = q - float(np.float32(v))
    assert abs(err.mean()) <= 4 * math.sqrt(var / n)
    assert abs(err.var() / var - 1) < 0.01


def test_rtn_mse_uniform_in_bin():
    """Appendix 7: input-averaged RTN MSE is step^2 / 12 inside a bin."""
    rng = np.random.default_rng(7)
    for lo, hi in zip(GRID[:-1], GRID[1:]):
        v = rng.uniform(lo, hi, 200000).astype(np.float32)
        q = _e2m1_values(oracle.e2m1_rne_array(v))
        mse = np.mean((q - v.astype(np.float64)) ** 2)
        assert abs(mse / ((hi - lo) ** 2 / 12) - 1) < 0.02


# ---------------------------------------------------------------- E4M3 ----
def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = _torch_e4m3_values(codes)
    ours = np.array([oracle.e4m3_value(c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert oracle.e4m3_value(0x7E) == 448.0


def test_e4m3_encode_matches_torch_rne():
    vals = _torch_e4m3_values(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(3)
    rand = np.concatenate([rng.uniform(0, 464, 100000),
                           np.exp(rng.uniform(np.log(1e-6), np.log(463.9), 100000))])
    x = np.concatenate([vals, mids, rand]).astype(np.float32)
    x = x[x < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = oracle.e4m3_rne_satfinite_array(x)
    assert np.array_equal(ours, ref)
    # satfinite: beyond the largest finite value everything lands on 448
    big = np.array([448.0, 449.0, 464.0, 500.0, 1e6, 3.4e38], np.float32)
    assert np.all(oracle.e4m3_rne_satfinite_array(big) == 0x7E)


# -------------------------------------------------------------- Philox ----
def _curand():
    for name in ("libcurand.so", "libcurand.so.10"):
        for d in ("/usr/local/cuda/lib64", ""):
            path = os.path.join(d, name) if d else name
            try:
                return ctypes.CDLL(path)
            except OSError:
                continue
    found = ctypes.util.find_library("curand")
    return ctypes.CDLL(found) if found else None


def _curand_philox_host(seed, n):
    lib = _curand()
    if lib is None:
        pytest.skip("cuRAND host library not available")
    gen = ctypes.c_void_p()
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(n, np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


@pytest.mark.parametrize("seed", [0, 1, 0x123456789ABCDEF0, 0xFFFFFFFFFFFFFFFF, 2 ** 32 + 7])
def test_philox_matches_curand_host_generator(seed):
    """cuRAND's host Philox4x32-10 emits block i from counter (0, 0, i, 0) under
    key (seed lo, seed hi); the oracle's round function must reproduce it."""
    n_blocks = 512
    ref = _curand_philox_host(seed, 4 * n_blocks).reshape(n_blocks, 4)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in list(range(16)) + [100, 255, 511]:
        ours = oracle.philox4x32_10([0, 0, i, 0], key)
        assert np.array_equal(ours, ref[i]), i
    # the SR bits of element idx < 8 in stream s are 16 bits of block s
    for s in (0, 3, 77):
        for idx in range(8):
            word = int(ref[s][idx // 2])
            assert oracle.sr_bits(seed, s, idx) == (word >> (16 * (idx % 2))) & 0xFFFF


def test_sr_bits_counter_layout():
    """g = idx >> 3 goes to counter words 0-1, the stream to words 2-3; element
    idx takes the low (even idx) or high (odd idx) half of word (idx >> 1) & 3."""
    seed, stream = 0xDEADBEEF12345678, 0x0000000A00000005
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for idx in (0, 5, 7, 1 << 33, (1 << 40) + 3):
        g = idx >> 3
        block = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, stream & 0xFFFFFFFF, stream >> 32], key)
        word = int(block[(idx >> 1) & 3])
        assert oracle.sr_bits(seed, stream, idx) == (word >> (16 * (idx & 1))) & 0xFFFF


# ----------------------------------------------------------------- RHT ----
def _sylvester(n):
    """The recursion on the "OptiTrain-FP4" page: H_1 = [1], H_2k = [[H, H], [H, -H]]."""
    h = np.array([[1]], dtype=np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _rht_matrix(mask):
    """4*U column by column from the oracle's butterfly applied to unit vectors."""
    cols = []
    for j in range(16):
        e = np.zeros(16, np.float32)
        e[j] = 1.0
        cols.append(oracle.rht16(e, mask) * 4)
    return np.stack(cols, axis=1).astype(np.float64)


@pytest.mark.parametrize("mask", [0, 0xFFFF, 0x5A3C, 0x0001, 0x8000])
def test_rht_matches_sylvester_times_signs(mask):
    H = _sylvester(16)
    D = np.diag([-1 if (mask >> i) & 1 else 1 for i in range(16)])
    assert np.array_equal(_rht_matrix(mask), (H @ D).astype(np.float64))


def test_rht_orthogonality():
    """H16 H16^T = 16 I exactly; U^T U = I ("Pretraining LLMs with NVFP4", B.4)."""
    M = _rht_matrix(0).astype(np.int64)
    assert set(np.unique(M)) == {-1, 1}
    assert np.array_equal(M @ M.T, 16 * np.eye(16, dtype=np.int64))
    U = _rht_matrix(0xB7E1) / 4
    assert np.array_equal(U.T @ U, np.eye(16))


def test_rht_spreads_a_spike():
    for j in range(16):
        e = np.zeros(16, np.float32)
        e[j] = 1.0
        assert np.all(np.abs(oracle.rht16(e, 0x1234)) == 0.25)


def test_rht_preserves_inner_products():
    """(UA)^T (UB) = A^T B: exact for small integers (the butterfly is exact)."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        a = rng.integers(-8, 9, 16).astype(np.float32)
        b = rng.integers(-8, 9, 16).astype(np.float32)
        mask = int(rng.integers(0, 1 << 16))
        ua = oracle.rht16(a, mask).astype(np.float64)
        ub = oracle.rht16(b, mask).astype(np.float64)
        assert ua @ ub == a.astype(np.float64) @ b.astype(np.float64)
    for _ in range(200):
        a = rng.standard_normal(16).astype(np.float32)
        b = rng.standard_normal(16).astype(np.float32)
        mask = int(rng.integers(0, 1 << 16))
        lhs = oracle.rht16(a, mask).astype(np.float64) @ oracle.rht16(b, mask).astype(np.float64)
        rhs = a.astype(np.float64) @ b.astype(np.float64)
        assert abs(lhs - rhs) <= 1e-6 * (np.abs(a) @ np.abs(b)) + 1e-12


# ------------------------------------------------------------ quantize ----
def _rand_bits(rows, cols, seed, scale=1.0, outliers=0):
    return inputs.normal(rows, cols, seed, scale, outliers)


def test_tensor_scale_puts_the_amax_block_on_448():
    """The tensor scale keeps every block scale inside E4M3 and the block that
    holds the tensor amax gets the largest scale, 448."""
    for seed in range(4):
        x = _rand_bits(64, 256, seed, outliers=3)
        q = oracle.quantize(x)
        xf = inputs.bf16_bits_to_f32(x)
        assert q["amax"] == np.abs(xf).max()
        r, c = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
        assert q["scales"][r, c // 16] == 0x7E
        assert q["scales"].max() <= 0x7E
        assert abs(float(q["s_enc"]) * float(q["s_g"]) - 1.0) < 1e-6


def test_zero_tensor():
    x = np.zeros((32, 64), np.uint16)
    q = oracle.quantize(x)
    assert q["amax"] == 0 and q["s_enc"] == 1 and q["s_g"] == 1
    assert not q["codes"].any() and not q["scales"].any()


def test_block_amax_lands_on_six_with_near_fp8_precision():
    """Block amax -> FP4 max 6 and the amax element kept to E4M3 precision
    ("Pretraining LLMs with NVFP4", Sec. 2: at least 1 of 16 at near-FP8)."""
    x = _rand_bits(128, 512, 11, outliers=4)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    q = oracle.quantize(x)
    codes = _unpack(q["codes"])
    deq = oracle.dequantize(q["codes"], q["scales"], q["s_g"])
    blocks = np.abs(xf).reshape(128, 32, 16)
    arg = blocks.argmax(axis=2)
    checked = 0
    for r in range(128):
        for b in range(32):
            if q["scales"][r, b] < 0x08:        # subnormal scale: invariant not claimed
                continue
            j = 16 * b + arg[r, b]
            amax_b = blocks[r, b].max()
            assert codes[r, j] & 7 == 7
            assert abs(abs(deq[r, j]) - amax_b) <= (2 ** -4 + 2 ** -20) * amax_b
            checked += 1
    assert checked > 3000


def test_rne_dequantized_error_within_half_step():
    x = inputs.student_t(64, 1024, 12)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    q = oracle.quantize(x)
    deq = oracle.dequantize(q["codes"], q["scales"], q["s_g"])
    unit = np.repeat(_torch_e4m3_values(q["scales"]), 16, axis=1) * float(q["s_g"])
    # position of |x| on the grid of this block, in grid units
    a = np.abs(xf) / np.where(unit == 0, 1, unit)
    k = np.clip(np.searchsorted(GRID, a, side="right") - 1, 0, 6)
    half_step = np.where(a >= 6, np.inf, (GRID[k + 1] - GRID[k]) / 2)
    bound = half_step * unit * (1 + 2 ** -20) + 1e-30
    sat = a >= 6
    assert np.all(np.abs(deq - xf)[~sat] <= bound[~sat])
    assert np.all(np.abs(deq)[sat] == 6 * unit[sat])


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("use_rht", [False, True])
def test_colwise_equals_rowwise_of_transpose(rounding, use_rht):
    x = _rand_bits(48, 80, 21, outliers=2)
    kw = dict(scaling=0, rounding=rounding, use_rht=use_rht, sign_mask=0x3C5A, seed=99, stream_id=4)
    col = oracle.quantize(x, oracle.COLWISE, **kw)
    row_t = oracle.quantize(np.ascontiguousarray(x.T), oracle.ROWWISE, **kw)
    assert col["amax"] == row_t["amax"]
    assert np.array_equal(col["codes"], row_t["codes"])
    assert np.array_equal(col["scales"], row_t["scales"])


@pytest.mark.parametrize("rounding", [0, 1])
def test_2d_colwise_is_exact_transpose(rounding):
    """16x16 scaling gives the same quantized tensor in both orientations
    ("Pretraining LLMs with NVFP4", Sec. 4 Two-dimensional scaling)."""
    x = _rand_bits(64, 96, 31, scale=0.02)
    kw = dict(scaling=1, rounding=rounding, seed=5, stream_id=1)
    row = oracle.quantize(x, oracle.ROWWISE, **kw)
    col = oracle.quantize(x, oracle.COLWISE, **kw)
    assert np.array_equal(_unpack(row["codes"]), _unpack(col["codes"]).T)
    # one scale per 16x16 tile, repeated along the tile's 16 rows
    tiles_r = row["scales"].reshape(4, 16, 6)
    assert np.all(tiles_r == tiles_r[:, :1, :])
    assert np.array_equal(tiles_r[:, 0, :], col["scales"].reshape(6, 16, 4)[:, 0, :].T)
    # the tile scale comes from the tile amax
    xf = np.abs(inputs.bf16_bits_to_f32(x)).reshape(4, 16, 6, 16).max(axis=(1, 3))
    r, c = np.unravel_index(np.argmax(xf), xf.shape)
    assert tiles_r[r, 0, c] == 0x7E


def test_rht_quantize_equals_quantize_of_rotated_input():
    """With the RHT on, the oracle quantizes U x blockwise ("Full-Stack FP4"
    Eq. (2)); for small-integer inputs U x is exact, so rotating by the
    Sylvester matrix first and quantizing without RHT must agree bit for bit."""
    rng = np.random.default_rng(8)
    xf = rng.integers(-8, 9, (32, 64)).astype(np.float32)
    mask = 0x9E37
    U = (_sylvester(16) @ np.diag([-1 if (mask >> i) & 1 else 1 for i in range(16)])) / 4.0
    rot = (xf.reshape(32, 4, 16).astype(np.float64) @ U.T).reshape(32, 64).astype(np.float32)
    x = inputs.to_bf16_bits(xf)
    x_rot = inputs.to_bf16_bits(rot)
    assert np.array_equal(inputs.bf16_bits_to_f32(x_rot), rot)     # exact in bf16
    for rounding in (0, 1):
        a = oracle.quantize(x, use_rht=True, sign_mask=mask, rounding=rounding, seed=3)
        b = oracle.quantize(x_rot, use_rht=False, rounding=rounding, seed=3)
        assert a["amax"] == b["amax"]
        assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["scales"], b["scales"])


def test_sr_quantize_is_seeded_and_stream_separated():
    x = inputs.student_t(16, 256, 4)
    a = oracle.quantize(x, rounding=1, seed=10, stream_id=1)
    b = oracle.quantize(x, rounding=1, seed=10, stream_id=1)
    c = oracle.quantize(x, rounding=1, seed=10, stream_id=2)
    d = oracle.quantize(x, rounding=1, seed=11, stream_id=1)
    assert np.array_equal(a["codes"], b["codes"])
    assert not np.array_equal(a["codes"], c["codes"])
    assert not np.array_equal(a["codes"], d["codes"])
    assert np.array_equal(a["scales"], c["scales"])


def test_quantize_row_subset_matches_full():
    x = _rand_bits(64, 128, 2, outliers=1)
    full = oracle.quantize(x, rounding=1, seed=1)
    part = oracle.quantize(x, rounding=1, seed=1, rows_subset=(17, 40))
    assert np.array_equal(full["codes"][17:40], part["codes"])
    assert np.array_equal(full["scales"][17:40], part["scales"])


def test_quantize_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((16, 24), np.uint16))
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((16, 32), np.uint16), scaling=1, use_rht=True)
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((24, 32), np.uint16), scaling=1)


# --------------------------------------------------------- extreme range ----
# Tensors whose block amaxes span 2^-40 of the tensor amax (subnormal and zero
# block scales), with tensor amaxes from the smallest bfloat16 subnormal (the
# tensor scale saturates at FLT_MAX and S_enc / s_b overflows) to 3e38.  The
# encode is checked against the format's definition evaluated in float64:
# the code of x is the E2M1 grid point nearest to |x| / (s_b * s_g) with
# s_b decoded by torch, i.e. x^ = x_E2M1 * s * s_g ("Full-Stack FP4", Sec. 2).
FLT_MAX = float(np.finfo(np.float32).max)
EXTREME_AMAX = [2688.0, 2.0 ** -133, float(np.float32(1e-36)), 3.0e38]


def _extreme(amax, span=40, seed=0):
    return inputs.extreme_range(64, 256, seed + 7, amax, span_log2=span)


def test_tensor_scale_saturates_for_a_subnormal_amax():
    """amax = 2^-133 (smallest bfloat16 subnormal): 2688 / amax overflows, so
    S_enc = FLT_MAX and s_g = RN(1 / FLT_MAX) = 2^-128 (1 / FLT_MAX is
    2^-128 (1 + 2^-24 + ...), whose nearest binary32 value, a subnormal with
    spacing 2^-149, is 2^-128)."""
    s_enc, s_g = oracle.tensor_scale(2.0 ** -133)
    assert s_enc == np.float32(FLT_MAX)
    exact = Fraction(1) / Fraction(int(np.float32(FLT_MAX)))
    assert Fraction(float(s_g)) == Fraction(1, 2 ** 128)
    assert abs(exact - Fraction(1, 2 ** 128)) < Fraction(1, 2 ** 150)


def _nearest_grid_f64(a):
    """Index of the E2M1 grid point nearest to a >= 0 (saturating at 6), and
    the distance of a to the nearest decision boundary (midpoint)."""
    k = np.clip(np.searchsorted(GRID, a, side="right") - 1, 0, 7)
    k1 = np.minimum(k + 1, 7)
    mid = (GRID[k] + GRID[k1]) / 2
    idx = np.where((k < 7) & (a > mid), k1, k)
    margin = np.where(k < 7, np.abs(a - mid), np.inf)
    return idx, margin


@pytest.mark.parametrize("amax", EXTREME_AMAX)
@pytest.mark.parametrize("orientation", [oracle.ROWWISE, oracle.COLWISE])
@pytest.mark.parametrize("scaling", [0, 1])
def test_rne_encode_is_the_nearest_grid_point_across_the_range(amax, orientation, scaling):
    """Every RNE code (no RHT) is the grid point nearest to |x| S_enc / s_b
    computed in float64, with x's sign bit (also for -0); blocks whose scale
    rounded to 0 encode every element as a signed zero."""
    x = _extreme(amax)
    q = oracle.quantize(x, orientation, scaling=scaling)
    xf = inputs.bf16_bits_to_f32(x)
    if orientation == oracle.COLWISE:
        xf = np.ascontiguousarray(xf.T)
    assert q["amax"] == np.float32(np.abs(xf).max())
    codes = _unpack(q["codes"])
    sb = np.repeat(_torch_e4m3_values(q["scales"]), 16, axis=1)
    s_enc = float(q["s_enc"])
    a = np.abs(xf.astype(np.float64)) * s_enc / np.where(sb == 0, 1.0, sb)
    idx, margin = _nearest_grid_f64(a)
    decided = (sb > 0) & (margin > 1e-5 * np.maximum(a, 1.0))
    assert decided.sum() >= 0.9 * (sb > 0).sum() > 0
    assert np.array_equal(codes[decided] & 7, idx[decided])
    assert np.all(codes[sb == 0] & 7 == 0)
    assert np.array_equal((codes & 8) != 0, np.signbit(xf))


@pytest.mark.parametrize("amax", EXTREME_AMAX)
@pytest.mark.parametrize("use_rht", [False, True])
def test_sr_codes_are_a_neighbouring_grid_point_across_the_range(amax, use_rht):
    """SR codes are one of the two grid points around |x| S_enc / s_b (the
    value itself when it is a grid point); with the RHT the rotated values
    come from the pinned rht16."""
    if use_rht and amax > 1e37:
        amax = 1.0e37        # the butterfly of 16 such values stays finite
    x = _extreme(float(inputs.bf16_bits_to_f32(inputs.to_bf16_bits(np.array([amax], np.float32)))[0]))
    q = oracle.quantize(x, rounding=1, use_rht=use_rht, sign_mask=0x6A5C, seed=3)
    xf = inputs.bf16_bits_to_f32(x)
    if use_rht:
        xf = np.stack([oracle.rht16(b, 0x6A5C) for b in xf.reshape(-1, 16)]).reshape(xf.shape)
    codes = _unpack(q["codes"])
    sb = np.repeat(_torch_e4m3_values(q["scales"]), 16, axis=1)
    a = np.abs(xf.astype(np.float64)) * float(q["s_enc"]) / np.where(sb == 0, 1.0, sb)
    lo = np.clip(np.searchsorted(GRID, a * (1 - 1e-6), side="right") - 1, 0, 7)
    hi = np.minimum(np.clip(np.searchsorted(GRID, a * (1 + 1e-6), side="left"), 0, 7), 7)
    mag = codes & 7
    ok = (sb == 0) & (mag == 0) | (sb > 0) & (mag >= lo) & (mag <= hi)
    assert ok.all(), np.argwhere(~ok)[:5]


@pytest.mark.parametrize("amax", EXTREME_AMAX)
def test_46_and_requantize_stay_finite_across_the_range(amax):
    """4/6 scaling and the Wgrad re-quantization on extreme tensors decode to
    values within the block's reach: every decoded |x^| <= 6 s_b s_g, zeros
    of x give zeros (4/6, no RHT)."""
    x = _extreme(amax)
    q = oracle.quantize(x, scaling=2)
    deq = oracle.dequantize(q["codes"], q["scales"], q["s_g"])
    xf = inputs.bf16_bits_to_f32(x)
    assert np.all(np.isfinite(deq))
    assert np.all(deq[xf == 0] == 0)
    unit = np.repeat(_torch_e4m3_values(q["scales"]), 16, axis=1) * float(q["s_g"])
    assert np.all(np.abs(deq) <= 6 * unit * (1 + 2 ** -20))
    if amax <= 1e37:
        r = oracle.requantize_col_rht(oracle.quantize(x), 0x1234, rounding=1, seed=2)
        assert np.all(np.isfinite(oracle.dequantize(r["codes"], r["scales"], r["s_g"])))


def test_overflowing_multiplier_encodes_by_the_quotient():
    """A tensor amax of about 1e-36 saturates S_enc at FLT_MAX; blocks whose
    amax is below about 1.6e-38 get E4M3 scales below 1, where S_enc / s_b
    overflows: their values are encoded as (x S_enc) / s_b, so a block of
    [a, a/2, a/100, 0, -0] keeps the ratios (6, 3, 0, 0, -0) instead of
    becoming all +-6 (and NaN for the zeros)."""
    a = np.float32(2.0 ** -128)                 # 2.9e-39: its block scale is below 1
    row = np.zeros(16, np.float32)
    row[:5] = [a, a / 2, a / 100, 0.0, -0.0]
    x = np.zeros((16, 32), np.float32)
    x[0, 16:] = row
    x[0, 0] = np.float32(1e-36)
    bits = inputs.to_bf16_bits(x)
    q = oracle.quantize(bits)
    assert q["s_enc"] == np.float32(FLT_MAX)
    sb = _torch_e4m3_values(q["scales"][:1, 1:2])[0, 0]
    assert 0 < sb < 1
    assert float(np.float32(FLT_MAX)) / sb > FLT_MAX      # r_b would overflow
    codes = _unpack(q["codes"])[0, 16:21]
    assert list(codes) == [7, 5, 0, 0, 8]


# ------------------------------------------------- 4/6 adaptive scaling ----
# "Full-Stack FP4" names 4/6 scaling (its related-work section: MSE-optimal
# adaptive block scaling) without printing the rule; the oracle's reading is
# "encode each 1x16 block with its amax mapped to 6 and to 4 (RNE), keep the
# closer one in squared error".  These pins check that reading against
# hand-built blocks and an independent float64 computation of both errors.
SCALE_46 = 2


def _e4m3_code_of(value):
    t = torch.tensor([value], dtype=torch.float32).to(torch.float8_e4m3fn)
    return int(t.view(torch.uint8).item())


def test_46_keeps_exact_four_and_exact_six_blocks():
    """S_enc = 2688 / 42 = 64.  Block 1 holds values of {0, 0.5 ... 4}: with its
    amax mapped to 4 the scale is 64 and every value is on the grid; with the
    amax mapped to 6 the scale is E4M3(42.67) = 44 and most are not.  Block 2
    holds values of {0 ... 6}: exact with the amax mapped to 6 (scale 64),
    inexact mapped to 4 (scale 96).  Block 0 holds the tensor amax, where
    both mappings saturate at 448 and the tie keeps 6."""
    blk0 = [42.0] + [0.0] * 15
    blk1 = [4, 3, 2, 1.5, 1, 0.5, 0, -4, -3, -2, -1.5, -1, -0.5, 0, 2, 4]
    blk2 = [6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, 6]
    xf = np.array([blk0 + blk1 + blk2], np.float32)
    x = inputs.to_bf16_bits(xf)
    q46 = oracle.quantize(x, scaling=SCALE_46)
    q6 = oracle.quantize(x)
    assert float(q46["s_enc"]) == 64.0
    assert list(q46["scales"][0]) == [0x7E, _e4m3_code_of(64.0), _e4m3_code_of(64.0)]
    assert list(q6["scales"][0]) == [0x7E, _e4m3_code_of(44.0), _e4m3_code_of(64.0)]
    deq46 = oracle.dequantize(q46["codes"], q46["scales"], q46["s_g"])[0]
    deq6 = oracle.dequantize(q6["codes"], q6["scales"], q6["s_g"])[0]
    assert np.array_equal(deq46[16:], xf[0, 16:].astype(np.float64))
    assert not np.array_equal(deq6[16:32], xf[0, 16:32].astype(np.float64))
    assert np.array_equal(deq6[32:], xf[0, 32:].astype(np.float64))


def _block_errors_f64(xf, s_enc, amax_b):
    """Squared error of both candidates in float64, from the pinned E4M3 and
    E2M1 primitives; the encode multiplications stay binary32 as read."""
    out = {}
    for m in (6.0, 4.0):
        sb32 = np.float32(np.float32(np.float32(amax_b) / np.float32(m)) * np.float32(s_enc))
        code = _e4m3_code_of(float(min(sb32, np.float32(448.0))))
        sb = float(_torch_e4m3_values(np.array([code], np.uint8))[0])
        r = np.float32(0.0) if sb == 0 else np.float32(np.float32(s_enc) / np.float32(sb))
        v = (xf.astype(np.float32) * r).astype(np.float32)
        g = _e2m1_values(oracle.e2m1_rne_array(v).astype(np.int64))
        err = float(np.sum((xf.astype(np.float64) * float(s_enc) - g * sb) ** 2))
        out[m] = (code, err)
    return out


@pytest.mark.parametrize("gen", ["normal", "student_t"])
def test_46_choice_is_the_lower_squared_error(gen):
    x = (inputs.normal(64, 256, 31, outlier_channels=2) if gen == "normal"
         else inputs.student_t(64, 256, 32))
    xf = inputs.bf16_bits_to_f32(x)
    q = oracle.quantize(x, scaling=SCALE_46)
    s_enc = float(q["s_enc"])
    checked = fours = 0
    for r in range(64):
        for b in range(16):
            blk = xf[r, 16 * b:16 * b + 16]
            e = _block_errors_f64(blk, s_enc, np.abs(blk).max())
            (c6, e6), (c4, e4) = e[6.0], e[4.0]
            if abs(e4 - e6) <= 1e-6 * max(e4, e6, 1e-30):
                continue   # too close for a float64 reference to decide a binary32 choice
            want = c4 if e4 < e6 else c6
            assert q["scales"][r, b] == want, (r, b, e6, e4)
            fours += want == c4 and c4 != c6
            checked += 1
    assert checked > 900 and fours > 50


def test_46_error_never_above_plain_scaling():
    x = inputs.student_t(32, 512, 33)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    q46 = oracle.quantize(x, scaling=SCALE_46)
    q6 = oracle.quantize(x)
    d46 = (oracle.dequantize(q46["codes"], q46["scales"], q46["s_g"]) - xf) ** 2
    d6 = (oracle.dequantize(q6["codes"], q6["scales"], q6["s_g"]) - xf) ** 2
    b46 = d46.reshape(32, 32, 16).sum(axis=2)
    b6 = d6.reshape(32, 32, 16).sum(axis=2)
    assert np.all(b46 <= b6 * (1 + 1e-5) + 1e-30)
    assert b46.sum() < b6.sum()


def test_46_sr_uses_the_rne_choice_of_scale():
    x = _rand_bits(32, 256, 34, outliers=1)
    rne = oracle.quantize(x, scaling=SCALE_46)
    sr = oracle.quantize(x, scaling=SCALE_46, rounding=1, seed=3, stream_id=1)
    assert np.array_equal(rne["scales"], sr["scales"])
    assert not np.array_equal(rne["codes"], sr["codes"])


# ------------------------------------------ Wgrad re-quantization (Eq. 2) ----
@pytest.mark.parametrize("k", [0, 2])
@pytest.mark.parametrize("rounding", [0, 1])
def test_requantize_equals_quantizing_the_dequantized_values(k, rounding):
    """With s_g a power of two (tensor amax 2688 * 2^k) every dequantized value
    e2m1 * s_b * s_g has at most 6 significant bits, so it is a bf16 value, and
    re-quantizing the operand must equal the (separately pinned) col-wise RHT
    quantization of those bf16 values ("Full-Stack FP4", Sec. 3.2 Eq. (2):
    Q_16x1(H^T Q_1x16(X)))."""
    xf = inputs.bf16_bits_to_f32(inputs.normal(96, 64, 40 + k, outlier_channels=1)).copy()
    xf[5, 7] = 2688.0 * 2 ** k
    x = inputs.to_bf16_bits(xf)
    q = oracle.quantize(x)
    assert float(q["s_g"]) == 2.0 ** k
    xhat = oracle.dequantize(q["codes"], q["scales"], q["s_g"])
    bits = inputs.to_bf16_bits(xhat.astype(np.float32))
    assert np.array_equal(inputs.bf16_bits_to_f32(bits).astype(np.float64), xhat)
    want = oracle.quantize(bits, oracle.COLWISE, rounding=rounding, use_rht=True, sign_mask=0x6C39,
                           seed=9, stream_id=4)
    got = oracle.requantize_col_rht(q, 0x6C39, rounding=rounding, seed=9, stream_id=4)
    assert got["amax"] == want["amax"]
    assert np.array_equal(got["codes"], want["codes"]) and np.array_equal(got["scales"], want["scales"])


def test_requantize_row_subset_and_zero_operand():
    q = oracle.quantize(_rand_bits(64, 48, 41, outliers=1))
    full = oracle.requantize_col_rht(q, 0x0F0F, rounding=1, seed=2)
    part = oracle.requantize_col_rht(q, 0x0F0F, rounding=1, seed=2, rows_subset=(16, 40))
    assert np.array_equal(full["codes"][16:40], part["codes"])
    assert np.array_equal(full["scales"][16:40], part["scales"])
    z = oracle.requantize_col_rht(oracle.quantize(np.zeros((32, 32), np.uint16)), 0xFFFF)
    # all values zero (the sign flips of the RHT leave negative zeros, code 0x8)
    assert z["amax"] == 0 and not (z["codes"] & 0x77).any() and not z["scales"].any()


# ------------------------------------------------ LoRA-SVD branch (Eq. 1) ----
def test_gemm_lora_adds_the_low_rank_product():
    """Full-Stack FP4, Sec. 3.2 Eq. (1): Y = Q(X) Q(W)^T + beta (X L1^T) L2^T.
    With an all-zero FP4 operand the result is exactly beta U V^T, checked
    against a triple loop on small integers; otherwise the low-rank term is
    added to the FP4 GEMM."""
    u_f = (np.arange(8 * 64, dtype=np.float32).reshape(8, 64) % 5) - 2
    v_f = (np.arange(6 * 64, dtype=np.float32).reshape(6, 64) % 3) - 1
    u, v = inputs.to_bf16_bits(u_f), inputs.to_bf16_bits(v_f)
    brute = np.array([[-0.75 * sum(int(u_f[i, k]) * int(v_f[j, k]) for k in range(64)) for j in range(6)]
                      for i in range(8)])
    zero = oracle.quantize(np.zeros((8, 64), np.uint16))
    b = oracle.quantize(inputs.normal(6, 64, 2))
    y, ab, la = oracle.gemm_lora_f64(zero, b, u, v, -0.75)
    assert np.array_equal(y, brute) and not ab.any()
    assert np.array_equal(la, np.abs(brute) * 0 + 0.75 * (np.abs(u_f).astype(np.float64) @ np.abs(v_f).T))
    a = oracle.quantize(inputs.normal(8, 64, 1))
    y, _, _ = oracle.gemm_lora_f64(a, b, u, v, -0.75)
    y0, _ = oracle.gemm_f64(a, b)
    assert np.allclose(y - y0, brute, rtol=0, atol=1e-9)


# ---------------------------------------------------------- dequantize ----
def test_dequantize_grid_values():
    codes4 = np.arange(16, dtype=np.uint8)
    packed = (codes4[0::2] | (codes4[1::2] << 4)).reshape(1, 8)
    ones = np.full((1, 1), 0x38, np.uint8)                # E4M3 1.0
    deq = oracle.dequantize(packed, ones, 1.0)[0]
    assert np.array_equal(deq[:8], GRID) and np.array_equal(deq[8:], -GRID)
    # x^ = x_E2M1 * s * s_g ("Full-Stack FP4", Sec. 2) with dyadic s and s_g
    sc = np.full((1, 1), 0x48, np.uint8)                 # E4M3 4.0 (exponent 9)
    deq = oracle.dequantize(packed, sc, 0.125)[0]
    assert np.array_equal(deq[:8], GRID * 4 * 0.125)


def test_round_bf16_single_rounding():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(5000), rng.standard_normal(5000) * 1e-30,
                        rng.standard_normal(5000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    ours = np.array([oracle.round_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(ours, ref)
    # above a bf16 tie by less than a float32 ulp: must round up, not to even
    assert oracle.round_bf16(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.round_bf16(1.0 + 2 ** -8) == 0x3F80
    assert oracle.round_bf16(-(1.0 + 3 * 2 ** -8)) == 0xBF82


# ---------------------------------------------------------------- GEMM ----
def _random_operand(rng, rows, K, scale_max=0x7E):
    codes = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    scales = rng.integers(0, scale_max + 1, (rows, K // 16), dtype=np.uint8)
    s_g = np.float32(rng.uniform(0.01, 3.0))
    return dict(codes=codes, scales=scales, s_g=s_g)


def _exact_gemm(a, b):
    """Exact rational y = s_gA s_gB sum_k (e2m1 * s)(e2m1 * s), decoded with the
    page grid and torch's E4M3 table."""
    ea = _e2m1_values(_unpack(a["codes"]))
    eb = _e2m1_values(_unpack(b["codes"]))
    sa = np.repeat(_torch_e4m3_values(a["scales"]), 16, axis=1)
    sb = np.repeat(_torch_e4m3_values(b["scales"]), 16, axis=1)
    M, K = ea.shape
    N = eb.shape[0]
    sg = Fraction(float(a["s_g"])) * Fraction(float(b["s_g"]))
    y = np.empty((M, N), object)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(ea[m, k]) * Fraction(sa[m, k]) * Fraction(eb[n, k]) * Fraction(sb[n, k])
            y[m, n] = acc * sg
    return y


def test_gemm_matches_exact_rational_brute_force():
    rng = np.random.default_rng(13)
    for _ in range(3):
        a = _random_operand(rng, 4, 32)
        b = _random_operand(rng, 4, 32)
        y, ab = oracle.gemm_f64(a, b)
        exact = _exact_gemm(a, b)
        for m in range(4):
            for n in range(4):
                assert y[m, n] == float(exact[m, n])


def test_gemm_integer_special_case():
    """All scales 1 and s_g = 1: an integer-valued dot product of E2M1 values."""
    rng = np.random.default_rng(14)
    a = _random_operand(rng, 8, 64)
    b = _random_operand(rng, 6, 64)
    a["scales"][:] = 0x38
    b["scales"][:] = 0x38
    a["s_g"] = b["s_g"] = np.float32(1.0)
    y, _ = oracle.gemm_f64(a, b)
    ia = (2 * _e2m1_values(_unpack(a["codes"]))).astype(np.int64)
    ib = (2 * _e2m1_values(_unpack(b["codes"]))).astype(np.int64)
    assert np.array_equal(y * 4, (ia @ ib.T).astype(np.float64))


def test_gemm_gram_matrix_is_symmetric_psd_diagonal():
    x = _rand_bits(24, 128, 15)
    q = oracle.quantize(x)
    y, ab = oracle.gemm_f64(q, q)
    assert np.array_equal(y, y.T)
    assert np.all(np.diag(y) >= 0) and np.array_equal(np.diag(y), np.diag(ab))


def test_gemm_row_subset():
    rng = np.random.default_rng(16)
    a = _random_operand(rng, 10, 64)
    b = _random_operand(rng, 7, 64)
    full, _ = oracle.gemm_f64(a, b)
    sub, _ = oracle.gemm_f64(a, b, row_ids=[9, 0, 4])
    assert np.array_equal(sub, full[[9, 0, 4]])


def test_sr_gemm_error_variance_matches_eq5():
    """Appendix 7, Eq. (5): with SR the output error is unbiased with variance
    sum_i (x_i^2 s_w,i^2 + w_i^2 s_x,i^2 + s_x,i^2 s_w,i^2)."""
    rng = np.random.default_rng(17)
    K = 256
    x = inputs.to_bf16_bits(rng.uniform(-1, 1, (3, K)).astype(np.float32))
    w = inputs.to_bf16_bits(rng.uniform(-1, 1, (4, K)).astype(np.float32))
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    wf = inputs.bf16_bits_to_f32(w).astype(np.float64)
    y_true = xf @ wf.T

    def sr_var(bits, q):
        vals = inputs.bf16_bits_to_f32(bits).astype(np.float64)
        unit = np.repeat(_torch_e4m3_values(q["scales"]), 16, axis=1) * float(q["s_g"])
        a = np.abs(vals) / unit
        k = np.clip(np.searchsorted(GRID, a, side="right") - 1, 0, 6)
        d = a - GRID[k]
        return d * (GRID[k + 1] - GRID[k] - d) * unit ** 2

    S = 400
    errs = []
    for s in range(S):
        qx = oracle.quantize(x, rounding=1, seed=1000 + s, stream_id=1)
        qw = oracle.quantize(w, rounding=1, seed=5000 + s, stream_id=2)
        y, _ = oracle.gemm_f64(qx, qw, with_abs=False)
        errs.append(y - y_true)
    errs = np.array(errs)
    var_x = sr_var(x, qx)
    var_w = sr_var(w, qw)
    pred = (xf ** 2) @ var_w.T + var_x @ (wf ** 2).T + var_x @ var_w.T
    emp = errs.var(axis=0)
    assert abs(emp.mean() / pred.mean() - 1) < 0.1
    assert np.all(np.abs(errs.mean(axis=0)) <= 5 * np.sqrt(pred / S))


# -------------------------------------------------------------- inputs ----
def test_input_generators_are_seeded_and_shaped():
    a = inputs.normal(32, 64, 1, outlier_channels=2)
    b = inputs.normal(32, 64, 1, outlier_channels=2)
    assert np.array_equal(a, b) and a.dtype == np.uint16
    assert inputs.rht_sign_mask(3) == inputs.rht_sign_mask(3)
    for rows, L in inputs.c5_sweep_sizes():
        assert rows % 16 == 0 and rows * L <= 1 << 29
    with open(os.path.join(GOLDEN, "model_3b_shapes.txt")) as f:
        shapes = dict(line.split() for line in f if line.strip() and not line.startswith("#"))
    assert int(shapes["hidden"]) == inputs.HIDDEN and int(shapes["ffn"]) == inputs.FFN
    assert int(shapes["heads"]) == inputs.N_HEADS and int(shapes["kv_heads"]) == inputs.N_KV_HEADS

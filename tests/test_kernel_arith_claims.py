"""The exactness claims the CUDA kernels' arithmetic relies on, checked on
the CPU with numpy binary32 (independent of both the kernels and the oracle):

1. every product g * s of an E2M1 magnitude and an E4M3 scale is exact in
   binary32, so RN(x - g s) is one fused multiply-add (4/6 block scales);
2. the re-quantization's values t = H16 D x (unscaled butterfly of inputs
   RN(RN(g s_b) s_g)) satisfy t / 4 exact whenever s_g >= 2^-114, so the
   transform's 1/4 may go into the multipliers; below that bound it can fail;
3. D's sign flip on the block scale gives the same value as on the product.
"""
import numpy as np

F32 = np.float32
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_values():
    """The 126 finite positive E4M3 (FN) values and zero, from the bit layout
    (bias 7, 3 mantissa bits, subnormals below 2^-6; code 0x7F is NaN)."""
    out = []
    for code in range(127):
        e, m = code >> 3, code & 7
        out.append(m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8))
    return out


def butterfly16(x):
    """Stages 0..3 of the 16-point Walsh-Hadamard butterfly in binary32, the
    kernels' order: pair (i, i ^ 2^s) -> (a + b, a - b)."""
    t = x.astype(F32).copy()
    for s in range(4):
        for i in range(16):
            if i & (1 << s):
                continue
            a, b = t[i], t[i | (1 << s)]
            t[i], t[i | (1 << s)] = F32(a + b), F32(a - b)
    return t


def test_e2m1_times_e4m3_is_exact_in_binary32():
    for g in E2M1:
        for s in e4m3_values():
            exact = g * s                                  # float64: exact for these
            assert float(F32(g) * F32(s)) == exact
            assert exact == 0 or 2.0 ** -10 <= exact <= 2688.0


def _requant_inputs(rng, sg, n_blocks):
    g = rng.choice(np.array(E2M1 + [-v for v in E2M1[1:]]), size=(n_blocks, 16))
    sb = np.array(e4m3_values())[rng.integers(1, 127, size=(n_blocks, 1))]
    # the smallest products appear in every block: g = 0.5 with s_b = 2^-9
    g[:, 0], sb[::4] = 0.5, 2.0 ** -9
    return (F32(g) * F32(sb)).astype(F32) * F32(sg)        # RN(RN(g s_b) s_g)


def test_quarter_of_the_butterfly_is_exact_when_sg_at_least_2_pow_minus_114():
    rng = np.random.default_rng(11)
    for sg in [2.0 ** -114, 1.3 * 2.0 ** -114, 2.0 ** -100, 2.0 ** -60, 1e-3, 1.0]:
        x = _requant_inputs(rng, sg, 2000)
        assert np.all((x == 0) | (np.abs(x) >= F32(2.0 ** -124)))
        for row in x:
            t = butterfly16(row)
            q = (t * F32(0.25)).astype(F32)
            assert np.array_equal(q.astype(np.float64) * 4, t.astype(np.float64)), sg


def test_quarter_can_round_below_the_bound():
    # with s_g = 2^-140 the inputs are subnormal and t / 4 loses bits
    rng = np.random.default_rng(12)
    x = _requant_inputs(rng, 2.0 ** -140, 2000)
    lost = 0
    for row in x:
        t = butterfly16(row)
        q = (t * F32(0.25)).astype(F32)
        lost += int(np.any(q.astype(np.float64) * 4 != t.astype(np.float64)))
    assert lost > 0


def test_sign_flip_on_the_scale_equals_the_flip_of_the_product():
    rng = np.random.default_rng(13)
    for _ in range(20000):
        g = F32(rng.choice(E2M1) * rng.choice([-1, 1]))
        sb = F32(e4m3_values()[rng.integers(0, 127)])
        sg = F32(2.0 ** rng.uniform(-126, 0))
        a = F32(F32(g * -sb) * sg)
        b = -F32(F32(g * sb) * sg)
        assert np.signbit(a) == np.signbit(b) and a == b

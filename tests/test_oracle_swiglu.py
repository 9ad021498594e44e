"""Pins for the oracle's SwiGLU expert over FP8 weights.

The expert is down(silu(gate x) * up x) with no bias ("Kimi-K2-Base",
Feed-forward: Activation SwiGLU, FFN bias No), FP8 e4m3 weights with 128x128
block scales and 1x128 activation quantisation.
"""
import numpy as np

from oracle import moe_oracle as O

ONE, TWO = 0x38, 0x40   # e4m3 codes of 1.0 and 2.0


def test_silu_closed_form():
    assert O.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.silu(np.array([50.0])), [50.0], rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array([-50.0])), [0.0], atol=1e-19)
    np.testing.assert_allclose(O.silu(np.array([1.0])), [1.0 / (1.0 + np.exp(-1.0))], rtol=1e-15)


def test_block_scale_grid_orientation():
    rng = np.random.default_rng(8)
    R, C = 256, 384
    q = rng.integers(0, 0x7E, (R, C)).astype(np.uint8)
    s = (2.0 ** rng.integers(-6, 6, (R // 128, C // 128))).astype(np.float32)
    w = O.decode_block_weight(q, s)
    for r, c in [(0, 0), (5, 200), (130, 10), (255, 383), (127, 256), (128, 255)]:
        assert w[r, c] == O.e4m3_value(int(q[r, c])) * float(s[r // 128, c // 128])


def _selection(rows, cols, src, code):
    w = np.zeros((rows, cols), dtype=np.uint8)
    w[np.arange(rows), src] = code
    return w


def test_selection_experts_closed_form():
    # gate row n reads input feature pi[n], up row n reads 2 * feature sig[n],
    # down row m reads hidden feature rho[m]: every output has a closed form,
    # and a transposed operand or a swapped gate/up role changes it
    rng = np.random.default_rng(9)
    n, d, H = 5, 384, 256
    x = rng.standard_normal((n, d)).astype(np.float32)
    xq, xs = O.quantize_1x128(x)
    xh = O.dequantize_1x128(xq, xs)
    pi, sig, rho = rng.integers(0, d, H), rng.integers(0, d, H), rng.integers(0, H, d)
    w1 = _selection(H, d, pi, ONE)
    w3 = _selection(H, d, sig, TWO)
    w2 = _selection(d, H, rho, ONE)
    ones_h = np.ones((H // 128, d // 128), np.float32)
    ones_d = np.ones((d // 128, H // 128), np.float32)
    o, hq, hs = O.swiglu_fp8(xq, xs, w1, ones_h, w3, ones_h, w2, ones_d)
    g = xh[:, pi]
    h = (g / (1 + np.exp(-g)) * (2 * xh[:, sig])).astype(np.float32)
    hq2, hs2 = O.quantize_1x128(h)
    np.testing.assert_array_equal(hq, hq2)
    np.testing.assert_array_equal(hs, hs2)
    hh = O.dequantize_1x128(hq2, hs2)
    np.testing.assert_array_equal(o, hh[:, rho])


def test_integer_exact_products():
    # integer-valued e4m3 weights and activations with power-of-two scales:
    # every product and sum is exact, so the result is the exact integer sum
    rng = np.random.default_rng(10)
    n, d, H = 3, 256, 128
    vals = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4], dtype=np.float64)
    codes = O.e4m3_encode(vals)
    xi = rng.integers(0, 9, (n, d)); xq = codes[xi]; x_int = vals[xi]
    xs = np.full((n, d // 128), 0.5, np.float32)
    w1i = rng.integers(0, 9, (H, d)); w3i = rng.integers(0, 9, (H, d)); w2i = rng.integers(0, 9, (d, H))
    s1 = np.array([[1.0, 2.0]], np.float32)            # [H/128, d/128]
    s3 = np.array([[0.25, 1.0]], np.float32)
    s2 = np.array([[1.0], [4.0]], np.float32)          # [d/128, H/128]
    g = np.zeros((n, H)); u = np.zeros((n, H))
    for t in range(n):
        for h_ in range(H):
            g[t, h_] = sum(x_int[t, i] * 0.5 * vals[w1i[h_, i]] * s1[0, i // 128] for i in range(d))
            u[t, h_] = sum(x_int[t, i] * 0.5 * vals[w3i[h_, i]] * s3[0, i // 128] for i in range(d))
    o, hq, hs = O.swiglu_fp8(xq, xs, codes[w1i], s1, codes[w3i], s3, codes[w2i], s2)
    h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
    hq2, hs2 = O.quantize_1x128(h)
    np.testing.assert_array_equal(hq, hq2)
    hh = O.dequantize_1x128(hq2, hs2)
    ref = np.zeros((n, d))
    for t in range(n):
        for m in range(d):
            ref[t, m] = sum(hh[t, j] * vals[w2i[m, j]] * s2[m // 128, 0] for j in range(H))
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=0)

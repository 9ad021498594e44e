"""Pins for the oracle's block pieces around the FFN: bf16 rounding, RMSNorm, the
residual addition and their composition with the MoE layer."""
import numpy as np
import torch

import moe_synth as S
from oracle import moe_oracle as O


def _bf16_bits_rne(v32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 by rounding the bit pattern (ties to even), as fp64 values."""
    b = v32.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def test_round_bf16_against_bit_rounding_and_torch():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(200_000) * 10.0 ** rng.integers(-6, 6, 200_000),
                        # exact midpoints between neighbouring bf16 values of both parities
                        (np.arange(256, 512) + 0.5) / 256.0, -(np.arange(256, 512) + 0.5) / 64.0]).astype(np.float32)
    got = O.round_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, _bf16_bits_rne(v))
    np.testing.assert_array_equal(got, torch.from_numpy(v).to(torch.bfloat16).double().numpy())


def test_round_bf16_worked_values():
    v = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9, 1.0 + 2.0 ** -9, 1.0 + 3 * 2.0 ** -8, 255.5, 0.0])
    # the midpoint 1 + 2^-8 goes to the even 1.0; 1 + 3*2^-8 is the midpoint above
    # 1 + 2^-7 (odd significand) and goes up to 1 + 2^-6; 255.5 -> 256 (ties to even)
    np.testing.assert_array_equal(O.round_bf16(v), [1.0, 1.0, 1.0 + 2.0 ** -7, 1.0, 1.0 + 2.0 ** -6, 256.0, 0.0])


def test_rms_norm_worked_examples(golden):
    for row in golden("rmsnorm_worked_example.txt"):
        n = int(row[0])
        vals = np.array([float(x) for x in row[1:]])
        h, g, y = vals[:n], vals[n:2 * n], vals[2 * n:3 * n]
        np.testing.assert_array_equal(O.rms_norm(h[None, :], g, eps=0.0)[0], y)


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(1)
    d = 7168
    # a constant row c with unit weights and no epsilon normalises to sign(c)
    for c in (0.37, -5.0, 1e-3):
        np.testing.assert_array_equal(O.rms_norm(np.full((1, d), c), np.ones(d), eps=0.0), np.sign(c))
    # epsilon enters under the root: h = 1e-3 everywhere, eps = 1e-6 -> 1e-3 / sqrt(2e-6)
    y = O.rms_norm(np.full((1, d), 1e-3), np.ones(d), eps=1e-6)
    np.testing.assert_array_equal(y, O.round_bf16(np.full((1, d), 1e-3 / np.sqrt(2e-6))))
    # a zero row stays zero (no division by zero with eps > 0)
    assert (O.rms_norm(np.zeros((1, d)), np.ones(d)) == 0).all()
    # per-feature weights scale their own column only: gamma = 2 on one feature
    h = rng.standard_normal((3, d))
    g = np.ones(d)
    g[17] = 2.0
    a, b = O.rms_norm(h, np.ones(d), eps=0.0), O.rms_norm(h, g, eps=0.0)
    np.testing.assert_array_equal(np.delete(a, 17, axis=1), np.delete(b, 17, axis=1))
    np.testing.assert_array_equal(b[:, 17], 2.0 * a[:, 17])   # times 2 is exact in bf16


def test_rms_norm_invariances():
    rng = np.random.default_rng(2)
    d = 1024
    h = rng.standard_normal((5, d))
    g = rng.uniform(0.5, 1.5, d)
    # exact power-of-two rescaling of a row cancels (eps = 0)
    np.testing.assert_array_equal(O.rms_norm(8.0 * h, g, eps=0.0), O.rms_norm(h, g, eps=0.0))
    # unit weights: the mean square of the output is 1 up to the bf16 rounding
    y = O.rms_norm(h, np.ones(d), eps=0.0)
    np.testing.assert_allclose((y * y).mean(axis=1), 1.0, rtol=2e-3)
    # rows are independent: permuting rows permutes the output
    perm = np.array([3, 0, 4, 1, 2])
    np.testing.assert_array_equal(O.rms_norm(h[perm], g), O.rms_norm(h, g)[perm])


def test_residual_add_rounds_twice():
    # the FFN output is a bf16 tensor before the addition: 1 + 2^-9 rounds to 1 first
    np.testing.assert_array_equal(O.residual_add(np.array([[0.0]]), np.array([[1.0 + 2.0 ** -9]])), [[1.0]])
    # then the sum of two bf16 values is rounded: 1 + 2^-8 (exact sum) -> 1 (ties to even)
    np.testing.assert_array_equal(O.residual_add(np.array([[1.0]]), np.array([[2.0 ** -8]])), [[1.0]])
    np.testing.assert_array_equal(O.residual_add(np.array([[1.0]]), np.array([[3 * 2.0 ** -8]])),
                                  [[1.0 + 2.0 ** -6]])


def test_block_ffn_wiring_with_silent_experts():
    # all-zero expert weights make the FFN output exactly 0, so the block returns
    # h itself (the residual is the block input, not the normalised x) and the next
    # input is RMSNorm_next(h); two different weights catch a swapped gamma
    shape = S.MoEShape("blk", T=6, d=256, E=8, topk=2, H=128)
    inp = S.gen_moe_inputs(shape, seed=3)
    ex = inp.experts
    zero = S.ExpertWeights(torch.zeros_like(ex.w13), ex.w13_s, torch.zeros_like(ex.w2), ex.w2_s)
    rng = np.random.default_rng(3)
    h = torch.from_numpy(rng.standard_normal((shape.T, shape.d)).astype(np.float32)).to(torch.bfloat16)
    g_post = np.full(shape.d, 0.5)
    g_next = np.full(shape.d, 2.0)
    out = O.moe_block_ffn(h, g_post, inp.w_gate, inp.bias, zero, shape.topk, shape.route_scale, gamma_next=g_next)
    hf = h.float().numpy().astype(np.float64)
    np.testing.assert_array_equal(out["y"], 0.0)
    np.testing.assert_array_equal(out["h_next"], hf)
    np.testing.assert_array_equal(out["x_next"], O.rms_norm(hf, g_next))
    np.testing.assert_array_equal(out["x"], O.rms_norm(hf, g_post))
    # the layer saw the normalised input: its quantised x decodes to rms_norm(h, g_post)
    deq = O.dequantize_1x128(out["xq"], out["xs"])
    np.testing.assert_allclose(deq, out["x"], rtol=2 ** -3, atol=1e-30)


def test_block_ffn_adds_the_layer_output():
    shape = S.MoEShape("blk2", T=5, d=256, E=8, topk=2, H=128)
    inp = S.gen_moe_inputs(shape, seed=4)
    rng = np.random.default_rng(4)
    h = torch.from_numpy(rng.standard_normal((shape.T, shape.d)).astype(np.float32)).to(torch.bfloat16)
    g = np.ones(shape.d)
    out = O.moe_block_ffn(h, g, inp.w_gate, inp.bias, inp.experts, shape.topk, shape.route_scale)
    ref = O.moe_layer(O.rms_norm(h.float().numpy(), g).astype(np.float32), inp.w_gate, inp.bias, inp.experts,
                      shape.topk, shape.route_scale)
    np.testing.assert_array_equal(out["y"], ref["y"])
    np.testing.assert_array_equal(out["h_next"], O.residual_add(h.float().numpy(), ref["y"]))
    assert "x_next" not in out

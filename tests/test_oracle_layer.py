"""Closed-form pins for the oracle's whole MoE layer.

Combine rule: y = shared(x) + sum_j w_j * expert_{I_j}(x) with sum_j w_j = 2.827
("Kimi-K2-Base", Mixture of experts: the routed scaling factor multiplies the
renormalised top-k weights; the shared expert is always on and unweighted).
"""
import numpy as np
import pytest
import torch

import moe_synth as S
from oracle import moe_oracle as O

SMALL = S.MoEShape("pin_t24_d256_e12_h128", T=24, d=256, E=12, topk=4, H=128)


def _inputs(shape, seed=0):
    return S.gen_moe_inputs(shape, seed=seed, device="cpu")


def _expert_out(inp, e, x):
    xq, xs = O.quantize_1x128(np.asarray(x, np.float32))
    ex = inp.experts
    o, _, _ = O.swiglu_fp8(xq, xs, ex.w13[e, 0].numpy(), ex.w13_s[e, 0].numpy(),
                           ex.w13[e, 1].numpy(), ex.w13_s[e, 1].numpy(),
                           ex.w2[e].numpy(), ex.w2_s[e].numpy())
    return o


def test_identical_routed_experts_reduce_to_scaled_expert_plus_shared():
    inp = _inputs(SMALL)
    ex = inp.experts
    for e in range(1, SMALL.E):         # every routed expert a copy of expert 0
        ex.w13[e].copy_(ex.w13[0]); ex.w13_s[e].copy_(ex.w13_s[0])
        ex.w2[e].copy_(ex.w2[0]); ex.w2_s[e].copy_(ex.w2_s[0])
    r = O.moe_layer(inp.x, inp.w_gate, inp.bias, ex, SMALL.topk, SMALL.route_scale)
    x = inp.x.float().numpy()
    want = _expert_out(inp, SMALL.E, x) + 2.827 * _expert_out(inp, 0, x)
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-12)


def test_slot_weight_multiplies_its_own_expert():
    # experts are copies of expert 0 whose down_proj scales are multiplied by
    # 2^e: expert e's output is exactly 2^e * R(x), so y = S(x) + sum_j w_j 2^{I_j} R(x)
    inp = _inputs(SMALL, seed=1)
    ex = inp.experts
    for e in range(1, SMALL.E):
        ex.w13[e].copy_(ex.w13[0]); ex.w13_s[e].copy_(ex.w13_s[0])
        ex.w2[e].copy_(ex.w2[0]); ex.w2_s[e].copy_(ex.w2_s[0] * 2.0 ** e)
    r = O.moe_layer(inp.x, inp.w_gate, inp.bias, ex, SMALL.topk, SMALL.route_scale)
    x = inp.x.float().numpy()
    R = _expert_out(inp, 0, x)
    mult = (r["w"] * 2.0 ** r["idx"]).sum(axis=1)
    want = _expert_out(inp, SMALL.E, x) + mult[:, None] * R
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-12)


def test_zero_input_gives_zero_output():
    inp = _inputs(SMALL, seed=2)
    x = torch.zeros_like(inp.x)
    r = O.moe_layer(x, inp.w_gate, inp.bias, inp.experts, SMALL.topk, SMALL.route_scale)
    assert (r["y"] == 0).all()
    assert (r["xs"] == 0).all() and (r["xq"] == 0).all()
    # all logits 0: scores 0.5, choice decided by the bias alone, equal weights
    order = np.lexsort((np.arange(SMALL.E), -inp.bias.double().numpy()))[:SMALL.topk]
    assert (r["idx"] == order[None, :]).all()
    np.testing.assert_allclose(r["w"], 2.827 / SMALL.topk, rtol=1e-15)


def test_token_subset_matches_full_rows():
    inp = _inputs(SMALL, seed=3)
    full = O.moe_layer(inp.x, inp.w_gate, inp.bias, inp.experts, SMALL.topk, SMALL.route_scale)
    part = O.moe_layer(inp.x, inp.w_gate, inp.bias, inp.experts, SMALL.topk, SMALL.route_scale,
                       tokens=[3, 17, 5])
    np.testing.assert_allclose(part["y"][[3, 5, 17]], full["y"][[3, 5, 17]], rtol=1e-12, atol=1e-14)
    assert np.isnan(part["y"][0]).all()
    np.testing.assert_array_equal(part["offsets"], full["offsets"])


def test_dense_swiglu_is_one_expert():
    inp = _inputs(SMALL, seed=4)
    ex = inp.experts
    x = inp.x.float().numpy()
    y, toks = O.dense_swiglu(inp.x, ex.w13[2], ex.w13_s[2], ex.w2[2], ex.w2_s[2])
    np.testing.assert_array_equal(y, _expert_out(inp, 2, x))

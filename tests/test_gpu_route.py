"""moe_route (tcgen05 bf16 router GEMM + warp top-k) against the oracle's gate."""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _parity import reconcile_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check(shape, x, wg, b):
    cfg = moe.cfg_of(shape)
    idx, w, scores = moe.route(x.to(DEV), wg.to(DEV), b.to(DEV), cfg, want_scores=True)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    r = O.route(x.float().numpy(), wg.float().numpy(), b.double().numpy(), shape.topk, shape.route_scale)
    np.testing.assert_allclose(scores.cpu().numpy(), r["scores"], rtol=2e-5, atol=2e-6)
    ref_idx = reconcile_routing(idx.cpu().numpy(), r, shape.topk)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    sel = np.take_along_axis(r["scores"], ref_idx, axis=1)
    w_ref = sel / sel.sum(1, keepdims=True) * shape.route_scale
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(w.cpu().numpy().sum(1), shape.route_scale, rtol=1e-5)
    return idx, r


@pytest.mark.parametrize("T", [1, 64, 130, 333])
def test_toy_router(T):
    shape = S.MoEShape("toy", T=T, d=1024, E=32, topk=8, H=256)
    x = S.gen_x(T, shape.d, seed=T)
    wg, b = S.gen_router(shape, seed=T)
    _check(shape, x, wg, b)


# batches past 512 tokens: 128-token tiles; one, three (the last ragged) and four
# 128-expert blocks of W_g, and the Kimi width
@pytest.mark.parametrize("T,E,d", [(600, 32, 1024), (1000, 384, 1024), (777, 300, 512), (520, 512, 256),
                                   (2048, 384, 7168)])
def test_router_token_tiles(T, E, d):
    shape = S.MoEShape(f"wide_router_{T}_{E}", T=T, d=d, E=E, topk=8, H=256)
    x = S.gen_x(T, d, seed=T + E)
    wg, b = S.gen_router(shape, seed=T + E)
    _check(shape, x, wg, b)


def test_kimi_router_decode_batch():
    shape = S.DECODE
    x = S.gen_x(shape.T, shape.d, seed=0)
    wg, b = S.gen_router(shape, seed=0)
    idx, r = _check(shape, x, wg, b)
    assert len(np.unique(idx.cpu().numpy())) > 300


def test_skewed_bias_routes_to_hot_experts():
    shape = S.MoEShape("skew_small", T=512, d=1024, E=384, topk=8, H=256, hot_experts=S.SKEWED.hot_experts,
                       hot_bias=0.5)
    x = S.gen_x(shape.T, shape.d, seed=5)
    wg, b = S.gen_router(shape, seed=5)
    idx, r = _check(shape, x, wg, b)
    hot = np.isin(idx.cpu().numpy(), shape.hot_experts).mean()
    assert hot > 0.5


def test_exact_ties_go_to_lower_id():
    # x = 0: all logits 0, scores 0.5; the bias alone decides, with repeated values
    shape = S.MoEShape("ties", T=40, d=256, E=64, topk=8, H=128)
    x = torch.zeros(shape.T, shape.d, dtype=torch.bfloat16)
    wg, _ = S.gen_router(shape, seed=1)
    b = torch.tensor([0.01 * (i % 5) for i in range(shape.E)], dtype=torch.float32)
    cfg = moe.cfg_of(shape)
    idx, w, _ = moe.route(x.to(DEV), wg.to(DEV), b.to(DEV), cfg)
    torch.cuda.synchronize()
    want = [4, 9, 14, 19, 24, 29, 34, 39]   # bias 0.04 at ids = 4 mod 5, lowest ids first
    assert (idx.cpu().numpy() == np.array(want)[None, :]).all()
    np.testing.assert_allclose(w.cpu().numpy(), 2.827 / 8, rtol=1e-6)

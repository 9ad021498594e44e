"""moe_layer_forward end to end against the oracle's MoE layer."""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _parity import assert_close_layer, reconcile_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _layer(shape, inp_cpu=None, seed=0, tokens=None, ex_dev=None, inp_dev=None):
    if inp_cpu is None:
        inp_cpu = S.gen_moe_inputs(shape, seed=seed, device="cpu")
    ex = inp_cpu.experts.to(DEV) if ex_dev is None else ex_dev
    x, wg, b = (inp_cpu.x.to(DEV), inp_cpu.w_gate.to(DEV), inp_cpu.bias.to(DEV))
    y, idx, w = moe.layer_forward(x, wg, b, ex, moe.cfg_of(shape), want_routing=True)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    r = O.route(inp_cpu.x.float().numpy(), inp_cpu.w_gate.float().numpy(), inp_cpu.bias.double().numpy(),
                shape.topk, shape.route_scale)
    use_idx = reconcile_routing(idx.cpu().numpy(), r, shape.topk)
    ref = O.moe_layer(inp_cpu.x, inp_cpu.w_gate, inp_cpu.bias, inp_cpu.experts, shape.topk, shape.route_scale,
                      n_shared=shape.n_shared, tokens=tokens, idx_override=use_idx)
    toks = ref["tokens"]
    return assert_close_layer(y.cpu()[toks], ref["y"][toks], what=shape.name), y, ref


@pytest.mark.parametrize("T", [1, 31, 64, 200])
def test_toy_layer(T):
    shape = S.MoEShape(f"toy_t{T}", T=T, d=1024, E=32, topk=8, H=256)
    _layer(shape, seed=T)


def test_toy_layer_reference_workload():
    _layer(S.TOY, seed=0)


def test_toy_layer_skewed():
    shape = S.MoEShape("toy_skew", T=256, d=1024, E=32, topk=8, H=256, hot_experts=(0, 8, 16, 24), hot_bias=0.5)
    _, y, ref = _layer(shape, seed=3)
    assert ref["counts"][[0, 8, 16, 24]].min() >= 200   # the hot experts take most tokens


def test_y_buffer_reuse_and_repeatability():
    shape = S.TOY
    inp = S.gen_moe_inputs(shape, seed=9, device="cpu")
    ex = inp.experts.to(DEV)
    cfg = moe.cfg_of(shape)
    ws = moe.workspace(cfg, shape.T, DEV)
    y1 = moe.layer_forward(inp.x.to(DEV), inp.w_gate.to(DEV), inp.bias.to(DEV), ex, cfg, ws=ws)
    y2 = moe.layer_forward(inp.x.to(DEV), inp.w_gate.to(DEV), inp.bias.to(DEV), ex, cfg, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "the layer is deterministic"


@pytest.fixture(scope="module")
def kimi_weights():
    shape = S.DECODE
    ex = S.gen_experts(shape.E + shape.n_shared, shape.d, shape.H, seed=0, device=DEV)
    torch.cuda.synchronize()
    return ex


def _kimi(shape, ex_dev, n_tokens, seed=0):
    x = S.gen_x(shape.T, shape.d, seed=seed)
    wg, b = S.gen_router(shape, seed=seed)
    cfg = moe.cfg_of(shape)
    y, idx, w = moe.layer_forward(x.to(DEV), wg.to(DEV), b.to(DEV), ex_dev, cfg, want_routing=True)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    r = O.route(x.float().numpy(), wg.float().numpy(), b.double().numpy(), shape.topk, shape.route_scale)
    use_idx = reconcile_routing(idx.cpu().numpy(), r, shape.topk)
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(shape.T, n_tokens, replace=False))
    # the oracle needs only the experts the sampled tokens use
    need = sorted(set(use_idx[toks].ravel().tolist()) | {shape.E})
    host = S.ExpertWeights(*(torch.zeros((shape.E + 1,) + t.shape[1:], dtype=t.dtype)
                             for t in (ex_dev.w13, ex_dev.w13_s, ex_dev.w2, ex_dev.w2_s)))
    for e in need:
        host.w13[e].copy_(ex_dev.w13[e].cpu()); host.w13_s[e].copy_(ex_dev.w13_s[e].cpu())
        host.w2[e].copy_(ex_dev.w2[e].cpu()); host.w2_s[e].copy_(ex_dev.w2_s[e].cpu())
    ref = O.moe_layer(x, wg, b, host, shape.topk, shape.route_scale, tokens=toks, idx_override=use_idx)
    assert_close_layer(y.cpu()[toks], ref["y"][toks], what=shape.name)
    # permutation-level invariants over all tokens
    np.testing.assert_allclose(w.cpu().numpy().sum(1), shape.route_scale, rtol=1e-5)
    return y, use_idx


def _hot_share(shape, idx):
    return float(np.isin(idx, shape.hot_experts).mean())


def test_kimi_decode_layer_sampled(kimi_weights):
    _kimi(S.DECODE, kimi_weights, n_tokens=4)


def test_kimi_prefill_layer_sampled(kimi_weights):
    _kimi(S.PREFILL, kimi_weights, n_tokens=3, seed=1)


def test_kimi_skewed_layer_sampled(kimi_weights):
    # the skewed batch (T=16384, +0.5 bias on 16 hot experts): the hot experts hold
    # thousands of rows each, so dozens of 128-token tiles share every weight block
    # and the dynamic scheduler hands them out
    y, idx = _kimi(S.SKEWED, kimi_weights, n_tokens=3, seed=2)
    assert torch.isfinite(y.float()).all()
    # the stated +0.5 bias gives the 16 hot experts about nine tenths of the assignments
    assert _hot_share(S.SKEWED, idx) > 0.8


def test_kimi_skewed40_layer_sampled(kimi_weights):
    # the same mechanism at +0.18, the bias that gives the hot experts about 40%
    y, idx = _kimi(S.SKEWED40, kimi_weights, n_tokens=3, seed=3)
    assert torch.isfinite(y.float()).all()
    assert 0.3 < _hot_share(S.SKEWED40, idx) < 0.5

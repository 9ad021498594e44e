"""moe_layer_forward end to end against the oracle's MoE layer at toy sizes (the
full Kimi K2 shapes are in test_gpu_fullsize.py)."""
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


# T = 48 and 49 straddle the switch from the decode kernels (k T / E <= 12 rows per
# routed expert) to the token-major ones at this shape
@pytest.mark.parametrize("T", [1, 31, 48, 49, 64, 200])
def test_toy_layer(T):
    shape = S.MoEShape(f"toy_t{T}", T=T, d=1024, E=32, topk=8, H=256)
    _layer(shape, seed=T)


# several shared experts in the token-major regime (each a group of T rows after the
# routed segments), and one-tile routed experts (T = 100: 25 rows each on average)
# next to experts of a ragged second tile (T = 388: 97 on average)
@pytest.mark.parametrize("T,n_shared", [(100, 2), (100, 4), (388, 1)])
def test_toy_layer_shared_experts(T, n_shared):
    shape = S.MoEShape(f"toy_shared_t{T}_s{n_shared}", T=T, d=1024, E=32, topk=8, H=256, n_shared=n_shared)
    _layer(shape, seed=T + n_shared)


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


@pytest.mark.parametrize("shape", [S.MoEShape("gather_t31", T=31, d=1024, E=32, topk=8, H=256),
                                   S.MoEShape("gather_wide_t200", T=200, d=1024, E=32, topk=8, H=256),
                                   S.MoEShape("gather_wide_t480_s2", T=480, d=512, E=32, topk=8, H=384, n_shared=2),
                                   S.MoEShape("gather_t48_s2", T=48, d=512, E=32, topk=8, H=384, n_shared=2),
                                   S.MoEShape("wide_t100_s2", T=100, d=512, E=32, topk=8, H=384, n_shared=2),
                                   S.MoEShape("gather_t1", T=1, d=256, E=16, topk=4, H=128)])
def test_one_call_layer_equals_the_separate_calls(shape):
    # in the decode regime moe_layer_forward's gate/up kernel gathers each token's
    # codes and scales by sorted_tok instead of reading the permutation's copy; beyond
    # it (T = 200 and 480 here, with some experts on a second, ragged tile) the one
    # call runs the token-major kernels on the copy. Either way the output must equal
    # the chain of separate calls bit for bit
    inp = S.gen_moe_inputs(shape, seed=shape.T + 7, device=DEV)
    cfg = moe.cfg_of(shape)
    y = moe.layer_forward(inp.x, inp.w_gate, inp.bias, inp.experts, cfg)
    idx, w, _ = moe.route(inp.x, inp.w_gate, inp.bias, cfg)
    xq, sx = moe.quant_fp8_1x128(inp.x)
    offs, st, inv, xqp, sxp = moe.permute(idx, xq, sx, cfg)
    o = moe.expert_gemm_fp8(xqp, sxp, offs, inp.experts, cfg, shape.T)
    y_chain = moe.combine(o, w, inv, cfg, shape.T)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert torch.equal(y, y_chain)

"""The one-call layer and block captured in a CUDA graph: every call only enqueues
kernels on the caller's stream (no allocation, no synchronisation, no host read
of device data), so a captured graph replays the whole forward. Replays with new
inputs copied into the captured buffers equal eager calls bit for bit."""
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _capture(fn):
    """Warm up fn on a side stream, then capture it into a CUDA graph."""
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize(DEV)
    return g


# T = 48: decode kernels (the gate/up kernel gathers rows); T = 200: token-major kernels
@pytest.mark.parametrize("T", [48, 200])
def test_layer_forward_replays_in_a_cuda_graph(T):
    shape = S.MoEShape(f"toy_graph_t{T}", T=T, d=1024, E=32, topk=8, H=256)
    cfg = moe.cfg_of(shape)
    inp = S.gen_moe_inputs(shape, seed=T, device=DEV)
    ex, wg, b = inp.experts, inp.w_gate, inp.bias
    x = inp.x.clone()
    ws = moe.workspace(cfg, T, DEV)
    y = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=DEV)
    g = _capture(lambda: moe.layer_forward(x, wg, b, ex, cfg, ws=ws, y=y))
    ws_eager = moe.workspace(cfg, T, DEV)
    for seed in (T + 1, T + 2, T + 3):
        x_new = S.gen_x(T, cfg.d, seed=seed, device=DEV)
        x.copy_(x_new)
        g.replay()
        y_eager = moe.layer_forward(x_new, wg, b, ex, cfg, ws=ws_eager)
        torch.cuda.synchronize(DEV)
        assert torch.equal(y, y_eager), f"replay with inputs of seed {seed}"
    moe.check_device_error(DEV)


def test_block_ffn_forward_replays_in_a_cuda_graph():
    T = 96
    shape = S.MoEShape("toy_graph_block", T=T, d=1024, E=32, topk=8, H=256)
    cfg = moe.cfg_of(shape)
    inp = S.gen_moe_inputs(shape, seed=5, device=DEV)
    ex, wg, b = inp.experts, inp.w_gate, inp.bias
    g_post = S.gen_norm_weight(cfg.d, seed=6, device=DEV, name="post")
    g_next = S.gen_norm_weight(cfg.d, seed=7, device=DEV, name="next")
    h = S.gen_residual(T, cfg.d, seed=8, device=DEV)
    ws = moe.workspace(cfg, T, DEV)
    h_out = torch.empty_like(h)
    x_next = torch.empty_like(h)
    g = _capture(lambda: moe.block_ffn_forward(h, g_post, wg, b, ex, cfg, gamma_next=g_next, ws=ws, h_out=h_out,
                                               x_next=x_next))
    for seed in (11, 12):
        h_new = S.gen_residual(T, cfg.d, seed=seed, device=DEV)
        h.copy_(h_new)
        g.replay()
        h_ref, x_ref = moe.block_ffn_forward(h_new, g_post, wg, b, ex, cfg, gamma_next=g_next)
        torch.cuda.synchronize(DEV)
        assert torch.equal(h_out, h_ref) and torch.equal(x_next, x_ref), f"replay with residual of seed {seed}"
    moe.check_device_error(DEV)


def test_dense_ffn_replays_in_a_cuda_graph():
    T, d, H = 256, 1024, 512
    shape = S.DenseShape("toy_graph_dense", T=T, d=d, H=H)
    inp = S.gen_dense_inputs(shape, seed=3, device=DEV)
    x = inp.x.clone()
    ws = moe.dense_workspace(d, H, T, DEV)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    g = _capture(lambda: moe.dense_swiglu_fp8(x, inp.w13, inp.w13_s, inp.w2, inp.w2_s, ws=ws, y=y))
    for seed in (4, 5):
        x_new = S.gen_x(T, d, seed=seed, device=DEV)
        x.copy_(x_new)
        g.replay()
        y_ref = moe.dense_swiglu_fp8(x_new, inp.w13, inp.w13_s, inp.w2, inp.w2_s)
        torch.cuda.synchronize(DEV)
        assert torch.equal(y, y_ref), f"replay with inputs of seed {seed}"
    moe.check_device_error(DEV)

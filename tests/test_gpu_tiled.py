"""The tiled weight layout (moe_pack_weights_fp8, cfg.w_tiled = 1): the packing
itself, bit-exact against its definition, and every expert GEMM kind reading the
tiled weights: outputs equal, bit for bit, those from the row-major weights (which
the other GPU tests pin to the oracle); only the addresses of the weight loads
differ."""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _tiled(ex):
    return S.ExpertWeights(moe.pack_weights_fp8(ex.w13), ex.w13_s, moe.pack_weights_fp8(ex.w2), ex.w2_s)


@pytest.mark.parametrize("groups,rows,cols", [(1, 128, 128), (3, 256, 384), (2, 384, 7168), (5, 2048, 128)])
def test_pack_is_the_tile_transpose(groups, rows, cols):
    g = torch.Generator(device=DEV).manual_seed(rows + cols)
    w = torch.randint(0, 256, (groups, rows, cols), dtype=torch.uint8, device=DEV, generator=g)
    t = moe.pack_weights_fp8(w)
    torch.cuda.synchronize()
    ref = w.view(groups, rows // 128, 128, cols // 128, 128).permute(0, 1, 3, 2, 4).contiguous()
    assert torch.equal(t.view(-1), ref.view(-1))
    # element (g, r, c) sits at tile (g, r // 128, c // 128), offset (r % 128, c % 128)
    gi, r, c = groups - 1, rows - 1, cols - 1
    flat = ((gi * (rows // 128) + r // 128) * (cols // 128) + c // 128) * 16384 + (r % 128) * 128 + c % 128
    assert int(t.view(-1)[flat]) == int(w[gi, r, c])


def test_pack_rejects_bad_shapes_and_overlap():
    # a buffer twice the packed size, so that even the overlapping destination lies
    # inside the allocation
    w = torch.zeros((4, 256, 256), dtype=torch.uint8, device=DEV)
    L = moe.load()
    import ctypes
    st = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    p = ctypes.c_void_p(w.data_ptr())
    assert L.moe_pack_weights_fp8(p, 2, 200, 256, ctypes.c_void_p(w.data_ptr()), st) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_pack_weights_fp8(p, 2, 256, 256, ctypes.c_void_p(w.data_ptr() + 65536), st) == moe.MOE_ERR_ARG
    assert L.moe_pack_weights_fp8(p, 0, 256, 256, p, st) == moe.MOE_OK   # nothing to do


def _routing(shape, seed, hot=()):
    rng = np.random.default_rng(seed)
    T, k, E = shape.T, shape.topk, shape.E
    if hot:
        p = np.full(E, 0.1 / (E - len(hot)))
        p[list(hot)] = 0.9 / len(hot)
        return np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)


# decode kinds (swap-AB, paired and single down blocks), token-major kinds (256-row
# items, the K-pair one-block down kernel for d/128 odd), ragged and multi-tile groups
@pytest.mark.parametrize("shape,hot", [
    (S.MoEShape("t_toy37", T=37, d=1024, E=32, topk=8, H=256), ()),
    (S.MoEShape("t_odd_d8", T=8, d=384, E=16, topk=4, H=256), ()),
    (S.MoEShape("t_tiles400", T=400, d=512, E=32, topk=8, H=384), ()),
    (S.MoEShape("t_odd_wide", T=400, d=384, E=32, topk=8, H=384), ()),
    (S.MoEShape("t_pair_odd_d", T=600, d=384, E=32, topk=8, H=384), ()),
    (S.MoEShape("t_wide_k", T=48, d=2048, E=16, topk=4, H=640), ()),
    (S.MoEShape("t_skew", T=700, d=256, E=16, topk=4, H=256, n_shared=2), (0, 5, 9, 12)),
])
def test_expert_gemm_tiled_equals_row_major(shape, hot):
    inp = S.gen_moe_inputs(shape, seed=shape.T, device=DEV)
    ex, ext = inp.experts, _tiled(inp.experts)
    cfg, cfgt = moe.cfg_of(shape), moe.cfg_of(shape, w_tiled=True)
    idx = torch.from_numpy(_routing(shape, shape.T, hot)).to(DEV)
    xq, sx = moe.quant_fp8_1x128(inp.x)
    offs, _, _, xqp, sxp = moe.permute(idx, xq, sx, cfg)
    o = moe.expert_gemm_fp8(xqp, sxp, offs, ex, cfg, shape.T)
    ot = moe.expert_gemm_fp8(xqp, sxp, offs, ext, cfgt, shape.T)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert torch.equal(o, ot)


@pytest.mark.parametrize("T,n_shared", [(1, 1), (31, 1), (48, 2), (49, 1), (200, 1), (100, 4)])
def test_layer_tiled_equals_row_major(T, n_shared):
    shape = S.MoEShape(f"t_layer{T}", T=T, d=1024, E=32, topk=8, H=256, n_shared=n_shared)
    inp = S.gen_moe_inputs(shape, seed=T + 11, device=DEV)
    y = moe.layer_forward(inp.x, inp.w_gate, inp.bias, inp.experts, moe.cfg_of(shape))
    yt = moe.layer_forward(inp.x, inp.w_gate, inp.bias, _tiled(inp.experts), moe.cfg_of(shape, w_tiled=True))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert torch.equal(y, yt)


# few groups against 152 CTAs: the decode GEMMs' first-round prefetch guesses items of
# groups that do not exist and must skip them; one 128-row block per group
@pytest.mark.parametrize("E,k,n_sh,H,d,T", [(8, 2, 0, 128, 256, 3), (4, 4, 1, 128, 384, 5), (16, 8, 2, 384, 256, 2)])
def test_layer_tiled_few_groups(E, k, n_sh, H, d, T):
    shape = S.MoEShape(f"t_few{E}", T=T, d=d, E=E, topk=k, H=H, n_shared=n_sh)
    inp = S.gen_moe_inputs(shape, seed=E + T, device=DEV)
    y = moe.layer_forward(inp.x, inp.w_gate, inp.bias, inp.experts, moe.cfg_of(shape))
    yt = moe.layer_forward(inp.x, inp.w_gate, inp.bias, _tiled(inp.experts), moe.cfg_of(shape, w_tiled=True))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert torch.equal(y, yt)


def test_block_tiled_equals_row_major():
    shape = S.MoEShape("t_block", T=96, d=1024, E=32, topk=8, H=256)
    inp = S.gen_moe_inputs(shape, seed=5, device=DEV)
    h = S.gen_residual(shape.T, shape.d, seed=6, device=DEV)
    g1 = S.gen_norm_weight(shape.d, seed=7, device=DEV, name="post")
    g2 = S.gen_norm_weight(shape.d, seed=8, device=DEV, name="next")
    a = moe.block_ffn_forward(h, g1, inp.w_gate, inp.bias, inp.experts, moe.cfg_of(shape), gamma_next=g2)
    b = moe.block_ffn_forward(h, g1, inp.w_gate, inp.bias, _tiled(inp.experts), moe.cfg_of(shape, w_tiled=True),
                              gamma_next=g2)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bad_layout_flag_is_rejected():
    shape = S.MoEShape("t_flag", T=4, d=256, E=16, topk=4, H=128)
    cfg = moe.cfg_of(shape)
    cfg.w_tiled = 2
    assert moe.workspace_bytes(cfg, 4) == 0
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device=DEV)
    wg = torch.zeros((16, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(moe.MoeError):
        moe.route(x, wg, torch.zeros(16, device=DEV), cfg, ws=torch.empty(1 << 20, dtype=torch.uint8, device=DEV))

"""No call writes past its outputs: every output buffer (and the workspace) is
followed by a 4 KB region filled with a pattern, checked after each call. The
calls run through the C ABI at toy sizes with the caller's own buffers."""
import ctypes

import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CANARY = 4096
PATTERN = 0xA5


class Canaried:
    """A device buffer of `shape` and `dtype` followed by CANARY pattern bytes."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((n + CANARY,), PATTERN, dtype=torch.uint8, device=DEV)
        self.t = self.raw[:n].view(dtype).view(*shape)
        self.n = n

    @property
    def p(self):
        return ctypes.c_void_p(self.raw.data_ptr())

    def intact(self):
        return bool((self.raw[self.n:] == PATTERN).all())


def _st():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def _ok(rc):
    if rc != 0:
        raise RuntimeError(moe.load().moe_last_error_string().decode())


@pytest.mark.parametrize("shape", [S.TOY, S.MoEShape("canary_wide", T=300, d=512, E=16, topk=4, H=256)])
def test_no_call_writes_past_its_outputs(shape):
    L = moe.load()
    inp = S.gen_moe_inputs(shape, seed=1, device=DEV)
    ex = inp.experts
    cfg = moe.cfg_of(shape)
    cref = ctypes.byref(cfg)
    T, d, k, E, H = shape.T, shape.d, shape.topk, shape.E, shape.H
    R = (k + shape.n_shared) * T
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    nws = L.moe_workspace_bytes(cref, T)
    ws = Canaried((nws,), torch.uint8)
    idx, w, scores = Canaried((T, k), torch.int32), Canaried((T, k), torch.float32), Canaried((T, E), torch.float32)
    _ok(L.moe_route(P(inp.x), P(inp.w_gate), P(inp.bias), cref, T, idx.p, w.p, scores.p, ws.p, nws, _st()))
    xq, sx = Canaried((T, d), torch.uint8), Canaried((T, d // 128), torch.float32)
    _ok(L.moe_quant_fp8_1x128(P(inp.x), 1, T, d, xq.p, sx.p, 0, _st()))
    offs, st, inv = Canaried((E + 1,), torch.int32), Canaried((T * k,), torch.int32), Canaried((T, k), torch.int32)
    xqp, sxp = Canaried((R, d), torch.uint8), Canaried((d // 128, R), torch.float32)
    _ok(L.moe_permute(idx.p, xq.p, sx.p, cref, T, offs.p, st.p, inv.p, xqp.p, sxp.p, ws.p, nws, _st()))
    offs2, st2, inv2 = Canaried((E + 1,), torch.int32), Canaried((T * k,), torch.int32), Canaried((T, k), torch.int32)
    xqp2, sxp2 = Canaried((R, d), torch.uint8), Canaried((d // 128, R), torch.float32)
    _ok(L.moe_permute_noalloc(idx.p, xq.p, sx.p, cref, T, offs2.p, st2.p, inv2.p, xqp2.p, sxp2.p, _st()))
    hq, hs = Canaried((R, H), torch.uint8), Canaried((H // 128, R), torch.float32)
    _ok(L.moe_expert_gateup_fp8(xqp.p, sxp.p, offs.p, P(ex.w13), P(ex.w13_s), cref, T, hq.p, hs.p, ws.p, nws, _st()))
    o = Canaried((R, d), torch.bfloat16)
    _ok(L.moe_expert_down_fp8(hq.p, hs.p, offs.p, P(ex.w2), P(ex.w2_s), cref, T, o.p, ws.p, nws, _st()))
    o2 = Canaried((R, d), torch.bfloat16)
    _ok(L.moe_expert_gemm_fp8(xqp.p, sxp.p, offs.p, P(ex.w13), P(ex.w13_s), P(ex.w2), P(ex.w2_s), cref, T, o2.p,
                              ws.p, nws, _st()))
    y = Canaried((T, d), torch.bfloat16)
    _ok(L.moe_combine(o.p, w.p, inv.p, cref, T, y.p, _st()))
    gamma = S.gen_norm_weight(d, device=DEV)
    xn, xnq, xns = Canaried((T, d), torch.bfloat16), Canaried((T, d), torch.uint8), Canaried((T, d // 128), torch.float32)
    _ok(L.moe_rmsnorm_quant_fp8(P(inp.x), P(gamma), ctypes.c_float(1e-6), T, d, xn.p, xnq.p, xns.p, 0, _st()))
    h_out, x_next = Canaried((T, d), torch.bfloat16), Canaried((T, d), torch.bfloat16)
    _ok(L.moe_combine_residual_rmsnorm(o.p, w.p, inv.p, cref, T, P(inp.x), P(gamma), ctypes.c_float(1e-6),
                                       h_out.p, x_next.p, _st()))
    y2, idx2, w2 = Canaried((T, d), torch.bfloat16), Canaried((T, k), torch.int32), Canaried((T, k), torch.float32)
    _ok(L.moe_layer_forward(P(inp.x), P(inp.w_gate), P(inp.bias), P(ex.w13), P(ex.w13_s), P(ex.w2), P(ex.w2_s),
                            cref, T, y2.p, idx2.p, w2.p, ws.p, nws, _st()))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    bufs = dict(ws=ws, idx=idx, w=w, scores=scores, xq=xq, sx=sx, offsets=offs, sorted_tok=st, inv_pos=inv,
                xq_perm=xqp, sx_perm=sxp, offsets_na=offs2, sorted_tok_na=st2, inv_pos_na=inv2, xq_perm_na=xqp2,
                sx_perm_na=sxp2, hq=hq, hs=hs, o=o, o_gemm=o2, y=y, rms_y=xn, rms_q=xnq, rms_s=xns, h_out=h_out,
                x_next=x_next, layer_y=y2, layer_idx=idx2, layer_w=w2)
    bad = [name for name, b in bufs.items() if not b.intact()]
    assert not bad, f"writes past the end of {bad}"
    # and the calls computed something: the split path equals the one-call layer
    assert torch.equal(y.t, y2.t) and torch.equal(o.t, o2.t)


def test_dense_no_write_past_outputs():
    L = moe.load()
    T, d, H = 200, 512, 384
    inp = S.gen_dense_inputs(S.DenseShape("canary_dense", T=T, d=d, H=H), seed=2, device=DEV)
    nws = L.dense_swiglu_workspace_bytes(d, H, T)
    ws, y = Canaried((nws,), torch.uint8), Canaried((T, d), torch.bfloat16)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    _ok(L.dense_swiglu_fp8(P(inp.x), P(inp.w13), P(inp.w13_s), P(inp.w2), P(inp.w2_s), d, H, T, y.p, ws.p, nws,
                           _st()))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert ws.intact() and y.intact()

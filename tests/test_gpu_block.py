"""The block pieces next to the layer (RMSNorm + quantisation of the layer input;
combine + residual addition + the next block's RMSNorm) against the oracle."""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _parity import reconcile_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EPS = O.RMS_NORM_EPS


def _ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits)."""
    a = np.maximum(np.abs(v), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _near_bf16(got: np.ndarray, ref: np.ndarray, what: str, ulps: float = 1.0, max_frac: float = 2e-3):
    """got equals ref except in rare elements, which differ by at most `ulps` bf16 ulps:
    fp32 arithmetic on the GPU and fp64 in the oracle can round to different neighbours
    when the exact value lies next to a bf16 rounding boundary."""
    diff = got != ref
    frac = diff.mean()
    assert frac <= max_frac, f"{what}: {frac:.2e} of the elements differ"
    if diff.any():
        assert (np.abs(got - ref)[diff] <= ulps * _ulp_bf16(ref[diff]) * (1 + 1e-9)).all(), f"{what}: beyond {ulps} ulp"
    return diff


@pytest.mark.parametrize("T,d", [(1, 256), (37, 1024), (64, 7168)])
def test_rmsnorm_quant(T, d):
    h = S.gen_residual(T, d, seed=T)
    g = S.gen_norm_weight(d, seed=T)
    y, q, s = moe.rmsnorm_quant_fp8(h.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    y = y.float().cpu().numpy().astype(np.float64)
    q, s = q.cpu().numpy(), s.cpu().numpy()
    y_ref = O.rms_norm(h, g, EPS)
    diff = _near_bf16(y, y_ref, "y")
    # the codes are the quantiser's on the GPU's own bf16 y ...
    q2, s2 = moe.quant_fp8_1x128(torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).to(DEV))
    np.testing.assert_array_equal(q, q2.cpu().numpy())
    np.testing.assert_array_equal(s, s2.cpu().numpy())
    # ... and the oracle's on every 128-group whose y values all agree
    qr, sr = O.quantize_1x128(y_ref.astype(np.float32))
    same = ~diff.reshape(T, d // 128, 128).any(axis=2)
    np.testing.assert_array_equal(s[same], sr[same])
    np.testing.assert_array_equal(q.reshape(T, d // 128, 128)[same], qr.reshape(T, d // 128, 128)[same])
    # y not written, transposed scales: the same codes
    y_none, q3, s3 = moe.rmsnorm_quant_fp8(h.to(DEV), g.to(DEV), write_y=False, s_transposed=True)
    assert y_none is None
    np.testing.assert_array_equal(q3.cpu().numpy(), q)
    np.testing.assert_array_equal(s3.cpu().numpy(), s.T)


def test_rmsnorm_quant_zero_row_and_empty():
    d = 512
    h = torch.zeros((2, d), dtype=torch.bfloat16)
    h[1] = S.gen_residual(1, d, seed=7)[0]
    g = S.gen_norm_weight(d, seed=7)
    y, q, s = moe.rmsnorm_quant_fp8(h.to(DEV), g.to(DEV))
    assert (y[0].float() == 0).all() and (q[0] == 0).all() and (s[0] == 0).all()
    e = torch.empty((0, d), dtype=torch.bfloat16, device=DEV)
    y0, q0, s0 = moe.rmsnorm_quant_fp8(e, g.to(DEV))
    assert y0.shape == (0, d) and q0.shape == (0, d)


def _combine_case(T, d, E, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    p = O.permute(idx, E)
    R = (k + 1) * T
    o = S.randn((R, d), 0.3, "cpu", seed, "o", dtype=torch.bfloat16)
    w = torch.from_numpy(rng.uniform(0.1, 1.0, (T, k)).astype(np.float32))
    res = S.gen_residual(T, d, seed=seed, std=0.5)
    g = S.gen_norm_weight(d, seed=seed, name="norm_next")
    return idx, p, o, w, res, g


# T > 512 takes the 64-register variant (no batched row loads)
@pytest.mark.parametrize("T,d", [(1, 128), (48, 1024), (33, 7168), (600, 1024)])
def test_combine_residual_rmsnorm(T, d):
    E, k = 16, 4
    idx, p, o, w, res, g = _combine_case(T, d, E, k, seed=T + 1)
    cfg = moe.MoeCfg(d, E, k, 256, 1, 2.827)
    inv = torch.from_numpy(p["inv_pos"].astype(np.int32))
    h_out, x_next = moe.combine_residual_rmsnorm(o.to(DEV), w.to(DEV), inv.to(DEV), cfg, T, res.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    # GPU self-consistency: the same combine as moe_combine, then the bf16 residual add
    y = moe.combine(o.to(DEV), w.to(DEV), inv.to(DEV), cfg, T)
    assert torch.equal(h_out, (res.to(DEV).float() + y.float()).to(torch.bfloat16))
    # and the same RMSNorm as moe_rmsnorm_quant_fp8 on that row
    x2, _, _ = moe.rmsnorm_quant_fp8(h_out, g.to(DEV))
    assert torch.equal(x_next, x2)
    # against the oracle
    of = o.float().numpy().astype(np.float64)
    wf = w.numpy().astype(np.float64)
    y_ref = of[k * T + np.arange(T)] + sum(wf[:, j:j + 1] * of[p["inv_pos"][:, j]] for j in range(k))
    h_ref = O.residual_add(res, y_ref)
    got_h = h_out.float().cpu().numpy().astype(np.float64)
    # one bf16 ulp of y may move the sum by up to that ulp plus one of h
    diff = got_h != h_ref
    assert diff.mean() <= 2e-3
    if diff.any():
        bound = _ulp_bf16(O.round_bf16(y_ref))[diff] + _ulp_bf16(h_ref)[diff]
        assert (np.abs(got_h - h_ref)[diff] <= bound * (1 + 1e-9)).all()
    # the next block's RMSNorm, given the same h: the oracle's rms_norm of the GPU's own
    # h_out (an h that differs by one ulp can move x by more than two ulps of x where
    # the product crosses a binade, so the stages are checked one at a time)
    x_ref = O.rms_norm(got_h, g, EPS)
    _near_bf16(x_next.float().cpu().numpy().astype(np.float64), x_ref, "x_next", ulps=1.0)
    # without the norm: the same h, no x
    h2, none = moe.combine_residual_rmsnorm(o.to(DEV), w.to(DEV), inv.to(DEV), cfg, T, res.to(DEV))
    assert none is None
    assert torch.equal(h2, h_out)


def test_block_ffn_toy():
    # the FFN half of a MoE block through the library's calls, against the oracle's
    # moe_block_ffn: x = RMSNorm_post(h), the layer, h + y, RMSNorm_next
    shape = S.TOY
    inp = S.gen_moe_inputs(shape, seed=11)
    h = S.gen_residual(shape.T, shape.d, seed=11, std=0.05)
    g_post = S.gen_norm_weight(shape.d, seed=11, name="norm_post")
    g_next = S.gen_norm_weight(shape.d, seed=11, name="norm_next")
    cfg = moe.cfg_of(shape)
    ex = inp.experts.to(DEV)
    x, xq, sx = moe.rmsnorm_quant_fp8(h.to(DEV), g_post.to(DEV))
    idx, w, _ = moe.route(x, inp.w_gate.to(DEV), inp.bias.to(DEV), cfg)
    offs, st, inv, xqp, sxp = moe.permute(idx, xq, sx, cfg)
    o = moe.expert_gemm_fp8(xqp, sxp, offs, ex, cfg, shape.T)
    h_next, x_next = moe.combine_residual_rmsnorm(o, w, inv, cfg, shape.T, h.to(DEV), g_next.to(DEV))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    x_ref = O.rms_norm(h, g_post, EPS).astype(np.float32)
    r = O.route(x_ref, inp.w_gate.float().numpy(), inp.bias.double().numpy(), shape.topk, shape.route_scale)
    use_idx = reconcile_routing(idx.cpu().numpy(), r, shape.topk)
    ref = O.moe_block_ffn(h, g_post, inp.w_gate, inp.bias, inp.experts, shape.topk, shape.route_scale,
                          gamma_next=g_next, idx_override=use_idx)
    # both sides are bf16 numbers: the layer tolerance on the FFN output y (2e-2 of its
    # RMS), plus two bf16 ulps of the value for the roundings around the addition
    y_rms = np.sqrt((ref["y"] ** 2).mean())
    _close_bf16(h_next.float().cpu().numpy(), ref["h_next"], 2e-2 * y_rms, "h_next")
    x_rms = np.sqrt((ref["x_next"] ** 2).mean())
    _close_bf16(x_next.float().cpu().numpy(), ref["x_next"], 2e-2 * x_rms, "x_next")


def _close_bf16(got, ref, abs_tol, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = abs_tol + 2.0 * _ulp_bf16(ref)
    assert (err <= bound).all(), f"{what}: max excess {(err - bound).max():.3e}"
    assert err.mean() / np.abs(ref).mean() <= 5e-3, f"{what}: mean relative error {err.mean() / np.abs(ref).mean():.2e}"


def _split_chain(h, g_post, wg, b, ex, cfg, T, g_next):
    """The block's FFN half through the separate calls."""
    x, xq, sx = moe.rmsnorm_quant_fp8(h, g_post)
    idx, w, _ = moe.route(x, wg, b, cfg)
    offs, st, inv, xqp, sxp = moe.permute(idx, xq, sx, cfg)
    o = moe.expert_gemm_fp8(xqp, sxp, offs, ex, cfg, T)
    h_next, x_next = moe.combine_residual_rmsnorm(o, w, inv, cfg, T, h, g_next)
    return h_next, x_next, idx


def test_block_ffn_one_call_toy():
    # moe_block_ffn_forward: the same bits as the chain of separate calls (its
    # pieces are those calls' kernels, with the RMSNorm pass's codes feeding the
    # permutation), and the oracle's moe_block_ffn within the tolerances above
    shape = S.TOY
    inp = S.gen_moe_inputs(shape, seed=12)
    h = S.gen_residual(shape.T, shape.d, seed=12, std=0.05)
    g_post = S.gen_norm_weight(shape.d, seed=12, name="norm_post")
    g_next = S.gen_norm_weight(shape.d, seed=12, name="norm_next")
    cfg = moe.cfg_of(shape)
    ex = inp.experts.to(DEV)
    hd, gp, gn, wg, b = (t.to(DEV) for t in (h, g_post, g_next, inp.w_gate, inp.bias))
    h_next, x_next, idx, w = moe.block_ffn_forward(hd, gp, wg, b, ex, cfg, gamma_next=gn, want_routing=True)
    h_only, none = moe.block_ffn_forward(hd, gp, wg, b, ex, cfg)
    h_ref_chain, x_ref_chain, idx_chain = _split_chain(hd, gp, wg, b, ex, cfg, shape.T, gn)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert moe.last_launch_count() >= 1 and none is None
    assert torch.equal(idx, idx_chain)
    assert torch.equal(h_next, h_ref_chain) and torch.equal(x_next, x_ref_chain) and torch.equal(h_only, h_next)
    x_ref = O.rms_norm(h, g_post, EPS).astype(np.float32)
    r = O.route(x_ref, inp.w_gate.float().numpy(), inp.bias.double().numpy(), shape.topk, shape.route_scale)
    use_idx = reconcile_routing(idx.cpu().numpy(), r, shape.topk)
    ref = O.moe_block_ffn(h, g_post, inp.w_gate, inp.bias, inp.experts, shape.topk, shape.route_scale,
                          gamma_next=g_next, idx_override=use_idx)
    y_rms = np.sqrt((ref["y"] ** 2).mean())
    _close_bf16(h_next.float().cpu().numpy(), ref["h_next"], 2e-2 * y_rms, "h_next")
    x_rms = np.sqrt((ref["x_next"] ** 2).mean())
    _close_bf16(x_next.float().cpu().numpy(), ref["x_next"], 2e-2 * x_rms, "x_next")


def test_block_ffn_one_call_kimi_decode():
    # the Kimi K2 decode batch (T=256, d=7168, 384 experts): the one call equals the
    # chain of separate calls bit for bit, and the oracle on three tokens
    shape = S.DECODE
    T, d = shape.T, shape.d
    ex = S.gen_experts(shape.E + 1, d, shape.H, seed=0, device=DEV)
    wg, b = S.gen_router(shape, seed=4, device=DEV)
    h = S.gen_residual(T, d, seed=4, std=1.0, device=DEV)
    g_post = S.gen_norm_weight(d, seed=4, name="norm_post", device=DEV)
    g_next = S.gen_norm_weight(d, seed=4, name="norm_next", device=DEV)
    cfg = moe.cfg_of(shape)
    h_next, x_next, idx, w = moe.block_ffn_forward(h, g_post, wg, b, ex, cfg, gamma_next=g_next, want_routing=True)
    h_chain, x_chain, idx_chain = _split_chain(h, g_post, wg, b, ex, cfg, T, g_next)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert torch.equal(idx, idx_chain) and torch.equal(h_next, h_chain) and torch.equal(x_next, x_chain)
    hc = h.cpu()
    x_ref = O.rms_norm(hc, g_post.cpu(), EPS).astype(np.float32)
    r = O.route(x_ref, wg.cpu().float().numpy(), b.cpu().double().numpy(), shape.topk, shape.route_scale)
    use_idx = reconcile_routing(idx.cpu().numpy(), r, shape.topk)
    toks = [0, 97, T - 1]
    need = sorted(set(use_idx[toks].ravel().tolist()) | {shape.E})
    host = S.ExpertWeights(*(torch.zeros((shape.E + 1,) + t.shape[1:], dtype=t.dtype)
                             for t in (ex.w13, ex.w13_s, ex.w2, ex.w2_s)))
    for e in need:
        host.w13[e].copy_(ex.w13[e].cpu()); host.w13_s[e].copy_(ex.w13_s[e].cpu())
        host.w2[e].copy_(ex.w2[e].cpu()); host.w2_s[e].copy_(ex.w2_s[e].cpu())
    ref = O.moe_block_ffn(hc, g_post.cpu(), wg.cpu(), b.cpu(), host, shape.topk, shape.route_scale,
                          gamma_next=g_next.cpu(), tokens=toks, idx_override=use_idx)
    y_rms = np.sqrt((ref["y"][toks] ** 2).mean())
    _close_bf16(h_next.float().cpu().numpy()[toks], ref["h_next"][toks], 2e-2 * y_rms, "h_next")
    x_rms = np.sqrt((ref["x_next"][toks] ** 2).mean())
    _close_bf16(x_next.float().cpu().numpy()[toks], ref["x_next"][toks], 2e-2 * x_rms, "x_next")

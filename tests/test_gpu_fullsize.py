"""Parity at the full Kimi K2 shapes (d=7168, 384 routed experts + 1 shared, top-8,
hidden 2048; the dense FFN with hidden 18432), on the bench's launch configuration.

For each MoE batch (decode T=256, prefill T=4096, skewed and skewed40 T=16384):
- routing and permutation over all T tokens against the oracle (near-tie rule);
- the expert GEMMs' outputs o (moe_expert_gemm_fp8) against the oracle's SwiGLU
  expert on sampled rows: every hot expert with one row from each of its 128-token
  tiles, 64 more touched routed experts, the shared expert; each sampled segment's
  first and last row. An output of o may also differ by what the h codes next to an
  e4m3 rounding midpoint change when they take the neighbouring code (h depends on
  the order of its fp32 sums): the bound adds, per output, the sum over those
  features of one e4m3 step times the group scale times |w2|;
- the layer output y (moe_layer_forward) on 32 tokens including 0 and T-1.

The oracle runs one job per expert (its weights decoded once) in a spawned process
pool; the layer's expected rows are the scaled sum of those expert outputs, an
assembly checked against the oracle's own moe_layer on two tokens.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _oracle_pool import swiglu_jobs
from _parity import assert_close_layer, reconcile_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
N_EXPERTS = 64
N_TOKENS = 32
TILE = 128


@pytest.fixture(scope="module")
def kimi_weights():
    shape = S.DECODE
    ex = S.gen_experts(shape.E + shape.n_shared, shape.d, shape.H, seed=0, device=DEV)
    torch.cuda.synchronize()
    return ex


def _expert_arrays(ex, e):
    return (ex.w13[e, 0].cpu().numpy(), ex.w13_s[e, 0].cpu().numpy(), ex.w13[e, 1].cpu().numpy(),
            ex.w13_s[e, 1].cpu().numpy(), ex.w2[e].cpu().numpy(), ex.w2_s[e].cpu().numpy())


def _positions(lo, hi, rng):
    """Positions of a segment [lo, hi) to compare: its first and last row and one
    row of each 128-row tile."""
    n = hi - lo
    pos = {lo, hi - 1}
    for t0 in range(0, n, TILE):
        pos.add(lo + t0 + int(rng.integers(0, min(TILE, n - t0))))
    return sorted(pos)


def _check_workload(shape, ex, seed, pin_layer=False):
    T, d, k, E = shape.T, shape.d, shape.topk, shape.E
    rng = np.random.default_rng(seed)
    x = S.gen_x(T, d, seed=seed)
    wg, b = S.gen_router(shape, seed=seed)
    cfg = moe.cfg_of(shape)
    xd, wgd, bd = x.to(DEV), wg.to(DEV), b.to(DEV)
    # GPU: the split calls (routing, permutation, expert outputs) and the one-call layer
    idx, w, _ = moe.route(xd, wgd, bd, cfg)
    xq, sx = moe.quant_fp8_1x128(xd)
    offsets, sorted_tok, inv_pos, xq_perm, sx_perm = moe.permute(idx, xq, sx, cfg)
    o = moe.expert_gemm_fp8(xq_perm, sx_perm, offsets, ex, cfg, T)
    y = moe.layer_forward(xd, wgd, bd, ex, cfg)
    y_chain = moe.combine(o, w, inv_pos, cfg, T)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    # the one-call layer (at decode: activation rows gathered by the gate/up kernel)
    # and the chain of separate calls (the permutation's copy) give the same bits
    assert torch.equal(y, y_chain)
    # the one-pass quantise + permute call: the same outputs as the two calls
    fused = moe.quant_permute_fp8(idx, xd, cfg)
    torch.cuda.synchronize()
    for a, f in zip((offsets, sorted_tok, inv_pos, xq_perm, sx_perm), fused):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                           f.view(torch.int32) if f.dtype == torch.float32 else f)
    del fused

    # routing and permutation of all tokens
    xf = x.float().numpy()
    r = O.route(xf, wg.float().numpy(), b.double().numpy(), k, shape.route_scale)
    use_idx = reconcile_routing(idx.cpu().numpy(), r, k)
    p = O.permute(use_idx, E)
    assert np.array_equal(offsets.cpu().numpy(), p["offsets"])
    assert np.array_equal(sorted_tok.cpu().numpy(), p["sorted_tok"])
    assert np.array_equal(inv_pos.cpu().numpy(), p["inv_pos"])
    sel = np.take_along_axis(r["scores"], use_idx, axis=1)
    w_ref = sel / sel.sum(axis=1, keepdims=True) * shape.route_scale
    offs, st = p["offsets"], p["sorted_tok"]

    # rows to compare per expert: token ids, and the positions of o they sit at
    counts = np.diff(offs)
    touched = np.nonzero(counts > 0)[0]
    hot = [e for e in shape.hot_experts if counts[e] > 0]
    others = [e for e in touched if e not in set(hot)]
    sampled = sorted(set(hot) | set(rng.choice(others, min(N_EXPERTS, len(others)), replace=False).tolist()))
    want = {}   # expert -> {token: position in o}
    for e in sampled:
        for pos in _positions(offs[e], offs[e + 1], rng):
            want.setdefault(e, {})[int(st[pos])] = pos
    for t in _positions(0, T, rng):   # the shared expert's rows k*T + t
        want.setdefault(E, {})[t] = k * T + t
    layer_toks = sorted({0, T - 1} | set(rng.choice(np.arange(1, T - 1), N_TOKENS - 2, replace=False).tolist()))
    for t in layer_toks:
        for j in range(k):
            e = int(use_idx[t, j])
            want.setdefault(e, {})[t] = int(np.nonzero(st[offs[e]:offs[e + 1]] == t)[0][0]) + offs[e]
        want.setdefault(E, {})[t] = k * T + t
    toks_of = {e: np.array(sorted(m)) for e, m in want.items()}
    # the oracle's 1x128 quantisation of the rows used (a per-row operation)
    used = np.array(sorted(set(np.concatenate(list(toks_of.values())).tolist())))
    xq_o, xs_o = O.quantize_1x128(xf[used])
    row_of = {int(t): i for i, t in enumerate(used)}

    def make_job(e):
        sub = [row_of[int(t)] for t in toks_of[e]]
        return (xq_o[sub], xs_o[sub]) + _expert_arrays(ex, e)

    res = swiglu_jobs(sorted(toks_of), make_job, flips=True)
    outs = {e: v[0] for e, v in res.items()}
    o_gpu = o.float().cpu().numpy()

    # the expert GEMMs on every sampled expert's rows (and those of the layer tokens);
    # an output may also move by what h codes next to a rounding midpoint change
    for e in sorted(toks_of):
        tk = toks_of[e]
        rows = np.array([want[e][t] for t in tk])
        assert_close_layer(o_gpu[rows], outs[e], what=f"{shape.name} expert {e} ({len(rows)} rows)",
                           extra_allow=res[e][1])

    # the layer output: shared expert plus the routed experts scaled by the oracle's weights
    def ref_row(t):
        acc = np.zeros(d)
        for j in range(k):
            e = int(use_idx[t, j])
            acc += w_ref[t, j] * outs[e][np.searchsorted(toks_of[e], t)]
        return acc + outs[E][np.searchsorted(toks_of[E], t)]

    y_ref = np.stack([ref_row(t) for t in layer_toks])
    if pin_layer:
        # the assembly above is the oracle's layer: compare with moe_layer on two tokens
        two = [layer_toks[0], layer_toks[-1]]
        need = sorted(set(use_idx[two].ravel().tolist()) | {E})
        host = S.ExpertWeights(*(torch.zeros((E + 1,) + t.shape[1:], dtype=t.dtype)
                                 for t in (ex.w13, ex.w13_s, ex.w2, ex.w2_s)))
        for e in need:
            host.w13[e].copy_(ex.w13[e].cpu()); host.w13_s[e].copy_(ex.w13_s[e].cpu())
            host.w2[e].copy_(ex.w2[e].cpu()); host.w2_s[e].copy_(ex.w2_s[e].cpu())
        ref2 = O.moe_layer(x, wg, b, host, k, shape.route_scale, tokens=two, idx_override=use_idx)["y"][two]
        np.testing.assert_allclose(y_ref[[0, -1]], ref2, rtol=1e-12, atol=1e-12)
    assert_close_layer(y.cpu()[layer_toks], y_ref, what=f"{shape.name} layer ({len(layer_toks)} tokens)")
    return counts, use_idx


def test_fullsize_decode(kimi_weights):
    _check_workload(S.DECODE, kimi_weights, seed=0, pin_layer=True)


def test_fullsize_prefill(kimi_weights):
    _check_workload(S.PREFILL, kimi_weights, seed=1)


def test_fullsize_skewed(kimi_weights):
    # +0.5 on 16 hot experts: thousands of rows each, dozens of token tiles per
    # weight block, handed out by the dynamic scheduler among the cold experts' items
    counts, idx = _check_workload(S.SKEWED, kimi_weights, seed=2)
    assert float(np.isin(idx, S.SKEWED.hot_experts).mean()) > 0.8


def test_fullsize_skewed40(kimi_weights):
    counts, idx = _check_workload(S.SKEWED40, kimi_weights, seed=3)
    assert 0.3 < float(np.isin(idx, S.SKEWED40.hot_experts).mean()) < 0.5


@pytest.mark.parametrize("shape", [S.DECODE, S.PREFILL, S.SKEWED], ids=lambda s: s.name)
def test_fullsize_tiled_weights_equal_row_major(kimi_weights, shape):
    # the same layer with the weights in the tiled layout (moe_pack_weights_fp8):
    # every GEMM kind of the workload reads its tiles, and y is the same bit for bit
    x = S.gen_x(shape.T, shape.d, seed=5).to(DEV)
    wg, b = (t.to(DEV) for t in S.gen_router(shape, seed=5))
    ex = kimi_weights
    ext = S.ExpertWeights(moe.pack_weights_fp8(ex.w13), ex.w13_s, moe.pack_weights_fp8(ex.w2), ex.w2_s)
    y = moe.layer_forward(x, wg, b, ex, moe.cfg_of(shape))
    yt = moe.layer_forward(x, wg, b, ext, moe.cfg_of(shape, w_tiled=True))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    assert torch.equal(y, yt)
    del ext


def test_fullsize_dense():
    # the first block's dense FFN, T=8192: 64 tokens including the two sides of the
    # first 128-token tile boundary and the last token
    shape = S.DENSE
    inp = S.gen_dense_inputs(shape, seed=0, device=DEV)
    y = moe.dense_swiglu_fp8(inp.x, inp.w13, inp.w13_s, inp.w2, inp.w2_s)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    rng = np.random.default_rng(5)
    fixed = [0, 127, 128, shape.T - 1]
    rest = rng.choice(np.setdiff1d(np.arange(shape.T), fixed), 60, replace=False)
    toks = np.array(sorted(set(fixed) | set(rest.tolist())))
    assert len(toks) == 64
    ref, _ = O.dense_swiglu(inp.x.cpu()[toks], inp.w13.cpu(), inp.w13_s.cpu(), inp.w2.cpu(), inp.w2_s.cpu())
    assert_close_layer(y.cpu()[toks], ref, what="dense kimi")

"""moe_expert_gemm_fp8 (grouped tcgen05 FP8 GEMMs) against the oracle's SwiGLU experts."""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _parity import assert_close_layer

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(shape, seed, n_check=None, hot=()):
    inp = S.gen_moe_inputs(shape, seed=seed, device="cpu")
    cfg = moe.cfg_of(shape)
    T, k = shape.T, shape.topk
    rng = np.random.default_rng(seed)
    if hot:
        # each token takes the hot experts with probability 0.9 each, then cold ones
        p = np.full(shape.E, 0.1 / (shape.E - len(hot)))
        p[list(hot)] = 0.9 / len(hot)
        idx = np.stack([rng.choice(shape.E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        idx = np.stack([rng.choice(shape.E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ex = inp.experts.to(DEV)
    xq, sx = moe.quant_fp8_1x128(inp.x.to(DEV))
    offsets, sorted_tok, inv_pos, xq_perm, sx_perm = moe.permute(torch.from_numpy(idx).to(DEV), xq, sx, cfg)
    o = moe.expert_gemm_fp8(xq_perm, sx_perm, offsets, ex, cfg, T)
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    o = o.float().cpu().numpy()
    xq_c, sx_c = xq.cpu().numpy(), sx.cpu().numpy()
    offs = offsets.cpu().numpy()
    st = sorted_tok.cpu().numpy()
    w13, w13s, w2, w2s = (inp.experts.w13.numpy(), inp.experts.w13_s.numpy(), inp.experts.w2.numpy(),
                          inp.experts.w2_s.numpy())
    groups = [(e, np.arange(offs[e], offs[e + 1]), st[offs[e]:offs[e + 1]]) for e in range(shape.E)]
    groups += [(shape.E + s, k * T + s * T + np.arange(T), np.arange(T)) for s in range(shape.n_shared)]
    checked = 0
    for e, rows, toks in groups:
        if rows.size == 0:
            continue
        if n_check is not None:
            rows, toks = rows[:n_check], toks[:n_check]
        ref, _, _ = O.swiglu_fp8(xq_c[toks], sx_c[toks], w13[e, 0], w13s[e, 0], w13[e, 1], w13s[e, 1], w2[e], w2s[e])
        assert_close_layer(o[rows], ref, what=f"expert {e}")
        checked += rows.size
    return checked


@pytest.mark.parametrize("T", [1, 37, 64])
def test_toy_experts(T):
    shape = S.MoEShape("toy", T=T, d=1024, E=32, topk=8, H=256)
    assert _run(shape, seed=T) == 9 * T


def test_experts_with_several_token_tiles():
    # ~100 rows per routed expert and 400 shared rows: several 128-row token tiles
    shape = S.MoEShape("tiles", T=400, d=512, E=32, topk=8, H=384)
    assert _run(shape, seed=1) == 9 * 400


def test_experts_beyond_128_rows_span_several_token_tiles():
    # 150 rows per routed expert and 600 shared rows: two or more 128-token tiles per
    # expert, the last one ragged; every row is compared
    shape = S.MoEShape("wide_tiles", T=600, d=512, E=32, topk=8, H=256)
    assert _run(shape, seed=3) == 9 * 600


def test_several_tiles_with_odd_down_blocks():
    # 150 rows per routed expert with d = 384: several token tiles per expert, and the
    # down projection (three 128-row output blocks) on the one-block kernel
    shape = S.MoEShape("pair_odd_d", T=600, d=384, E=32, topk=8, H=384)
    assert _run(shape, seed=6) == 9 * 600


def test_skewed_segments_many_tiles_and_few_rows():
    # skewed routing at toy size: four hot experts with about 590 rows each (five
    # 128-token tiles, the last ragged) and cold experts of a few dozen rows
    shape = S.MoEShape("pair_ragged", T=700, d=256, E=16, topk=4, H=256)
    assert _run(shape, seed=7, hot=(0, 5, 9, 12)) == 5 * 700


def test_decode_down_with_odd_block_count():
    # d = 384: three 128-row output blocks, so the decode down GEMM cannot pair them
    shape = S.MoEShape("odd_d", T=8, d=384, E=16, topk=4, H=256)
    assert _run(shape, seed=4) == 5 * 8


def test_wide_k_and_many_blocks():
    shape = S.MoEShape("wide", T=48, d=2048, E=16, topk=4, H=640, n_shared=1)
    _run(shape, seed=2)


def test_wide_tiles_with_odd_block_counts():
    # 100 rows per routed expert (128-token tiles) with d = H = 384: the gate/up items
    # run three K blocks, and the down projection (three 128-row output blocks) takes
    # the one-block token-major kernel, whose last K pair holds a single K block
    shape = S.MoEShape("odd_wide", T=400, d=384, E=32, topk=8, H=384)
    assert _run(shape, seed=5) == 9 * 400

"""The seeded input generator: determinism, shapes and the stated distributions."""
import numpy as np
import torch

import moe_synth as S


def test_deterministic_and_seed_dependent():
    a = S.gen_x(8, 256, seed=0)
    b = S.gen_x(8, 256, seed=0)
    c = S.gen_x(8, 256, seed=1)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert a.dtype == torch.bfloat16


def test_router_and_hot_bias():
    sh = S.MoEShape("t", T=4, d=256, E=64, topk=8, H=128, hot_experts=(0, 8, 16), hot_bias=0.5)
    wg, b = S.gen_router(sh, seed=0)
    assert wg.shape == (64, 256) and wg.dtype == torch.bfloat16
    assert b.dtype == torch.float32
    assert (b[[0, 8, 16]] == 0.5).all()
    rest = torch.ones(64, dtype=torch.bool); rest[[0, 8, 16]] = False
    assert b[rest].abs().max() < 0.06
    assert abs(wg.float().std().item() - 0.02) < 0.002
    assert S.SKEWED.hot_experts == tuple(range(0, 384, 24))


def test_fp8_block_storage():
    w = torch.randn(256, 384) * 0.02
    w[:128, :128] = 0
    q, s = S.fp8_blocks(w)
    assert q.dtype == torch.uint8 and q.shape == (256, 384) and s.shape == (2, 3)
    assert s[0, 0] == 0 and (q[:128, :128] == 0).all()
    blk = w[128:, 128:256]
    assert s[1, 1] == blk.abs().max() / 448
    deq = q.view(torch.float8_e4m3fn).float().view(2, 128, 3, 128) * s[:, None, :, None]
    err = (deq.view(256, 384) - w).abs()
    assert (err <= w.abs() * 2 ** -4 + s.repeat_interleave(128, 0).repeat_interleave(128, 1) * 2 ** -10 + 1e-12).all()
    # no NaN code anywhere
    assert not ((q & 0x7F) == 0x7F).any()


def test_expert_layout():
    ex = S.gen_experts(3, 256, 128, seed=0)
    assert ex.w13.shape == (3, 2, 128, 256) and ex.w13_s.shape == (3, 2, 1, 2)
    assert ex.w2.shape == (3, 256, 128) and ex.w2_s.shape == (3, 2, 1)
    assert not torch.equal(ex.w13[0, 0], ex.w13[0, 1]) and not torch.equal(ex.w13[0], ex.w13[1])

"""moe_permute against the oracle's permutation: bit-exact for ids, positions and copied rows."""
import numpy as np
import pytest
import torch

import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _random_idx(T, E, k, rng):
    return np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)


def _check(idx, E, d=256, S=1):
    T, k = idx.shape
    cfg = moe.MoeCfg(d, E, k, 128, S, 2.827)
    rng = np.random.default_rng(T)
    x = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32))
    xq, sx = moe.quant_fp8_1x128(x.to(DEV))
    offsets, sorted_tok, inv_pos, xq_perm, sx_perm = moe.permute(torch.from_numpy(idx).to(DEV), xq, sx, cfg)
    torch.cuda.synchronize()
    p = O.permute(idx, E)
    np.testing.assert_array_equal(offsets.cpu().numpy(), p["offsets"])
    np.testing.assert_array_equal(sorted_tok.cpu().numpy(), p["sorted_tok"])
    np.testing.assert_array_equal(inv_pos.cpu().numpy(), p["inv_pos"])
    rows = np.concatenate([p["sorted_tok"]] + [np.arange(T)] * S)
    np.testing.assert_array_equal(xq_perm.cpu().numpy(), xq.cpu().numpy()[rows])
    np.testing.assert_array_equal(sx_perm.cpu().numpy(), sx.cpu().numpy()[rows].T)


@pytest.mark.parametrize("T,E,k", [(1, 32, 8), (33, 32, 8), (64, 32, 8), (1000, 384, 8), (4096, 384, 8),
                                   (77, 40, 1), (50, 64, 32),
                                   # eight full 32-token chunks, the most experts, one token into a ninth chunk
                                   (256, 384, 8), (255, 1024, 8), (257, 384, 8)])
def test_random_routing(T, E, k):
    _check(_random_idx(T, E, k, np.random.default_rng(T + E + k)), E)


def test_one_hot_expert_set_and_empty_experts():
    idx = np.tile(np.arange(8, dtype=np.int32)[::-1], (300, 1))   # every token picks 7..0
    _check(idx, 32)


def test_no_shared_and_two_shared():
    idx = _random_idx(70, 32, 8, np.random.default_rng(3))
    _check(idx, 32, S=0)
    _check(idx, 32, S=2)


def test_skewed_counts():
    rng = np.random.default_rng(4)
    T, E, k = 3000, 384, 8
    hot = np.arange(0, 384, 24)
    idx = np.empty((T, k), np.int32)
    for t in range(T):
        h = rng.choice(hot, 6, replace=False)
        rest = rng.choice(np.setdiff1d(np.arange(E), h), 2, replace=False)
        idx[t] = np.concatenate([h, rest])
    _check(idx, E, d=128)


def _check_quant_permute(idx, E, d, S, seed):
    """moe_quant_permute_fp8 on bf16 x: bit for bit the permutation of the
    quantiser's codes, and the oracle's codes of x in the oracle's row order."""
    T, k = idx.shape
    cfg = moe.MoeCfg(d, E, k, 128, S, 2.827)
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(T, d, generator=g) * torch.rand(T, 1, generator=g) * 10).to(torch.bfloat16)
    if T > 2:
        x[1, :128] = 0   # a group with amax = 0
    ti = torch.from_numpy(idx).to(DEV)
    xd = x.to(DEV)
    xq, sx = moe.quant_fp8_1x128(xd)
    ref = moe.permute(ti, xq, sx, cfg)
    got = moe.quant_permute_fp8(ti, xd, cfg)
    torch.cuda.synchronize()
    for name, a, b in zip(("offsets", "sorted_tok", "inv_pos", "xq_perm", "sx_perm"), ref, got):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                           b.view(torch.int32) if b.dtype == torch.float32 else b), name
    qo, so = O.quantize_1x128(x.float().numpy())
    p = O.permute(idx, E)
    rows = np.concatenate([p["sorted_tok"]] + [np.arange(T)] * S)
    np.testing.assert_array_equal(got[3].cpu().numpy(), qo[rows])
    np.testing.assert_array_equal(got[4].cpu().numpy().view(np.int32), so[rows].T.view(np.int32))


@pytest.mark.parametrize("T,E,k,d,S", [(1, 32, 8, 256, 1), (33, 32, 8, 384, 1), (70, 32, 8, 1024, 0),
                                       (70, 32, 8, 1024, 2), (50, 64, 32, 128, 1), (257, 384, 8, 7168, 1),
                                       (31, 40, 1, 16384, 4), (1000, 384, 8, 7168, 1)])
def test_quant_permute_equals_quant_then_permute(T, E, k, d, S):
    _check_quant_permute(_random_idx(T, E, k, np.random.default_rng(T + E + k + d)), E, d, S, seed=T + d)


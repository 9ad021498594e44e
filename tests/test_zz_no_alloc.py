"""moe_permute_noalloc, the permutation for callers that cannot provide scratch
memory (it keeps its scratch in a fixed device array inside the library), must
give exactly what moe_permute gives with a workspace, call after call.

This file is collected last on purpose: a run that stops at the first failure
has then already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from routed_fp8_expert_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32))


@pytest.mark.parametrize("T,E,k,d,S", [(256, 384, 8, 7168, 1), (1000, 64, 8, 1024, 2), (33, 32, 8, 256, 0)])
def test_matches_workspace_permutation_two_calls_in_a_row(T, E, k, d, S):
    cfg = moe.MoeCfg(d, E, k, 128, S, 2.827)
    for call, seed in enumerate((T, T + 1)):          # two calls, different inputs
        idx = _routing(T, E, k, seed).to(DEV)
        x = torch.randn(T, d, generator=torch.Generator().manual_seed(seed)).to(DEV)
        xq, sx = moe.quant_fp8_1x128(x)
        ref = moe.permute(idx, xq, sx, cfg)
        got = moe.permute_noalloc(idx, xq, sx, cfg)
        torch.cuda.synchronize()
        for name, a, b in zip(("offsets", "sorted_tok", "inv_pos", "xq_perm", "sx_perm"), got, ref):
            assert torch.equal(a, b), f"call {call}: {name} differs from moe_permute"


@pytest.mark.parametrize("T,E,k,S", [(8192, 1024, 8, 4), (4096, 1024, 16, 4)])
def test_at_the_scratch_limits_against_the_oracle(T, E, k, S):
    # T * topk = 65,536 assignments (the limit, reached exactly), E = 1024 experts and
    # four shared experts fill the array's regions; the result must be the oracle's
    # permutation, and the permuted rows and scales the gathers it defines
    d = 256
    cfg = moe.MoeCfg(d, E, k, 128, S, 2.827)
    idx = _routing(T, E, k, seed=T + k)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(k)).to(DEV)
    xq, sx = moe.quant_fp8_1x128(x)
    offsets, sorted_tok, inv_pos, xq_perm, sx_perm = moe.permute_noalloc(idx.to(DEV), xq, sx, cfg)
    torch.cuda.synchronize()
    p = O.permute(idx.numpy(), E)
    np.testing.assert_array_equal(offsets.cpu().numpy(), p["offsets"])
    np.testing.assert_array_equal(sorted_tok.cpu().numpy(), p["sorted_tok"])
    np.testing.assert_array_equal(inv_pos.cpu().numpy(), p["inv_pos"])
    src = np.concatenate([p["sorted_tok"]] + [np.arange(T)] * S)     # the row each permuted row copies
    xq_c, sx_c = xq.cpu().numpy(), sx.cpu().numpy()
    np.testing.assert_array_equal(xq_perm.cpu().numpy(), xq_c[src])
    np.testing.assert_array_equal(sx_perm.cpu().numpy(), sx_c[src].T)


def test_rejects_sizes_beyond_the_scratch():
    lib = moe.load()
    cfg = moe.MoeCfg(1024, 384, 8, 256, 1, 2.827)
    fake = ctypes.c_void_p(0x1000)
    st = lib.moe_permute_noalloc(fake, fake, fake, ctypes.byref(cfg), 8193, fake, fake, fake, fake, fake, None)
    assert st == _lib.MOE_ERR_UNSUPPORTED
    assert b"at most 8192 tokens" in lib.moe_last_error_string()
    cfg32 = moe.MoeCfg(1024, 384, 32, 256, 1, 2.827)
    st = lib.moe_permute_noalloc(fake, fake, fake, ctypes.byref(cfg32), 4096, fake, fake, fake, fake, fake, None)
    assert st == _lib.MOE_ERR_UNSUPPORTED
    # just past the assignment limit (T * topk = 7282 * 9 = 65,538; 65,536 is accepted
    # above), and more experts than 1024
    cfg9 = moe.MoeCfg(1024, 384, 9, 256, 1, 2.827)
    st = lib.moe_permute_noalloc(fake, fake, fake, ctypes.byref(cfg9), 7282, fake, fake, fake, fake, fake, None)
    assert st == _lib.MOE_ERR_UNSUPPORTED
    cfg_e = moe.MoeCfg(1024, 1025, 8, 256, 1, 2.827)
    st = lib.moe_permute_noalloc(fake, fake, fake, ctypes.byref(cfg_e), 64, fake, fake, fake, fake, fake, None)
    assert st == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_last_launch_count() == 0

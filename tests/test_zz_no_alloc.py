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

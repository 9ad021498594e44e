"""dense_swiglu_fp8 (the first block's dense FFN) against the oracle."""
import numpy as np
import pytest
import torch

import moe_synth as S
import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O
from _parity import assert_close_layer

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


# (200, 384, 384): three 128-row output blocks, so the down projection takes the
# one-block token-major kernel, whose K-pair boxes end on a half-empty pair
@pytest.mark.parametrize("T,d,H", [(1, 256, 128), (300, 1024, 1536), (129, 2048, 512), (200, 384, 384)])
def test_dense_small(T, d, H):
    inp = S.gen_dense_inputs(S.DenseShape("dense_small", T=T, d=d, H=H), seed=T)
    y = moe.dense_swiglu_fp8(inp.x.to(DEV), inp.w13.to(DEV), inp.w13_s.to(DEV), inp.w2.to(DEV), inp.w2_s.to(DEV))
    torch.cuda.synchronize()
    moe.check_device_error(DEV)
    ref, _ = O.dense_swiglu(inp.x, inp.w13, inp.w13_s, inp.w2, inp.w2_s)
    assert_close_layer(y, ref, what="dense")

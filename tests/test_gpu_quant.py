"""moe_quant_fp8_1x128 on the GPU against the oracle's quantiser: bit-exact."""
import numpy as np
import pytest
import torch

import routed_fp8_expert_gb300 as moe
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(x, transposed=False):
    q, s = moe.quant_fp8_1x128(x.to(DEV), s_transposed=transposed)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(1, 128), (257, 1024), (64, 7168)])
def test_bf16_random_bit_exact(rows, cols):
    g = torch.Generator().manual_seed(rows * cols)
    x = (torch.randn(rows, cols, generator=g) * torch.rand(rows, 1, generator=g) * 10).to(torch.bfloat16)
    q, s = _run(x)
    qo, so = O.quantize_1x128(x.float().numpy())
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))
    qt, st = _run(x, transposed=True)
    np.testing.assert_array_equal(qt, qo)
    np.testing.assert_array_equal(st.T.view(np.uint32), so.view(np.uint32))


def test_fp32_special_groups_bit_exact():
    rows, cols = 8, 512
    x = torch.randn(rows, cols) * 3
    x[0, :128] = 0.0                      # zero group
    x[1, 128:256] = -0.0                  # negative-zero group
    x[2, :128] = 7.5                      # constant group
    x[3, 256:384] = 1e-30                 # tiny values
    x[4, :] = torch.randn(cols) * 1e20    # huge range
    x[5, 5] = -0.0
    x[6, :128] = torch.linspace(-1, 1, 128)
    q, s = _run(x)
    qo, so = O.quantize_1x128(x.numpy())
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_e4m3_rounding_at_every_midpoint():
    # groups whose amax is 448 have scale exactly 1, so the codes are e4m3(x):
    # put every midpoint between adjacent codes, and its fp32 neighbours, in them
    vals = []
    for c in range(0x7E):
        lo, hi = O.e4m3_value(c), O.e4m3_value(c + 1)
        mid = np.float32((lo + hi) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9)), np.float32(lo)]
    vals = np.array(vals, dtype=np.float32)
    vals = np.concatenate([vals, -vals])
    per = 127
    n_groups = (len(vals) + per - 1) // per
    x = np.zeros((n_groups, 128), dtype=np.float32)
    for g in range(n_groups):
        chunk = vals[g * per:(g + 1) * per]
        x[g, :len(chunk)] = chunk
        x[g, 127] = 448.0
    q, s = _run(torch.from_numpy(x))
    qo, so = O.quantize_1x128(x)
    assert (so == 1.0).all()
    np.testing.assert_array_equal(q, qo)

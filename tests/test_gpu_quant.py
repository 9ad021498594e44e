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


# group counts that leave the last warp's run ragged (2,997 and 161,007 groups), the
# second large enough that every warp takes two runs of eight groups
@pytest.mark.parametrize("rows,cols", [(999, 384), (23001, 896)])
@pytest.mark.parametrize("bf16", [True, False])
def test_ragged_group_runs_bit_exact(rows, cols, bf16):
    g = torch.Generator().manual_seed(rows + cols)
    x = torch.randn(rows, cols, generator=g) * torch.rand(rows, 1, generator=g) * 4
    x = x.to(torch.bfloat16) if bf16 else x
    q, s = _run(x, transposed=True)
    qo, so = O.quantize_1x128(x.float().numpy())
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.T.view(np.uint32), so.view(np.uint32))


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


def _division_sweep(amax: np.ndarray) -> np.ndarray:
    """One 128-group per group maximum: entry 0 is amax, entries 1..127 sweep
    twelve binades below it (alternating signs), all bf16 values."""
    j = np.arange(1, 128)
    u = (1.0 + ((j * 37) % 128) / 128.0) / 2.0 * 2.0 ** -(j % 12)    # in (0, 1)
    sign = np.where(j % 2 == 0, 1.0, -1.0)
    g = np.empty((amax.size, 128), np.float64)
    g[:, 0] = amax
    g[:, 1:] = amax[:, None] * u[None, :] * sign[None, :]
    return O.round_bf16(g).astype(np.float32)


def test_quantiser_division_every_bf16_maximum():
    # every positive normal bf16 value is the maximum of one group, so s = amax / 448
    # takes all its values, and each group's codes depend on the correctly rounded
    # x / s of 127 other entries: bit-exact against the oracle's IEEE fp32 division
    e = np.arange(-126, 128)
    m = np.arange(128)
    amax = (np.ldexp(1.0 + m[None, :] / 128.0, e[:, None])).ravel()
    amax = amax[amax < 3.3e38]
    groups = _division_sweep(amax)
    cols = 7168
    pad = (-groups.shape[0]) % (cols // 128)
    groups = np.concatenate([groups, np.zeros((pad, 128), np.float32)])
    x = torch.from_numpy(groups.reshape(-1, cols)).to(torch.bfloat16)
    q, s = _run(x)
    qo, so = O.quantize_1x128(x.float().numpy())
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))
    np.testing.assert_array_equal(q, qo)


def test_quantiser_division_subnormal_scales():
    # group maxima below 448 * 2^-126 give subnormal scales (the quantiser divides
    # directly below scales of 2^-80)
    amax = np.ldexp(1.0 + np.arange(0, 128, 8) / 128.0, -120)
    groups = _division_sweep(amax)
    x = torch.from_numpy(groups.reshape(-1, 2048)).to(torch.bfloat16)
    q, s = _run(x)
    qo, so = O.quantize_1x128(x.float().numpy())
    assert (so < 1.17549435e-38).all()
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))
    np.testing.assert_array_equal(q, qo)


def test_quantiser_division_midpoints_across_scales():
    # scales s = (1 + m/8) 2^k from 2^-85 to 2^100, on both sides of 2^-80, below
    # which the quantiser divides directly: each group's amax is exactly 448 s, and
    # its entries are s times every e4m3 rounding midpoint and the fp32 neighbours
    # of those products, so every code decision sits on or next to a boundary;
    # bit-exact against the oracle's IEEE fp32 division
    mids = np.array([(O.e4m3_value(c) + O.e4m3_value(c + 1)) / 2 for c in range(0x7E)])
    groups = []
    for k in range(-85, 101):
        for m in (0, 3, 5):
            s = np.float32(np.ldexp(1.0 + m / 8.0, k))
            base = (mids * np.float64(s)).astype(np.float32)   # exact: few significant bits
            vals = np.concatenate([base, np.nextafter(base, np.float32(0)), np.nextafter(base, np.float32(np.inf))])
            vals = np.where(np.arange(vals.size) % 2 == 0, vals, -vals).astype(np.float32)
            for i in range(0, vals.size, 127):
                g = np.zeros(128, np.float32)
                chunk = vals[i:i + 127]
                g[:chunk.size] = chunk
                g[127] = np.float32(448.0) * s
                groups.append(g)
    x = np.stack(groups)
    pad = (-x.shape[0]) % 8
    x = np.concatenate([x, np.zeros((pad, 128), np.float32)]).reshape(-1, 1024)
    q, s = _run(torch.from_numpy(x))
    qo, so = O.quantize_1x128(x)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))
    np.testing.assert_array_equal(q, qo)


def _same_codes_up_to_nan_sign(q, qo):
    """Codes equal, except that a NaN code (S.1111.111) may carry either sign: the
    sign of a NaN produced by an invalid operation differs between machines."""
    nan, nan_o = (q & 0x7F) == 0x7F, (qo & 0x7F) == 0x7F
    np.testing.assert_array_equal(nan, nan_o)
    np.testing.assert_array_equal(q[~nan], qo[~nan])


@pytest.mark.parametrize("bf16", [False, True])
def test_nan_and_infinity_groups(bf16):
    # a NaN in a group makes its amax and scale NaN and every quotient NaN; an
    # infinity makes the scale infinite, its own quotient NaN (inf / inf) and the
    # group's finite quotients +-0 (x / inf); other groups are unaffected
    rows, cols = 6, 512
    x = torch.randn(rows, cols, generator=torch.Generator().manual_seed(7)) * 2
    x[0, 3] = float("nan")
    x[1, 130] = float("inf")
    x[2, 260] = float("-inf")
    x[3, 0], x[3, 129] = float("inf"), float("nan")
    x[4, 384:] = float("inf")
    if bf16:
        x = x.to(torch.bfloat16)
    q, s = _run(x)
    qo, so = O.quantize_1x128(x.float().numpy())
    _same_codes_up_to_nan_sign(q, qo)
    np.testing.assert_array_equal(np.isnan(s), np.isnan(so))
    fin = ~np.isnan(so)
    np.testing.assert_array_equal(s[fin], so[fin])
    # the groups with an infinity: scale +inf, finite elements quantise to +-0
    assert np.isinf(s[1, 1]) and (q[1, 128:256][np.arange(128) != 2] & 0x7F == 0).all()
    # groups untouched by the special values are those of the plain quantiser
    assert (q[5] == qo[5]).all() and (s[5] == so[5]).all()

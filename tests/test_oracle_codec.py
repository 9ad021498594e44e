"""Pins for the oracle's e4m3 codec (OCP 8-bit floating point, E4M3 variant)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def test_special_codes():
    # closed-form values of the format: bias 7, 3 mantissa bits, no infinities
    assert O.e4m3_value(0x00) == 0.0
    assert O.e4m3_value(0x01) == 2.0 ** -9                 # smallest subnormal
    assert O.e4m3_value(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert O.e4m3_value(0x08) == 2.0 ** -6                 # smallest normal
    assert O.e4m3_value(0x38) == 1.0
    assert O.e4m3_value(0x40) == 2.0
    assert O.e4m3_value(0x7E) == 448.0                     # largest finite
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))
    assert O.e4m3_value(0xFE) == -448.0
    assert O.e4m3_value(0x80) == 0.0 and np.signbit(O.e4m3_value(0x80))
    # 126 positive finite nonzero values, strictly increasing with the code
    pos = [O.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(pos, pos[1:]))


def test_decode_encode_identity_all_finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    fin = ~np.isnan(vals)
    assert fin.sum() == 254
    np.testing.assert_array_equal(O.e4m3_encode(vals[fin]), codes[fin])


def test_midpoints_round_to_even_code():
    for c in range(0x7E):  # every pair of adjacent positive finite codes
        lo, hi = O.e4m3_value(c), O.e4m3_value(c + 1)
        mid = (lo + hi) / 2
        want = c if c % 2 == 0 else c + 1
        assert O.e4m3_encode(np.array([mid]))[0] == want, hex(c)
        assert O.e4m3_encode(np.array([-mid]))[0] == (want | 0x80)
        # just off the midpoint goes to the nearer code
        eps = (hi - lo) * 1e-3
        assert O.e4m3_encode(np.array([mid - eps]))[0] == c
        assert O.e4m3_encode(np.array([mid + eps]))[0] == c + 1


def test_saturation_and_nan():
    v = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, -1e30, np.nan])
    got = O.e4m3_encode(v)
    assert list(got[:6]) == [0x7E] * 6
    assert got[6] == 0xFE
    assert got[7] == 0x7F


def test_agrees_with_torch_cast_on_clamped_values():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(200_000) * s for s in (1e-3, 0.1, 10, 200)])
    v = np.clip(v, -448, 448).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(v), ref)

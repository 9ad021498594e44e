"""Pins for the 1x128 dynamic activation quantiser (scale = amax / 448, fp32)."""
import numpy as np

from oracle import moe_oracle as O


def test_constant_group_maps_to_max_code():
    a = np.full((3, 256), 5.0, dtype=np.float32)
    a[1, :128] = -7.25
    q, s = O.quantize_1x128(a)
    assert s.dtype == np.float32 and s.shape == (3, 2)
    assert s[0, 0] == np.float32(5.0) / np.float32(448.0)
    assert (q[0] == 0x7E).all()
    assert (q[1, :128] == 0xFE).all()


def test_zero_group():
    a = np.zeros((2, 256), dtype=np.float32)
    a[1, 128:] = 1.0
    q, s = O.quantize_1x128(a)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0
    assert (q[0] == 0).all() and (q[1, :128] == 0).all()
    assert (q[1, 128:] == 0x7E).all()


def test_scale_is_group_amax_over_448_and_groups_are_column_blocks():
    rng = np.random.default_rng(2)
    a = rng.standard_normal((5, 384)).astype(np.float32)
    a[2, 130] = -9.5  # amax of row 2, group 1, negative
    q, s = O.quantize_1x128(a)
    for r in range(5):
        for g in range(3):
            blk = a[r, g * 128:(g + 1) * 128]
            assert s[r, g] == np.float32(np.abs(blk).max()) / np.float32(448)
    assert q[2, 130] == 0xFE
    # every group holds exactly its amax element(s) at the max code
    mags = q & 0x7F
    for r in range(5):
        for g in range(3):
            assert mags[r, g * 128:(g + 1) * 128].max() == 0x7E


def test_round_trip_error_bound():
    # e4m3 with 3 mantissa bits: |x - q*s| <= 2^-4 |x| for normals, and at most
    # half the subnormal step 2^-10 * s below the normal range
    rng = np.random.default_rng(3)
    a = (rng.standard_normal((64, 512)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(np.float32)
    q, s = O.quantize_1x128(a)
    back = O.dequantize_1x128(q, s)
    sg = np.repeat(s.astype(np.float64), 128, axis=1)
    bound = np.maximum(np.abs(a) * 2.0 ** -4, sg * 2.0 ** -10) * (1 + 1e-6)
    assert (np.abs(back - a) <= bound).all()


def test_division_not_reciprocal_multiply():
    # choose x, s where fp32(x / s) != fp32(x * fp32(1/s)) and the difference
    # crosses an e4m3 rounding boundary; the quantiser must take the division
    rng = np.random.default_rng(4)
    found = 0
    for _ in range(2000):
        amax = np.float32(rng.uniform(0.5, 4.0))
        s = np.float32(amax / np.float32(448))
        x = np.float32(rng.uniform(-amax, amax))
        if np.float32(x / s) != np.float32(x * np.float32(np.float32(1) / s)):
            row = np.zeros(128, dtype=np.float32)
            row[0], row[1] = amax, x
            q, ss = O.quantize_1x128(row[None])
            assert ss[0, 0] == s
            assert q[0, 1] == O.e4m3_encode(np.array([np.float32(x / s)]))[0]
            found += 1
    assert found > 0


def test_negative_zero_and_sign():
    a = np.zeros((1, 128), dtype=np.float32)
    a[0, 0] = 3.0
    a[0, 1] = -0.0
    a[0, 2] = -3.0
    q, _ = O.quantize_1x128(a)
    assert q[0, 0] == 0x7E and q[0, 2] == 0xFE and q[0, 1] == 0x80 and q[0, 3] == 0x00

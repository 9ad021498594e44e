"""Where an h code may legitimately differ between the GPU and the oracle.

h = silu(g) * u depends on the order of its fp32 sums, so the GPU's quotient h / s
sits a little off the oracle's. Away from an e4m3 rounding midpoint both round to
the same code; next to one they may take neighbouring codes. The margin: fp32 sums
of the per-K-block partials and an fp32 SiLU move the quotient by at most ~4e-4 on
the shapes of the tests (emulated in fp32 with K up to 7168), so 4e-3 plus 1e-5 of
the quotient leaves a factor of ten. numpy only (used by the oracle pool's workers).
"""
import numpy as np

from oracle import moe_oracle as O

# e4m3 magnitudes in code order (codes 0x00..0x7E) and the midpoints between neighbours
MAGS = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
MIDS = (MAGS[1:] + MAGS[:-1]) / 2


def midpoint_distance(r: np.ndarray) -> np.ndarray:
    """Distance of |r| to the nearest e4m3 rounding midpoint (in units of the quotient)."""
    a = np.abs(r)
    i = np.clip(np.searchsorted(MIDS, a), 1, len(MIDS) - 1)
    return np.minimum(np.abs(a - MIDS[i - 1]), np.abs(a - MIDS[i]))


def clear_of_midpoint(r: np.ndarray) -> np.ndarray:
    return midpoint_distance(r) > 4e-3 + 1e-5 * np.abs(r)


def quotients(h: np.ndarray, s: np.ndarray) -> np.ndarray:
    """h / s per 1x128 group in fp32, as the quantiser forms them (zero groups: 0)."""
    n, H = h.shape
    s_div = np.where(s != 0, s, np.float32(1)).astype(np.float32)
    return (h.reshape(n, H // 128, 128) / s_div[:, :, None]).astype(np.float32).reshape(n, H)


def flip_steps(h: np.ndarray, q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """For each h element whose quotient lies next to a rounding midpoint, the value
    change of taking the neighbouring code instead (the larger of its two e4m3 steps
    times the group's scale); 0 elsewhere. [n, H] fp64."""
    n, H = h.shape
    r = quotients(h, s).astype(np.float64)
    m = (q & 0x7F).astype(np.int64)
    up = MAGS[np.minimum(m + 1, 0x7E)] - MAGS[m]
    down = MAGS[m] - MAGS[np.maximum(m - 1, 0)]
    step = np.maximum(up, down) * np.repeat(s.astype(np.float64), 128, axis=1)
    return np.where(clear_of_midpoint(r), 0.0, step)

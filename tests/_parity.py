"""Shared checks of the GPU parity tests.

Tolerances (layer outputs, fp64 oracle as reference): max |y - ref| <= 2e-2 RMS(ref)
(plus the bf16 storage rounding of ref, element by element) and
mean |y - ref| / mean |ref| <= 5e-3. Routing: expert ids identical except for
tokens whose k-th / (k+1)-th biased-score gap is below 1e-5, where the GPU's set
must be a valid top-k within 1e-5 of the oracle's k-th score.
"""
import numpy as np
import torch

MAX_REL_RMS = 2e-2
MEAN_REL = 5e-3
TIE_GAP = 1e-5


def bf16_half_ulp(ref):
    """Half a bf16 ulp at |ref|: the largest error of rounding ref to bf16 (8
    significant bits), 2^(floor(log2|ref|) - 8)."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def assert_close_layer(y, ref, what="", bf16_out=True, extra_allow=None):
    """max|y - ref| <= 2e-2 RMS(ref) and mean|y - ref| / mean|ref| <= 5e-3.

    The outputs checked here (the layer's y, the experts' o, the dense FFN's y) are
    bf16 tensors, while ref is the oracle's fp64 value before rounding: element by
    element the bound on the max error adds the half-ulp that storing ref in bf16
    may cost (2^-8 |ref| at most, 1-2% of RMS at a 4-5 sigma output), so that the
    computation, not the storage format, is what the tolerance judges.

    extra_allow (element by element, optional): a further bound derived for an
    intermediate whose codes may legitimately differ (the expert outputs o, whose
    h codes next to an e4m3 rounding midpoint may take the neighbouring code)."""
    y = y.float().cpu().numpy() if isinstance(y, torch.Tensor) else np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    err = np.abs(y - ref)
    rms = np.sqrt((ref ** 2).mean())
    mean_rel = err.mean() / np.abs(ref).mean()
    allow = MAX_REL_RMS * rms + (bf16_half_ulp(ref) if bf16_out else 0.0)
    if extra_allow is not None:
        allow = allow + np.asarray(extra_allow, np.float64)
    excess = err - allow
    i = np.unravel_index(np.argmax(excess), err.shape)
    assert excess[i] <= 0, (f"{what}: |err| {err[i]:.3e} at {i} > {MAX_REL_RMS} * RMS {rms:.3e}"
                            f"{' + bf16 half-ulp of ref' if bf16_out else ''}{' + h-code allowance' if extra_allow is not None else ''}"
                            f" ({allow[i] if np.ndim(allow) else allow:.3e})")
    assert mean_rel <= MEAN_REL, f"{what}: mean relative error {mean_rel:.3e} > {MEAN_REL}"
    return err.max() / rms, mean_rel


def reconcile_routing(gpu_idx, r, k):
    """Compare GPU expert ids with the oracle's route(). Returns the index table
    to evaluate the oracle with.

    The chosen SET must equal the oracle's, except on near-tie tokens (k-th to
    (k+1)-th gap < 1e-5) where the GPU's set must be a valid top-k within 1e-5.
    The ORDER inside the set is not unique when two chosen experts' scores are
    within rounding of each other; it must be descending in the oracle's biased
    scores up to 1e-5. The returned table holds the GPU's order (slot order does
    not change y)."""
    gpu_idx = np.asarray(gpu_idx)
    ref = r["idx"]
    c = r["choice"]
    out = ref.copy()
    near = r["gap"] < TIE_GAP
    for t in range(ref.shape[0]):
        g = gpu_idx[t]
        assert len(set(g.tolist())) == k, f"token {t}: repeated expert ids {g.tolist()}"
        cg = c[t, g]
        assert (cg[:-1] >= cg[1:] - TIE_GAP).all(), f"token {t}: GPU order {g.tolist()} is not descending"
        if set(g.tolist()) != set(ref[t].tolist()):
            assert near[t], f"token {t}: ids {g.tolist()} != oracle {ref[t].tolist()} (gap {r['gap'][t]:.3e})"
            kth = np.sort(c[t])[::-1][k - 1]
            assert (cg >= kth - TIE_GAP).all()
        out[t] = g
    return out

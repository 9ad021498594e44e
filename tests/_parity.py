"""Shared checks of the GPU parity tests.

Tolerances (layer outputs, fp64 oracle as reference): max |y - ref| <= 2e-2 RMS(ref)
and mean |y - ref| / mean |ref| <= 5e-3. Routing: expert ids identical except for
tokens whose k-th / (k+1)-th biased-score gap is below 1e-5, where the GPU's set
must be a valid top-k within 1e-5 of the oracle's k-th score.
"""
import numpy as np
import torch

MAX_REL_RMS = 2e-2
MEAN_REL = 5e-3
TIE_GAP = 1e-5


def assert_close_layer(y, ref, what=""):
    y = y.float().cpu().numpy() if isinstance(y, torch.Tensor) else np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    err = np.abs(y - ref)
    rms = np.sqrt((ref ** 2).mean())
    mean_rel = err.mean() / np.abs(ref).mean()
    assert err.max() <= MAX_REL_RMS * rms, f"{what}: max|err| {err.max():.3e} > {MAX_REL_RMS} * RMS {rms:.3e}"
    assert mean_rel <= MEAN_REL, f"{what}: mean relative error {mean_rel:.3e} > {MEAN_REL}"
    return err.max() / rms, mean_rel


def reconcile_routing(gpu_idx, r, k):
    """Compare GPU expert ids with the oracle's route(). Returns the index table
    to evaluate the oracle with (the GPU's ids on near-tie tokens)."""
    gpu_idx = np.asarray(gpu_idx)
    ref = r["idx"]
    c = r["choice"]
    out = ref.copy()
    near = r["gap"] < TIE_GAP
    for t in range(ref.shape[0]):
        if (gpu_idx[t] == ref[t]).all():
            continue
        assert near[t], f"token {t}: ids {gpu_idx[t].tolist()} != oracle {ref[t].tolist()} (gap {r['gap'][t]:.3e})"
        kth = np.sort(c[t])[::-1][k - 1]
        assert len(set(gpu_idx[t].tolist())) == k
        assert (c[t, gpu_idx[t]] >= kth - TIE_GAP).all()
        out[t] = gpu_idx[t]
    return out

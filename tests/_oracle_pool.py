"""The oracle's expert SwiGLU over many (expert, rows) jobs at once, in a process
pool started with the spawn method (numpy only: no torch, no CUDA in the
workers, and none forked from a process that has touched the GPU).

Each job is one call of the oracle's ``swiglu_fp8`` on the given rows of one
expert; nothing here adds arithmetic of its own.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _job(args):
    from oracle import moe_oracle as O
    key, flips, xq, xs, w1q, w1s, w3q, w3s, w2q, w2s = args
    o, hq, hs = O.swiglu_fp8(xq, xs, w1q, w1s, w3q, w3s, w2q, w2s)
    if not flips:
        return key, (o, None)
    # the most each output may move when h codes next to a rounding midpoint take
    # the neighbouring code: sum over those features of step x |w2|
    from _hmargin import flip_steps
    h = O.swiglu_h(xq, xs, w1q, w1s, w3q, w3s)
    steps = flip_steps(h, hq, hs)
    return key, (o, steps @ np.abs(O.decode_block_weight(w2q, w2s)).T)


def _init(root):
    import sys
    if root not in sys.path:
        sys.path.insert(0, root)


def swiglu_jobs(keys, make_job, workers=None, flips=False):
    """For each key, make_job(key) -> (xq [n, d] uint8, xs [n, d/128] fp32, w1q, w1s,
    w3q, w3s, w2q, w2s) as numpy arrays. Returns {key: o fp64 [n, d]}, or with
    flips=True {key: (o, allowance [n, d])}, the allowance bounding what h codes next
    to a rounding midpoint may change. Jobs are made a few per worker at a time, so
    the experts' weights are not all held at once."""
    keys = list(keys)
    if not keys:
        return {}
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    n = workers or max(1, min(len(keys), (os.cpu_count() or 2) - 1, 16))
    ctx = mp.get_context("spawn")
    # one BLAS thread per worker (the pool supplies the parallelism): the workers
    # read these when they start, before numpy loads
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in saved:
        os.environ[v] = "1"
    try:
        out = {}
        with ctx.Pool(n, initializer=_init, initargs=(root,)) as pool:
            for i in range(0, len(keys), 2 * n):
                batch = [(k, flips) + tuple(make_job(k)) for k in keys[i:i + 2 * n]]
                out.update(pool.imap_unordered(_job, batch, chunksize=1))
        return out if flips else {k: v[0] for k, v in out.items()}
    finally:
        for v, val in saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val

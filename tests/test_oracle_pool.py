"""The spawned oracle pool used by the full-size GPU parity tests gives the serial
oracle's results exactly (it only distributes calls of the oracle's SwiGLU)."""
import numpy as np

import moe_synth as S
from oracle import moe_oracle as O
from _oracle_pool import swiglu_jobs


def test_pool_matches_serial_oracle():
    ex = S.gen_experts(3, 256, 128, seed=4)
    rng = np.random.default_rng(0)
    rows = {0: 5, 1: 1, 2: 9}
    xq = {e: rng.integers(0, 126, (n, 256)).astype(np.uint8) for e, n in rows.items()}
    xs = {e: rng.uniform(1e-3, 1e-1, (n, 2)).astype(np.float32) for e, n in rows.items()}

    def make(e):
        return (xq[e], xs[e]) + tuple(t.numpy() for t in ex.expert(e))

    out = swiglu_jobs(sorted(rows), make, workers=2)
    assert sorted(out) == [0, 1, 2]
    for e in rows:
        ref, _, _ = O.swiglu_fp8(xq[e], xs[e], *[t.numpy() for t in ex.expert(e)])
        assert np.array_equal(out[e], ref)


def test_flip_steps_next_to_a_midpoint():
    # a group with amax 448 has scale 1, so the quotients are the h values: 100.001
    # lies 1e-3 above the midpoint between the e4m3 values 96 and 104 (within the
    # margin 4e-3 + 1e-5 * 100), 99 and 101 lie a whole unit from it
    from _hmargin import flip_steps
    h = np.zeros((2, 128), np.float32)
    h[0, 0] = 448.0
    h[0, 5], h[0, 6], h[0, 7] = 100.001, 99.0, 101.0
    h[1, :] = 0.0                                   # an all-zero group: scale 0, no steps
    q, s = O.quantize_1x128(h)
    assert s[0, 0] == 1.0 and s[1, 0] == 0.0
    assert O.e4m3_decode(q[0, 5:8]).tolist() == [104.0, 96.0, 104.0]
    st = flip_steps(h, q, s)
    assert st[0, 5] == 8.0                          # 104 <-> 96 or 112: one step of 8
    assert st[0, 6] == 0 and st[0, 7] == 0 and st[0, 0] == 0 and (st[1] == 0).all()
    # quotients of 0 lie within the margin of the first midpoint (2^-10): a step of
    # the smallest subnormal code, 2^-9
    assert (st[0, 8:] == 2.0 ** -9).all()
    # the allowance (steps @ |w2|^T) bounds the output change of that code's flip
    w2 = np.random.default_rng(2).normal(0, 0.02, (64, 128))
    allow = st @ np.abs(w2).T
    q2 = q.copy()
    q2[0, 5] = O.e4m3_encode(np.array([96.0]))[0]
    d_o = (O.e4m3_decode(q2) - O.e4m3_decode(q)) @ w2.T
    assert (np.abs(d_o) <= allow + 1e-15).all() and np.abs(d_o[0]).max() > 0

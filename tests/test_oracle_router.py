"""Pins for the oracle's gate: sigmoid scores, biased top-k choice, weights.

Sources: "Kimi-K2-Base", Mixture of experts (Router score sigmoid; load balancing
by e_score_correction_bias added for the top-k choice only; routed scaling factor
2.827 applied after renormalising the top-k weights; no group-limited routing).
"""
import itertools

import numpy as np
import pytest

from oracle import moe_oracle as O


def brute_topk(c, k):
    """Best subset by enumeration: maximal sum of choice scores; among equal sums
    the lexicographically smallest sorted id tuple."""
    best, best_key = None, None
    for sub in itertools.combinations(range(len(c)), k):
        key = (-sum(c[i] for i in sub), sub)
        if best_key is None or key < best_key:
            best, best_key = sub, key
    return set(best)


@pytest.mark.parametrize("E,k", [(12, 3), (16, 8), (9, 8)])
def test_topk_matches_subset_enumeration(E, k):
    rng = np.random.default_rng(E * 100 + k)
    c = rng.standard_normal((6, E))
    got = O.topk_select(c, k)
    for t in range(c.shape[0]):
        assert set(got[t].tolist()) == brute_topk(c[t].tolist(), k)
        assert list(got[t]) == sorted(got[t], key=lambda i: (-c[t, i], i))


def test_topk_ties_go_to_lower_id():
    c = np.array([[0.5, 0.9, 0.5, 0.9, 0.1, 0.5]])
    assert O.topk_select(c, 4)[0].tolist() == [1, 3, 0, 2]
    # integer-valued ties: brute force agrees on the set
    rng = np.random.default_rng(7)
    c = rng.integers(0, 3, (20, 10)).astype(np.float64)
    got = O.topk_select(c, 4)
    for t in range(20):
        assert set(got[t].tolist()) == brute_topk(c[t].tolist(), 4)


def test_sigmoid_closed_form():
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    x = np.array([-3.0, -0.5, 0.7, 4.0])
    np.testing.assert_allclose(O.sigmoid(x) + O.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.sigmoid(np.log(np.array([3.0]))), [0.75], rtol=1e-15)


def test_logits_orientation():
    # x [T, d] against W_g [E, d]: logit[t, e] = <x_t, W_g[e]>
    x = np.zeros((2, 4)); x[0, 1] = 1.0; x[1, 3] = 2.0
    wg = np.zeros((3, 4)); wg[0, 1] = 5.0; wg[2, 3] = -1.0
    l = O.router_logits(x, wg)
    assert l.shape == (2, 3)
    np.testing.assert_array_equal(l, [[5.0, 0, 0], [0, 0, -2.0]])


def test_bias_chooses_but_does_not_weight():
    # scores s = sigmoid(l); expert 3 has a low score but a large bias: it is
    # chosen, and its weight comes from its unbiased score
    T, d, E = 1, 4, 6
    l = np.array([2.0, 1.0, 0.5, -1.0, 0.0, 0.2])
    x = np.eye(1, d)                       # picks column 0 of each gate row
    wg = np.zeros((E, d)); wg[:, 0] = l
    bias = np.zeros(E); bias[3] = 10.0
    r = O.route(x, wg, bias, topk=2, route_scale=2.827)
    assert r["idx"][0].tolist() == [3, 0]
    s = O.sigmoid(l)
    np.testing.assert_allclose(r["w"][0], [s[3] / (s[3] + s[0]) * 2.827, s[0] / (s[3] + s[0]) * 2.827],
                               rtol=1e-14)
    np.testing.assert_allclose(r["choice"][0], s + bias, rtol=1e-15)


def test_weights_sum_to_route_scale_and_ids_distinct():
    rng = np.random.default_rng(5)
    T, d, E, k = 40, 64, 32, 8
    x = rng.standard_normal((T, d)); wg = rng.standard_normal((E, d)) * 0.1
    bias = rng.standard_normal(E) * 0.01
    r = O.route(x, wg, bias, k, 2.827)
    np.testing.assert_allclose(r["w"].sum(1), 2.827, rtol=0, atol=1e-12)
    for t in range(T):
        assert len(set(r["idx"][t].tolist())) == k
    assert (r["w"] > 0).all()
    # gap = k-th minus (k+1)-th best choice score, non-negative
    srt = np.sort(r["choice"], axis=1)[:, ::-1]
    np.testing.assert_array_equal(r["gap"], srt[:, k - 1] - srt[:, k])
    assert (r["gap"] >= 0).all()

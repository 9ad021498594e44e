"""Pins for the oracle's token permutation into per-expert segments."""
import numpy as np

from oracle import moe_oracle as O


def _ints(s):
    return [int(v) for v in s.split(",")]


def test_hand_worked_example(golden):
    rows = {r[0]: r[1:] for r in golden("permute_worked_example.txt")}
    E = int(rows["E"][0])
    idx = np.array([_ints(p) for p in rows["idx"]])
    p = O.permute(idx, E)
    assert p["counts"].tolist() == _ints(rows["counts"][0])
    assert p["offsets"].tolist() == _ints(rows["offsets"][0])
    assert p["sorted_tok"].tolist() == _ints(rows["sorted_tok"][0])
    assert p["inv_pos"].tolist() == [_ints(q) for q in rows["inv_pos"]]


def test_invariants_random():
    rng = np.random.default_rng(11)
    T, E, k = 300, 40, 8
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = O.permute(idx, E)
    assert p["counts"].sum() == k * T
    assert p["offsets"][0] == 0 and p["offsets"][-1] == k * T
    np.testing.assert_array_equal(np.diff(p["offsets"]), p["counts"])
    np.testing.assert_array_equal(p["counts"], np.bincount(idx.ravel(), minlength=E))
    # sorted_tok[inv_pos[t, j]] == t, and each position is used exactly once
    assert (p["sorted_tok"][p["inv_pos"]] == np.arange(T)[:, None]).all()
    assert sorted(p["inv_pos"].ravel().tolist()) == list(range(k * T))
    for e in range(E):
        seg = p["sorted_tok"][p["offsets"][e]:p["offsets"][e + 1]]
        assert (np.diff(seg) > 0).all()
        assert (idx[seg] == e).any(axis=1).all()


def test_empty_and_single_hot_expert():
    idx = np.zeros((0, 8), dtype=np.int32)
    p = O.permute(idx, 16)
    assert p["offsets"].tolist() == [0] * 17 and p["sorted_tok"].size == 0
    # every token picks experts 0..7: experts 8.. get empty segments
    idx = np.tile(np.arange(8), (5, 1))
    p = O.permute(idx, 16)
    assert p["counts"].tolist() == [5] * 8 + [0] * 8
    assert p["sorted_tok"].tolist() == list(range(5)) * 8

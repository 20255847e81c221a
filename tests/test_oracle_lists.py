"""Pins of the oracle's per-expert routing lists (wide page, WideRoute: each
(token, slot) pair code t*K + k appended to its expert's list) against invariants and
a brute-force per-expert filter."""
import numpy as np
import pytest


def _ids(rng, T, K, E, skew=False):
    p = None
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
    return np.stack([rng.choice(E, size=K, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,K,E,skew", [(1, 16, 896, False), (37, 16, 896, False), (64, 8, 64, True), (200, 4, 33, False), (5, 1, 1, False)])
def test_invariants_and_bruteforce(orc, T, K, E, skew):
    rng = np.random.default_rng(T + K + E)
    ids = _ids(rng, T, K, E, skew)
    off, pairs = orc.routing_lists(ids, E)
    assert off[0] == 0 and off[E] == T * K
    assert np.all(np.diff(off) >= 0)
    assert sorted(pairs.tolist()) == list(range(T * K))
    for e in range(E):
        lst = pairs[off[e]:off[e + 1]].tolist()
        assert lst == [t * K + k for t in range(T) for k in range(K) if ids[t, k] == e]
        assert all(ids[p // K, p % K] == e for p in lst)
        assert all(a < b for a, b in zip(lst, lst[1:]))
    np.testing.assert_array_equal(np.diff(off), np.bincount(ids.ravel(), minlength=E))


def test_empty_batch(orc):
    off, pairs = orc.routing_lists(np.zeros((0, 16), np.int32), 896)
    assert np.all(off == 0) and pairs.size == 0


def test_bad_id_rejected(orc):
    with pytest.raises(ValueError):
        orc.routing_lists(np.array([[0, 5]], np.int32), 5)

"""Pins of the oracle's unit windows (wide page, module docstring: the grouped
engine reads each expert with tokens once per 8 of them) by closed forms and by
invariants checked against the routing lists they cut."""
import numpy as np
import pytest


def test_closed_form(orc):
    # experts with 0, 17, 1, 8, 0 listed pairs and windows of 8: 3 + 1 + 1 units
    off = np.array([0, 0, 17, 18, 26, 26], np.int32)
    uo, ue, us, ul = orc.unit_windows(off, 8)
    assert uo.tolist() == [0, 0, 3, 4, 5, 5]
    assert ue.tolist() == [1, 1, 1, 2, 3]
    assert us.tolist() == [0, 8, 16, 17, 18]
    assert ul.tolist() == [8, 8, 1, 1, 8]


def test_window_one_and_window_large(orc):
    off = np.array([0, 3, 3, 7], np.int32)
    uo, ue, us, ul = orc.unit_windows(off, 1)  # one unit per listed pair
    assert uo.tolist() == [0, 3, 3, 7] and us.tolist() == list(range(7)) and set(ul.tolist()) == {1}
    uo, ue, us, ul = orc.unit_windows(off, 1000)  # one unit per touched expert
    assert uo.tolist() == [0, 1, 1, 2] and ue.tolist() == [0, 2] and ul.tolist() == [3, 4]


def test_empty_lists(orc):
    uo, ue, us, ul = orc.unit_windows(np.zeros(9, np.int32), 8)
    assert uo.tolist() == [0] * 9 and ue.size == 0


@pytest.mark.parametrize("T,K,E,W,seed", [(1020, 16, 896, 8, 0), (64, 16, 896, 8, 1), (300, 8, 33, 5, 2),
                                          (17, 4, 7, 3, 3)])
def test_invariants_on_real_lists(orc, T, K, E, W, seed):
    rng = np.random.default_rng(seed)
    logp = -1.1 * np.log(np.arange(1, E + 1))  # skewed loads: heavy and empty experts
    ids = np.argsort(-(logp[None, :] + rng.gumbel(size=(T, E))), axis=1)[:, :K].astype(np.int32)
    off, pairs = orc.routing_lists(ids, E)
    uo, ue, us, ul = orc.unit_windows(off, W)
    n = uo[-1]
    assert uo[0] == 0 and np.all(np.diff(uo) >= 0) and ue.size == n
    # the units, in order, tile the list positions 0 .. T*K-1 exactly once
    assert us[0] == 0 and np.array_equal(us[1:], (us + ul)[:-1]) and us[-1] + ul[-1] == T * K
    assert np.all((ul >= 1) & (ul <= W))
    counts = np.diff(off)
    for e in range(E):
        u0, u1 = uo[e], uo[e + 1]
        assert np.all(ue[u0:u1] == e)
        # every position of a unit of e lies in e's list, so its pairs are routed to e
        if u1 > u0:
            assert us[u0] == off[e] and us[u1 - 1] + ul[u1 - 1] == off[e + 1]
            assert np.all(ids.ravel()[pairs[us[u0]:us[u1 - 1] + ul[u1 - 1]]] == e)
        # the fewest windows: all full but the last (the expert streams once per W pairs)
        assert u1 - u0 == -(-counts[e] // W)
        assert np.all(ul[u0:max(u0, u1 - 1)] == W)

"""Pins of the oracle's specified exp and sigmoid (Cody-Waite reduction + degree-7
Taylor, correctly rounded 1/(1+e)) against double-precision libm and closed forms."""
import math

import numpy as np


def _ulp(x: float) -> float:
    return float(np.spacing(np.float32(abs(x))))


def test_exp_spec_within_2ulp(orc):
    ys = np.concatenate([np.linspace(-17.49, 88.49, 20001), np.random.default_rng(0).uniform(-17.5, 88.5, 20000)])
    ys = ys.astype(np.float32)
    worst = 0.0
    for y in ys:
        got = orc.exp_spec(float(y))
        ref = math.exp(float(y))
        err = abs(got - ref) / _ulp(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_exp_spec_exact_points(orc):
    assert orc.exp_spec(0.0) == 1.0
    # a dropped polynomial term or a wrong reduction constant shows here
    assert abs(orc.exp_spec(1.0) - math.e) <= 2 * _ulp(math.e)
    assert abs(orc.exp_spec(-10.0) - math.exp(-10.0)) <= 2 * _ulp(math.exp(-10.0))


def test_sigmoid_closed_forms(orc):
    s = orc.sigmoid(np.array([0.0, 17.5, 100.0, 1e30, -88.5, -100.0, -1e30, float("inf"), float("-inf")], np.float32))
    assert s[0] == 0.5
    assert np.all(s[1:4] == 1.0) and s[7] == 1.0
    assert np.all(s[4:7] == 0.0) and s[8] == 0.0
    assert np.isnan(orc.sigmoid(np.array([np.nan], np.float32))[0])


def test_sigmoid_against_libm(orc):
    xs = np.concatenate([np.linspace(-88.4, 17.4, 40001), np.random.default_rng(1).normal(0, 3, 20000)])
    xs = xs.astype(np.float32)
    xs = xs[(xs > -88.5) & (xs < 17.5)]
    got = orc.sigmoid(xs).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-xs.astype(np.float64)))
    ulps = np.abs(got - ref) / np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert ulps.max() <= 3.0, ulps.max()


def test_sigmoid_monotone_and_symmetric(orc):
    xs = np.sort(np.random.default_rng(2).uniform(-30, 30, 50000).astype(np.float32))
    s = orc.sigmoid(xs)
    assert np.all(np.diff(s) >= 0)
    pos = xs[(xs > 0) & (xs < 17)]
    a = orc.sigmoid(pos).astype(np.float64) + orc.sigmoid(-pos).astype(np.float64)
    assert np.max(np.abs(a - 1.0)) < 3e-7

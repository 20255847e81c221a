"""Pins of the oracle's sigmoid+bias top-k ("EpMoeLayer.topk" of the DEP page: one
group, sigmoid scoring, correction bias, renormalize, scale; the wide page's WideRoute: an
exact top-16 with renormalised weights) against closed forms and a
brute-force sort."""
import numpy as np
import pytest

from helpers import bits_from_f32, expand_list, golden_lines


@pytest.mark.parametrize("row", list(golden_lines("topk_closed_forms.txt")), ids=lambda r: r[0])
def test_golden(orc, row):
    name, E, K, renorm, scale, logits, bias, ids, wbits = row
    E, K = int(E), int(K)
    lg = np.array([expand_list(logits)], np.float32)
    b = np.array(expand_list(bias), np.float32)
    got_ids, got_w, got_wb = orc.topk_route(lg, b, K, bool(int(renorm)), float(scale))
    assert got_ids[0].tolist() == [int(v) for v in ids.split(",")]
    exp_w = [int(v, 16) for v in expand_list(wbits, str)]
    assert [bits_from_f32(float(v)) for v in got_w[0]] == exp_w
    assert got_wb[0].tolist() == [((u + 0x7FFF + ((u >> 16) & 1)) >> 16) for u in exp_w]


def _brute(orc, logits, bias, K):
    s = orc.sigmoid(logits)
    c = (s + bias).astype(np.float32) if bias is not None else s
    out = []
    for t in range(logits.shape[0]):
        order = sorted(range(logits.shape[1]), key=lambda e: (-float(c[t, e]), e))
        out.append(order[:K])
    return np.array(out, np.int32), s


@pytest.mark.parametrize("E", [16, 17, 32, 64, 96])
@pytest.mark.parametrize("K", [1, 4, 16])
@pytest.mark.parametrize("kind", ["random", "ties"])
def test_bruteforce_selection(orc, E, K, kind):
    if K > E:
        pytest.skip()
    rng = np.random.default_rng(E * 100 + K)
    T = 12
    if kind == "random":
        logits = rng.normal(0, 2, (T, E)).astype(np.float32)
        bias = rng.normal(0, 0.05, E).astype(np.float32)
    else:  # sigmoid saturates to exactly 0 or 1, bias on a coarse grid: many equal keys
        logits = rng.choice(np.array([-100, 20, 0], np.float32), size=(T, E))
        bias = (rng.integers(-2, 3, E) / 16.0).astype(np.float32)
    ids, w, wb = orc.topk_route(logits, bias, K, True, 1.0)
    exp_ids, s = _brute(orc, logits, bias, K)
    np.testing.assert_array_equal(ids, exp_ids)
    for t in range(T):
        sel = s[t, ids[t]].astype(np.float64)
        if sel.sum() > 0:
            # renormalised: sums to 1 within a few ulp, proportional to the unbiased scores
            assert abs(w[t].astype(np.float64).sum() - 1.0) <= 16 * 2.0 ** -24
            np.testing.assert_allclose(w[t] * sel.sum(), sel, rtol=4e-7, atol=1e-30)
        else:
            assert np.all(w[t] == 0)


def test_ids_distinct_and_valid(orc):
    rng = np.random.default_rng(9)
    logits = rng.normal(0, 1.7, (50, 896)).astype(np.float32)
    bias = rng.normal(0, 0.01, 896).astype(np.float32)
    ids, w, _ = orc.topk_route(logits, bias, 16)
    for t in range(50):
        assert len(set(ids[t].tolist())) == 16
        assert ids[t].min() >= 0 and ids[t].max() < 896
        c = orc.sigmoid(logits[t]) + bias
        chosen = c[ids[t]]
        assert np.all(np.diff(chosen) <= 0)  # slots in descending key order
        rest = np.delete(c, ids[t])
        assert rest.max() <= chosen.min()


def test_no_bias_and_no_renorm(orc):
    logits = np.array([[0.0, 3.0, -1.0, 2.0]], np.float32)
    ids, w, _ = orc.topk_route(logits, None, 2, renormalize=False)
    assert ids[0].tolist() == [1, 3]
    s = orc.sigmoid(logits[0])
    assert w[0].tolist() == [s[1], s[3]]


def test_all_scores_zero(orc):
    logits = np.full((1, 20), -200.0, np.float32)
    ids, w, _ = orc.topk_route(logits, None, 4)
    assert ids[0].tolist() == [0, 1, 2, 3]
    assert np.all(w == 0)


def test_k_equals_e(orc):
    logits = np.array([[1.0, -1.0, 0.5]], np.float32)
    ids, w, _ = orc.topk_route(logits, None, 3)
    assert ids[0].tolist() == [0, 2, 1]

"""Pins of the oracle's Finalize (wide page, class Finalize: FP32 fma over k in
order, one BF16 rounding) and its shared-expert variant (GLM-5-next finalize page:
weight x routed_scaling_factor, -1 rows skipped, shared row added once in FP32)."""
from fractions import Fraction

import numpy as np
import pytest

import synth
from helpers import bf16_value, f32_from_bits, golden_lines, round_fraction_to_bf16


@pytest.mark.parametrize("row", list(golden_lines("finalize_closed_forms.txt")), ids=lambda r: r[0])
def test_golden(orc, row):
    name, wbits, rbits, exp = row
    w = np.array([f32_from_bits(int(v, 16)) for v in wbits.split(",")], np.float32)[None, :]
    K = w.shape[1]
    rows = np.array([int(v, 16) for v in rbits.split(",")], np.uint16).reshape(K, 1)
    rows = np.repeat(rows, 8, axis=1)  # H = 8, every column the same case
    out = orc.finalize(rows, w, T=1, K=K)
    assert np.all(out == int(exp, 16))


def test_one_hot_reproduces_rows(orc):
    T, K, H = 5, 16, 64
    rows = synth.normal_bf16(1, 4, (T * K, H))
    w = np.zeros((T, K), np.float32)
    pick = np.random.default_rng(0).integers(0, K, T)
    w[np.arange(T), pick] = 1.0
    out = orc.finalize(rows, w, T, K)
    np.testing.assert_array_equal(out, rows[np.arange(T) * K + pick])


def test_integer_rows_pow2_weights_closed_form(orc):
    rng = np.random.default_rng(2)
    T, K, H = 3, 16, 32
    ri = rng.integers(-64, 65, (T * K, H))
    rows = synth.f32_to_bf16_bits(ri.astype(np.float32))
    wexp = rng.integers(-6, 3, (T, K))
    wsgn = rng.choice([-1, 1], (T, K))
    w = (wsgn * np.exp2(wexp)).astype(np.float32)
    out = orc.finalize(rows, w, T, K)
    for t in range(T):
        for c in range(H):
            exact = sum(Fraction(int(wsgn[t, k])) * Fraction(2) ** int(wexp[t, k]) * int(ri[t * K + k, c]) for k in range(K))
            assert out[t, c] == round_fraction_to_bf16(exact)


def test_bf16_weights_equal_fp32_weights(orc):
    T, K, H = 4, 16, 40
    rows = synth.normal_bf16(2, 4, (T * K, H))
    wb = synth.normal_bf16(2, 7, (T, K), 0.1)
    wf = synth.bf16_bits_to_f32(wb)
    np.testing.assert_array_equal(orc.finalize(rows, wb, T, K), orc.finalize(rows, wf, T, K))


def test_all_minus_one_gives_shared(orc):
    T, K, H = 3, 8, 48
    rows = synth.normal_bf16(3, 4, (T * K, H))
    shared = synth.normal_bf16(3, 8, (T, H))
    idx = np.full((T, K), -1, np.int32)
    w = np.ones((T, K), np.float32)
    out = orc.finalize(rows, w, T, K, row_index=idx, shared=shared, scale=2.5)
    np.testing.assert_array_equal(out, shared)


def test_gather_with_zero_shared_equals_plain(orc):
    T, K, H = 4, 8, 24
    n = T * K
    rows = synth.normal_bf16(4, 4, (n, H))
    perm = np.random.default_rng(4).permutation(n).astype(np.int32).reshape(T, K)
    w = synth.normal_bf16(4, 7, (T, K), 0.2)
    plain = orc.finalize(rows[perm.reshape(-1)], w, T, K)
    zero = np.zeros((T, H), np.uint16)
    np.testing.assert_array_equal(orc.finalize(rows, w, T, K, row_index=perm, shared=zero), plain)


def test_scale_and_shared_closed_form(orc):
    rng = np.random.default_rng(6)
    T, K, H = 2, 8, 16
    n = 20
    ri = rng.integers(-32, 33, (n, H))
    rows = synth.f32_to_bf16_bits(ri.astype(np.float32))
    idx = rng.integers(-1, n, (T, K)).astype(np.int32)
    wexp = rng.integers(-4, 2, (T, K))
    w = synth.f32_to_bf16_bits(np.exp2(wexp).astype(np.float32))
    si = rng.integers(-100, 101, (T, H))
    shared = synth.f32_to_bf16_bits(si.astype(np.float32))
    out = orc.finalize(rows, w, T, K, row_index=idx, shared=shared, scale=2.5)
    for t in range(T):
        for c in range(H):
            exact = Fraction(int(si[t, c]))
            for k in range(K):
                if idx[t, k] >= 0:
                    exact += Fraction(5, 2) * Fraction(2) ** int(wexp[t, k]) * int(ri[idx[t, k], c])
            assert out[t, c] == round_fraction_to_bf16(exact)


def test_bad_index_rejected(orc):
    rows = np.zeros((4, 8), np.uint16)
    w = np.ones((1, 2), np.float32)
    with pytest.raises(ValueError):
        orc.finalize(rows, w, 1, 2, row_index=np.array([[0, 4]], np.int32))
    with pytest.raises(ValueError):
        orc.finalize(rows, w, 1, 2, row_index=np.array([[-2, 0]], np.int32))

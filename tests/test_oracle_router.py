"""Pins of the oracle's FP64 router logits (FP32 router logits of the wide and DEP
pages: logits = x @ gate^T) against exact integer arithmetic and an independent
FP64 matmul."""
import numpy as np

import synth


def _bf16_ints(rng, shape, lo, hi):
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return synth.f32_to_bf16_bits(v), v.astype(np.int64)


def test_integer_exact(orc):
    rng = np.random.default_rng(3)
    xb, xi = _bf16_ints(rng, (4, 7168), -8, 8)
    wb, wi = _bf16_ints(rng, (24, 7168), -8, 8)
    out, ab = orc.router_logits(xb, wb)
    np.testing.assert_array_equal(out, (xi @ wi.T).astype(np.float64))
    np.testing.assert_array_equal(ab, (np.abs(xi) @ np.abs(wi).T).astype(np.float64))


def test_random_against_numpy_f64(orc):
    x = synth.normal_bf16(5, 1, (6, 512), 1.0)
    w = synth.normal_bf16(5, 2, (40, 512), 0.02)
    out, ab = orc.router_logits(x, w)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(w).astype(np.float64).T
    assert np.all(np.abs(out - ref) <= 1e-12 * ab)
    # a transposed operand or a wrong row would be far off
    assert np.max(np.abs(out - ref)) < 1e-9


def test_sampled_matches_full(orc):
    x = synth.normal_bf16(6, 1, (5, 256), 1.0)
    w = synth.normal_bf16(6, 2, (33, 256), 0.02)
    full, fab = orc.router_logits(x, w)
    t = np.array([0, 4, 2, 3], np.int32)
    e = np.array([32, 0, 17, 5], np.int32)
    s, sab = orc.router_logits_sampled(x, w, t, e)
    np.testing.assert_array_equal(s, full[t, e])
    np.testing.assert_array_equal(sab, fab[t, e])


def test_token_ranges_on_threads_match_one_call(orc):
    """The threaded form (token ranges on host threads) gives the single call's values,
    bit for bit, including ranges of uneven length."""
    x = synth.normal_bf16(7, 1, (13, 384), 1.0)
    w = synth.normal_bf16(7, 2, (29, 384), 0.02)
    one, one_ab = orc.router_logits(x, w, threads=1)
    for n in (2, 5, 13, 40):
        par, par_ab = orc.router_logits(x, w, threads=n)
        np.testing.assert_array_equal(par, one)
        np.testing.assert_array_equal(par_ab, one_ab)

"""Pins of the oracle's RMSNorm (the ep page's rms_norm of the routed latent, eps
1e-5; the wide page's latent RMSNorm) by closed forms and invariants."""
import math

import numpy as np

import synth


def _bf(v):
    return synth.f32_to_bf16_bits(np.asarray(v, np.float32))


def test_closed_form_two_columns(orc):
    # x = (3, 4), g = (1, 2), eps = 0: mean square 12.5
    y = orc.rmsnorm(_bf([[3.0, 4.0]]), _bf([1.0, 2.0]), eps=0.0)
    r = 1.0 / math.sqrt(12.5)
    assert np.allclose(y, [[3.0 * r, 8.0 * r]], rtol=0, atol=1e-15)


def test_constant_row_normalises_to_sign(orc):
    x = _bf([[-0.375] * 64, [6.0] * 64])
    y = orc.rmsnorm(x, _bf([1.0] * 64), eps=0.0)
    assert np.array_equal(y, np.array([[-1.0] * 64, [1.0] * 64]))


def test_eps_enters_under_the_root(orc):
    # all ones, eps = 3: 1 / sqrt(1 + 3) = 0.5 exactly
    y = orc.rmsnorm(_bf([[1.0] * 32]), _bf([1.0] * 32), eps=3.0)
    assert np.array_equal(y, np.full((1, 32), 0.5))
    z = orc.rmsnorm(_bf([[0.0] * 32]), _bf([1.0] * 32), eps=1e-5)
    assert np.array_equal(z, np.zeros((1, 32)))


def test_unit_mean_square_and_scale_invariance(orc):
    x = synth.normal_bf16(5, 1, (4, 3584))
    g1 = _bf([1.0] * 3584)
    y = orc.rmsnorm(x, g1, eps=0.0)
    assert np.allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-12)
    x4 = _bf(synth.bf16_bits_to_f32(x) * 4.0)  # exact: a power of two
    assert np.allclose(orc.rmsnorm(x4, g1, eps=0.0), y, rtol=1e-14)
    g = synth.norm_weight()
    yg = orc.rmsnorm(x, g, eps=0.0)
    assert np.allclose(yg, y * synth.bf16_bits_to_f32(g).astype(np.float64)[None, :], rtol=1e-14)


def test_bounds_bracket_the_value(orc):
    y = np.array([1.0, -2.5, 1.0 + 2.0 ** -8, 3.0e-3, 0.0])
    lo, hi = orc.rmsnorm_bounds(y)
    f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
    r = f(orc.f64_to_bf16(y))  # the rounding of the exact value lies between them
    assert np.all(f(lo) <= r) and np.all(r <= f(hi))
    assert int(lo[2]) == 0x3F80 and int(hi[2]) == 0x3F81  # a tie: both neighbours allowed
    assert int(lo[0]) == int(hi[0]) == 0x3F80             # far from a boundary: one value

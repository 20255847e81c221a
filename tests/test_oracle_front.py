"""Pins of the oracle's latent down projection (the wide page's front GEMM: the latent
columns rounded once to BF16, module docstring): its one rounding of an FP64 sum to
BF16 against exact rationals and closed forms, and the whole function on integer
inputs whose sums are exact."""
import random
from fractions import Fraction

import numpy as np

import synth
from helpers import round_fraction_to_bf16


def test_f64_to_bf16_matches_exact_rational(orc):
    # doubles with up to 53 significant bits, normal BF16 range: one rounding of the
    # exact value, compared with a brute-force choice between the two neighbours
    rnd = random.Random(7)
    vals = []
    for _ in range(4000):
        m = rnd.getrandbits(53) | (1 << 52)
        e = rnd.randint(-120, 120)
        v = m * 2.0 ** (e - 52)
        vals.append(-v if rnd.random() < 0.5 else v)
    got = orc.f64_to_bf16(np.array(vals))
    for v, g in zip(vals, got):
        assert int(g) == round_fraction_to_bf16(Fraction(v)), v


def test_f64_to_bf16_rounds_once_not_twice(orc):
    # 1 + 2^-8 + 2^-30 lies just above the tie between 1 and 1 + 2^-7: one rounding
    # goes up. Through FP32 first it would become the tie 1 + 2^-8 and then go to 1.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert int(orc.f64_to_bf16([v])[0]) == 0x3F81
    assert orc.f32_to_bf16(np.float32(v)) == 0x3F80
    assert int(orc.f64_to_bf16([-v])[0]) == 0xBF81


def test_f64_to_bf16_closed_forms(orc):
    cases = [  # (value, bits): a list, since 0.0 and -0.0 would merge as dict keys
        (1.0, 0x3F80), (-2.5, 0xC020), (0.0, 0x0000), (-0.0, 0x8000),
        (1.0 + 2.0 ** -8, 0x3F80),  # tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),  # tie -> even (up)
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # tie above it -> even = 2^128 -> inf
        ((2 - 2.0 ** -8 - 2.0 ** -20) * 2.0 ** 127, 0x7F7F),
        (2.0 ** -126, 0x0080),  # smallest normal
        (2.0 ** -133, 0x0001),  # smallest subnormal
        (2.0 ** -134, 0x0000),  # tie -> even (zero)
        (3 * 2.0 ** -134, 0x0002),  # tie -> even (two steps)
        (2.0 ** -134 + 2.0 ** -160, 0x0001),
        (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
    ]
    got = orc.f64_to_bf16(np.array([v for v, _ in cases]))
    for (v, want), g in zip(cases, got):
        assert int(g) == want, (v, hex(int(g)), hex(want))
    assert int(orc.f64_to_bf16([float("nan")])[0]) & 0x7FC0 == 0x7FC0


def test_latent_down_integer_inputs_exact(orc):
    # small integers: every product and partial sum is an exact integer, so the
    # FP64 sum is the true sum; its BF16 is the integer rounded once
    rng = np.random.default_rng(3)
    T, L, H = 5, 40, 96
    xv = rng.integers(-8, 9, (T, H)).astype(np.float32)
    wv = rng.integers(-8, 9, (L, H)).astype(np.float32)
    ref, b, lo, hi = orc.latent_down(synth.f32_to_bf16_bits(xv), synth.f32_to_bf16_bits(wv))
    exact = xv.astype(np.int64) @ wv.astype(np.int64).T
    assert np.array_equal(ref, exact.astype(np.float64))
    want = np.array([[round_fraction_to_bf16(Fraction(int(v))) for v in row] for row in exact], np.uint16)
    assert np.array_equal(b, want)
    # the tolerance bounds bracket the exact rounding
    f = lambda bits: synth.bf16_bits_to_f32(bits).astype(np.float64)
    assert np.all(f(lo) <= f(b)) and np.all(f(b) <= f(hi))

"""Pins of the oracle's BF16 conversions against the format's definition, by
brute force over exact rationals."""
import random
from fractions import Fraction

import numpy as np

from helpers import bf16_value, bits_from_f32, f32_from_bits, round_fraction_to_bf16


def test_bf16_decode_all_patterns(orc):
    # every BF16 pattern decodes to the FP32 with the same upper 16 bits
    for b in list(range(0, 0x10000, 7)) + [0x0000, 0x8000, 0x0001, 0x7F7F, 0xFF7F, 0x7F80]:
        v = orc.bf16_to_f32(b)
        assert bits_from_f32(v) == (b << 16) or (v != v)


def test_bf16_known_values(orc):
    assert orc.f32_to_bf16(1.0) == 0x3F80
    assert orc.f32_to_bf16(-2.0) == 0xC000
    assert orc.f32_to_bf16(1.0 + 2.0 ** -8) == 0x3F80  # tie -> even
    assert orc.f32_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82  # tie -> even (up)
    assert orc.f32_to_bf16(float("inf")) == 0x7F80
    assert orc.f32_to_bf16(f32_from_bits(0x7F7FFFFF)) == 0x7F80  # rounds past max
    nan = orc.f32_to_bf16(float("nan"))
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F)


def test_bf16_round_matches_exact_rational(orc):
    rnd = random.Random(1)
    for _ in range(3000):
        u = rnd.getrandbits(32)
        if ((u >> 23) & 0xFF) in (0, 0xFF, 0xFE):  # keep to the normal range
            continue
        f = f32_from_bits(u)
        assert orc.f32_to_bf16(f) == round_fraction_to_bf16(Fraction(f))

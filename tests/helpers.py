"""Test-side helpers: golden-file parsing and independent exact arithmetic
(Python Fractions) used to pin the oracle. Nothing here is shared with the oracle
or with the CUDA library."""
from __future__ import annotations

import os
import struct
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def expand_list(text, conv=float):
    """'0*7,0.25' -> [0]*7 + [0.25]."""
    out = []
    for item in text.split(","):
        if "*" in item:
            v, n = item.split("*")
            out += [conv(v)] * int(n)
        else:
            out.append(conv(item))
    return out


def f32_from_bits(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def bits_from_f32(f: float) -> int:
    return struct.unpack("<I", struct.pack("<f", f))[0]


def bf16_value(b: int) -> float:
    return f32_from_bits((b & 0xFFFF) << 16)


def round_fraction_to_bf16(q: Fraction) -> int:
    """Exact value -> BF16 bits, round to nearest even, by brute-force comparison of
    the two neighbouring BF16 values (finite, normal range only)."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    # find exponent e with 2^e <= a < 2^(e+1)
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    step = Fraction(2) ** (e - 7)
    m = a / step  # in [128, 256)
    lo = int(m)
    d = m - lo
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    val = lo * step
    bits = bits_from_f32(float(val)) >> 16
    assert Fraction(bf16_value(bits)) == val
    return sign | bits


def e4m3_grid():
    """The 127 nonnegative finite E4M3 values and their codes, from the format's
    definition (bias 7, 3 mantissa bits, S.1111.111 NaN)."""
    vals, codes = [], []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals.append(v)
        codes.append(c)
    return vals, codes


def e4m3_bruteforce(values: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code (ties to the even code), |y| > 448 saturating, by a
    search over all finite E4M3 values. ``values`` are float64, exactly the inputs."""
    vals, codes = e4m3_grid()
    grid = np.array([float(v) for v in vals])
    a = np.abs(values)
    sign = np.where(np.signbit(values), 0x80, 0x00)
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equal-distance candidates (ties) take the even code
    code_arr = np.array(codes)
    even = (code_arr % 2 == 0)[None, :]
    pick_even = cand & even
    has_even = pick_even.any(axis=1)
    idx = np.where(has_even, pick_even.argmax(axis=1), cand.argmax(axis=1))
    out = code_arr[idx]
    out = np.where(a > 448.0, 0x7E, out)
    return (out | sign).astype(np.uint8)

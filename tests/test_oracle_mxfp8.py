"""Pins of the oracle's MXFP8 quantisation (OCP MX: blocks of 32, E8M0 scale
2^(floor(log2 amax) - 8), E4M3 elements, round to nearest even, saturating) against
the formats' definitions, a brute-force nearest-value search and round-trip bounds."""
import numpy as np
import pytest

import synth
from helpers import e4m3_bruteforce, golden_lines


@pytest.mark.parametrize("row", list(golden_lines("e4m3_codes.txt")), ids=lambda r: "_".join(r[:3]))
def test_e4m3_golden(orc, row):
    m, _, e, code = row
    y = float(m) * 2.0 ** int(e)
    if m.startswith("-") and float(m) == 0:
        y = -0.0
    assert orc.e4m3_encode(y) == int(code, 16)


def test_e4m3_decode_definition(orc):
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0xFE) == -448.0
    assert np.isnan(orc.e4m3_decode(0x7F)) and np.isnan(orc.e4m3_decode(0xFF))


@pytest.mark.parametrize("row", list(golden_lines("mxfp8_blocks.txt")), ids=lambda r: r[0])
def test_block_golden(orc, row):
    v, sb, code = (int(t, 16) for t in row)
    x = np.full((1, 32), v, np.uint16)
    q, s = orc.mxfp8_quantize(x)
    assert s[0, 0] == sb
    assert np.all(q == code)


def _all_finite_bf16():
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(b)
    return b[np.isfinite(f)]


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x4B00, 0x0080, 0x7F00, 0x2000, 0x0001])
def test_exhaustive_against_bruteforce(orc, amax_bits):
    """Every finite BF16 value whose magnitude is <= a fixed block maximum, encoded in
    blocks led by that maximum, against the brute-force nearest E4M3 code."""
    allb = _all_finite_bf16()
    amax = float(synth.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0])
    vals = allb[np.abs(synth.bf16_bits_to_f32(allb)) <= amax]
    nblk = -(-vals.size // 31)
    body = np.resize(vals, nblk * 31).reshape(nblk, 31)
    x = np.concatenate([np.full((nblk, 1), amax_bits, np.uint16), body], axis=1).reshape(1, -1)
    q, s = orc.mxfp8_quantize(x)
    # scale from the definition, with floor(log2) taken in exact float64
    fl = int(np.floor(np.log2(amax)))
    if 2.0 ** fl > amax:
        fl -= 1
    se = min(max(fl - 8, -127), 127)
    assert np.all(s == se + 127)
    y = synth.bf16_bits_to_f32(x.reshape(-1)).astype(np.float64) * 2.0 ** (-se)
    np.testing.assert_array_equal(q.reshape(-1), e4m3_bruteforce(y))


def test_round_trip_bounds(orc):
    rng = np.random.default_rng(4)
    f = (rng.normal(0, 1, (16, 1024)) * np.exp2(rng.integers(-40, 40, (16, 1)))).astype(np.float32)
    x = synth.f32_to_bf16_bits(f)
    q, s = orc.mxfp8_quantize(x)
    v = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(16, 32, 32)
    X = np.exp2(s.astype(np.float64) - 127)[:, :, None]
    deq = np.vectorize(orc.e4m3_decode)(q).astype(np.float64).reshape(16, 32, 32) * X
    amax = np.abs(v).max(axis=2, keepdims=True)
    r = amax / X
    assert np.all((r >= 256) & (r < 512))
    y = np.abs(v) / X
    normal = y >= 2.0 ** -6
    err = np.abs(deq - v)
    assert np.all(err[normal & (y <= 448)] <= 2.0 ** -4 * np.abs(v)[normal & (y <= 448)])
    sub = ~normal
    assert np.all(err[sub] <= (2.0 ** -10 * X.repeat(32, axis=2))[sub])
    sat = y > 448
    assert np.all(np.abs(np.abs(v) - 448 * X.repeat(32, axis=2))[sat] < (64 * X.repeat(32, axis=2))[sat])


def test_grid_values_round_trip_exactly(orc):
    # values already on the E4M3 grid times the block scale are reproduced exactly
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, (4, 64)).astype(np.uint8)
    codes[:, ::32] = 0x78  # amax 256 * 2^k in every block -> scale exponent k
    k = -3
    vals = np.vectorize(orc.e4m3_decode)(codes) * 2.0 ** k
    x = synth.f32_to_bf16_bits(vals.astype(np.float32))
    q, s = orc.mxfp8_quantize(x)
    assert np.all(s == k + 127)
    np.testing.assert_array_equal(q, codes)


def test_nan_inf_blocks(orc):
    x = np.full((1, 64), 0x3F80, np.uint16)
    x[0, 3] = 0x7F80  # +inf in block 0
    x[0, 40] = 0x7FC0  # NaN in block 1
    q, s = orc.mxfp8_quantize(x)
    assert s.tolist() == [[0xFF, 0xFF]]
    assert np.all(q == 0x7F)


# --- the round-up scale rule (rule 1): the smallest power of two X with amax / X <= 448


def test_ceil_rule_closed_forms(orc):
    # amax 448: the OCP scale already fits (1.75 * 2^8), scale byte 127, code 0x7E;
    # amax 450 (significand above 1.75): one step up, 450 / 2 = 225 -> E4M3 224 = 0x76;
    # amax -480: -240 = 0xF7; the floor rule saturates both to 448 (0x7E / 0xFE)
    x = synth.f32_to_bf16_bits(np.array([[448.0] + [0.5] * 31, [450.0] + [1.0] * 31, [-480.0] + [3.0] * 31],
                                        np.float32))
    q, s = orc.mxfp8_quantize(x, rule=1)
    assert s.ravel().tolist() == [127, 128, 128]
    assert q[:, 0].tolist() == [0x7E, 0x76, 0xF7]
    q0, s0 = orc.mxfp8_quantize(x, rule=0)
    assert s0.ravel().tolist() == [127, 127, 127] and q0[:, 0].tolist() == [0x7E, 0x7E, 0xFE]


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x3FE0, 0x3FE1, 0x43E0, 0x43E1, 0x7F7F, 0x0080, 0x0001, 0x0007])
def test_ceil_rule_exhaustive_against_bruteforce(orc, amax_bits):
    """As the floor-rule check, with the scale from the definition: the smallest integer
    k with 448 * 2^k >= amax (exact in float64), then clamped; every element is the
    nearest E4M3 code of v / 2^k and none saturates."""
    allb = _all_finite_bf16()
    amax = float(synth.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0])
    vals = allb[np.abs(synth.bf16_bits_to_f32(allb)) <= amax]
    nblk = -(-vals.size // 31)
    body = np.resize(vals, nblk * 31).reshape(nblk, 31)
    x = np.concatenate([np.full((nblk, 1), amax_bits, np.uint16), body], axis=1).reshape(1, -1)
    q, s = orc.mxfp8_quantize(x, rule=1)
    k = -200
    while 448.0 * 2.0 ** k < amax:
        k += 1
    se = min(max(k, -127), 127)
    assert np.all(s == se + 127)
    y = synth.bf16_bits_to_f32(x.reshape(-1)).astype(np.float64) * 2.0 ** (-se)
    assert np.all(np.abs(y) <= 448.0)
    np.testing.assert_array_equal(q.reshape(-1), e4m3_bruteforce(y))


def test_ceil_rule_matches_floor_below_1_75(orc):
    # block maxima whose significand is at most 1.75 give the same scale and codes
    rng = np.random.default_rng(9)
    f = (rng.uniform(-1, 1, (32, 32)) * np.exp2(rng.integers(-30, 30, (32, 1)))).astype(np.float32)
    f[:, 0] = (np.where(np.arange(32) % 2, 1.75, 1.0 + rng.uniform(0, 0.75, 32)) * np.exp2(rng.integers(-30, 30, 32))).astype(np.float32)
    x = synth.f32_to_bf16_bits(f)
    amax_sig = np.abs(synth.bf16_bits_to_f32(x)).max(axis=1)
    amax_sig = amax_sig / np.exp2(np.floor(np.log2(amax_sig)))
    keep = amax_sig <= 1.75
    q0, s0 = orc.mxfp8_quantize(x, rule=0)
    q1, s1 = orc.mxfp8_quantize(x, rule=1)
    assert keep.sum() >= 16
    np.testing.assert_array_equal(s1[keep], s0[keep])
    np.testing.assert_array_equal(q1[keep], q0[keep])


# ---------------------------------------------------------------------------
# The tcgen05 block-scaling tile layout of the scales (128 rows x 4 scale columns per
# 512-byte tile; inside a tile, row r and column c at 16 * (r % 32) + 4 * (r // 32) + c;
# tiles ordered row tile by row tile; padding 0).

def test_tcgen05_scale_layout_closed_forms(orc):
    """Positions worked out by hand for a 130 x 5 scale matrix (two row tiles, two
    column tiles: 2048 bytes), each scale byte distinct so that its position shows."""
    rows, nsc = 130, 5
    sc = (np.arange(rows * nsc) % 251 + 1).astype(np.uint8).reshape(rows, nsc)  # never 0
    t = orc.mxfp8_scales_tcgen05(sc)
    assert t.size == 2048
    expect = {  # (row, scale column) -> byte offset
        (0, 0): 0, (1, 0): 16, (31, 0): 496, (32, 0): 4, (33, 1): 21, (64, 2): 10, (96, 3): 15,
        (127, 3): 511, (0, 4): 512, (5, 4): 592, (100, 4): 512 + 16 * 4 + 4 * 3, (128, 0): 1024,
        (129, 3): 1024 + 16 + 3, (128, 4): 1536, (129, 4): 1552,
    }
    for (r, c), off in expect.items():
        assert t[off] == sc[r, c], (r, c, off)


def test_tcgen05_scale_layout_covers_every_scale_once(orc):
    """Every scale lands in its own byte; the remaining bytes (padding rows and columns)
    are 0; the layout reads back to the row-major matrix."""
    for rows, nsc in ((1, 1), (127, 4), (128, 4), (129, 7), (300, 112), (1020, 112)):
        sc = np.random.default_rng(rows * 1000 + nsc).integers(1, 256, (rows, nsc)).astype(np.uint8)
        t = orc.mxfp8_scales_tcgen05(sc)
        rt, ct = -(-rows // 128), -(-nsc // 4)
        assert t.size == rt * ct * 512
        r, c = np.meshgrid(np.arange(rows), np.arange(nsc), indexing="ij")
        off = ((r // 128) * ct + c // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + c % 4
        assert np.unique(off).size == rows * nsc
        np.testing.assert_array_equal(t[off], sc)
        pad = np.ones(t.size, bool)
        pad[off.ravel()] = False
        assert not t[pad].any()
        assert pad.sum() == t.size - rows * nsc

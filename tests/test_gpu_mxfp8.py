"""MXFP8 quantisation on the GPU against the oracle, bit for bit (OCP MX reading of
the pages' MXFP8 activations)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_dev, host

pytestmark = pytest.mark.gpu


def _compare(moe, orc, x, rule=0):
    q, s = moe.mxfp8_quantize_rows(bf16_dev(x), scale_rule=rule)
    torch.cuda.synchronize()
    eq, es = orc.mxfp8_quantize(x, rule=rule)
    np.testing.assert_array_equal(host(s), es)
    np.testing.assert_array_equal(host(q), eq)


@pytest.mark.parametrize("rows,cols", [(1, 3584), (8, 3584), (1020, 3584), (4096, 3584), (3, 32), (7, 96), (33, 288), (5, 7168)])
def test_normal_rows(moe, orc, rows, cols):
    _compare(moe, orc, synth.normal_bf16(30 + rows, 5, (rows, cols)))


def test_wide_dynamic_range(moe, orc):
    rng = np.random.default_rng(31)
    f = (rng.normal(0, 1, (64, 1024)) * np.exp2(rng.integers(-140, 128, (64, 1)))).astype(np.float32)
    f[np.isinf(f)] = 0
    _compare(moe, orc, synth.f32_to_bf16_bits(f))


def test_special_blocks(moe, orc):
    x = synth.normal_bf16(32, 5, (4, 256))
    x[0, 0:32] = 0
    x[0, 32:64] = 0x8000
    x[1, 0:32] = 0x0001
    x[1, 40] = 0x7F80          # +inf
    x[2, 70] = 0x7FC0          # NaN
    x[2, 100] = 0xFF80         # -inf
    x[3, 0:32] = 0x7F7F        # max finite
    x[3, 32:64] = np.arange(32, dtype=np.uint16) | 0x8000  # negative subnormals
    _compare(moe, orc, x)


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x4B00, 0x0080, 0x7F00, 0x2000, 0x0001, 0x43E0])
def test_exhaustive_patterns(moe, orc, amax_bits):
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(b)
    amax = synth.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0]
    vals = b[np.isfinite(f) & (np.abs(f) <= amax)]
    n = -(-vals.size // 31)
    body = np.resize(vals, n * 31).reshape(n, 31)
    x = np.concatenate([np.full((n, 1), amax_bits, np.uint16), body], axis=1)
    pad = (-x.shape[0]) % 4
    x = np.concatenate([x, np.zeros((pad, 32), np.uint16)]).reshape(-1, 128)
    _compare(moe, orc, x)


# --- the round-up scale rule (MXFP8_SCALE_CEIL): no element saturates


@pytest.mark.parametrize("rows,cols", [(8, 3584), (1020, 3584), (33, 288)])
def test_ceil_rule_normal_rows(moe, orc, rows, cols):
    _compare(moe, orc, synth.normal_bf16(60 + rows, 5, (rows, cols)), rule=moe.MXFP8_SCALE_CEIL)


def test_ceil_rule_special_and_wide_range(moe, orc):
    rng = np.random.default_rng(61)
    f = (rng.normal(0, 1, (64, 1024)) * np.exp2(rng.integers(-140, 128, (64, 1)))).astype(np.float32)
    f[np.isinf(f)] = 0
    x = synth.f32_to_bf16_bits(f)
    x[0, 0:32] = 0
    x[1, 40] = 0x7F80
    x[2, 70] = 0x7FC0
    x[3, 0:32] = 0x7F7F
    x[4, 32:64] = np.arange(32, dtype=np.uint16) | 0x8000
    _compare(moe, orc, x, rule=moe.MXFP8_SCALE_CEIL)


@pytest.mark.parametrize("amax_bits", [0x3FE0, 0x3FE1, 0x43E1, 0x7F7F, 0x0001, 0x0007])
def test_ceil_rule_exhaustive_patterns(moe, orc, amax_bits):
    """Block maxima at and just above a significand of 1.75 (the rules' boundary),
    the largest finite value and subnormals; every finite BF16 at most the maximum."""
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(b)
    amax = synth.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0]
    vals = b[np.isfinite(f) & (np.abs(f) <= amax)]
    n = -(-vals.size // 31)
    body = np.resize(vals, n * 31).reshape(n, 31)
    x = np.concatenate([np.full((n, 1), amax_bits, np.uint16), body], axis=1)
    pad = (-x.shape[0]) % 4
    x = np.concatenate([x, np.zeros((pad, 32), np.uint16)]).reshape(-1, 128)
    _compare(moe, orc, x, rule=moe.MXFP8_SCALE_CEIL)


def test_bad_rule_rejected(moe):
    x = bf16_dev(synth.normal_bf16(1, 5, (2, 64)))
    with pytest.raises(moe.MoeError):
        moe.mxfp8_quantize_rows(x, scale_rule=2)


@pytest.mark.parametrize("rows,cols", [(1, 32), (1, 3584), (127, 96), (128, 128), (129, 3584), (1020, 3584),
                                       (4096, 3584), (33, 288), (5, 7168)])
@pytest.mark.parametrize("rule", [0, 1])
def test_tcgen05_scale_layout(moe, orc, rows, cols, rule):
    """Scales in the tcgen05 block-scaling tile layout, bit for bit against the oracle's
    layout of its own scales (padding bytes 0); the E4M3 bytes equal the row-major
    call's."""
    x = synth.latent_rows(rows, seed=rows + cols)[:, :cols] if cols <= 3584 else synth.normal_bf16(5, 9, (rows, cols))
    xd = bf16_dev(np.ascontiguousarray(x))
    n = moe.mxfp8_tcgen05_scales_bytes(rows, cols)
    sc = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")  # padding must be written
    q, sc = moe.mxfp8_quantize_rows_tcgen05(xd, scales=sc, scale_rule=rule)
    torch.cuda.synchronize()
    eq, es = orc.mxfp8_quantize(np.ascontiguousarray(x), rule)
    np.testing.assert_array_equal(host(q), eq)
    np.testing.assert_array_equal(host(sc), orc.mxfp8_scales_tcgen05(es))

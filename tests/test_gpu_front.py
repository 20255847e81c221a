"""Front projection on the GPU (router logits FP32 + latent down projection BF16 in one
tensor-core launch; the wide page's front GEMM over the router rows and the latent
down rows, module docstring) against the oracle's FP64 sums: bit-exact on integer
inputs, otherwise logits within 1e-5 * sum|x w| and the latent a BF16 rounding of a
value within that bound."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_bits, bf16_dev, host

pytestmark = pytest.mark.gpu


def _ints(seed, shape, lo=-8, hi=8):
    v = np.random.default_rng(seed).integers(lo, hi + 1, size=shape).astype(np.float32)
    return synth.f32_to_bf16_bits(v)


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# (T, E, L, H): the decode shapes, ragged tiles (E, L not multiples of 128, T not a
# multiple of the token tile), one-tile and many-wave grids
SHAPES = [(1, 896, 3584, 7168), (8, 896, 3584, 7168), (17, 130, 200, 1024), (64, 896, 3584, 7168),
          (100, 7, 300, 512), (300, 256, 129, 2048), (1020, 128, 640, 1024)]


@pytest.mark.parametrize("T,E,L,H", SHAPES)
def test_integer_exact(moe, orc, T, E, L, H):
    x, wr, wd = _ints(T, (T, H)), _ints(E + 1, (E, H)), _ints(L + 2, (L, H))
    logits, latent = moe.front_projection(bf16_dev(x), bf16_dev(wr), bf16_dev(wd))
    exp_l, _ = orc.router_logits(x, wr)
    np.testing.assert_array_equal(host(logits).astype(np.float64), exp_l)
    _, exp_b, _, _ = orc.latent_down(x, wd)
    np.testing.assert_array_equal(bf16_bits(latent), exp_b)
    assert moe.device_error(clear=True) == 0


@pytest.mark.parametrize("T,E,L,H", [(8, 896, 3584, 7168), (33, 96, 200, 640), (257, 130, 384, 2048)])
def test_random_within_tolerance(moe, orc, T, E, L, H):
    x = synth.normal_bf16(50 + T, 1, (T, H))
    wr = synth.normal_bf16(50 + E, 2, (E, H), 0.02)
    wd = synth.normal_bf16(50 + L, 10, (L, H), 0.02)
    logits, latent = moe.front_projection(bf16_dev(x), bf16_dev(wr), bf16_dev(wd))
    exp_l, ab = orc.router_logits(x, wr)
    assert np.all(np.abs(host(logits).astype(np.float64) - exp_l) <= 1e-5 * ab)
    _, _, lo, hi = orc.latent_down(x, wd)
    g = _f(bf16_bits(latent))
    assert np.all(_f(lo) <= g) and np.all(g <= _f(hi))


@pytest.mark.parametrize("T", [64, 1020, 4096])
def test_full_size_sampled(moe, orc, T):
    """The decode shapes (896 router rows, 3584 latent rows, hidden 7168): 3000 sampled
    logits and 3000 sampled latent values against FP64."""
    x = synth.hidden_rows(T)
    wr, wd = synth.router_weight(), synth.latent_down_weight()
    logits, latent = moe.front_projection(bf16_dev(x), bf16_dev(wr), bf16_dev(wd))
    logits, latent = host(logits).astype(np.float64), bf16_bits(latent)
    rng = np.random.default_rng(T)
    t = rng.integers(0, T, 3000).astype(np.int32)
    t[:10] = T - 1  # the ragged last token tile
    e = rng.integers(0, 896, 3000).astype(np.int32)
    exp, ab = orc.router_logits_sampled(x, wr, t, e)
    assert np.all(np.abs(logits[t, e] - exp) <= 1e-5 * ab)
    l = rng.integers(0, 3584, 3000).astype(np.int32)
    ref, ab = orc.router_logits_sampled(x, wd, t, l)
    lo, hi = orc.f64_to_bf16(ref - 1e-5 * ab), orc.f64_to_bf16(ref + 1e-5 * ab)
    g = _f(latent[t, l])
    assert np.all(_f(lo) <= g) and np.all(g <= _f(hi))
    assert moe.device_error(clear=True) == 0


def test_deterministic_and_logits_match_router_tolerance(moe):
    x = bf16_dev(synth.hidden_rows(300))
    wr, wd = bf16_dev(synth.router_weight()), bf16_dev(synth.latent_down_weight())
    a = moe.front_projection(x, wr, wd)
    b = moe.front_projection(x, wr, wd)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    r = moe.router_logits(x, wr)
    assert torch.allclose(a[0], r, rtol=0, atol=1e-3)
    assert moe.device_error(clear=True) == 0

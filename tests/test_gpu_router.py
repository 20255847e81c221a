"""Router logits on the GPU (both kernel families) against the oracle's FP64 sums:
exact on integer inputs, within 1e-5 * sum|x w| otherwise (DEP page, EpMoeLayer:
FP32-output router projection; stock_order: mm(x, gate^T) with an FP32 output)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_dev, host

pytestmark = pytest.mark.gpu

ALGOS = {"simt": 1, "tcgen05": 2}


def _ints(seed, shape, lo=-8, hi=8):
    v = np.random.default_rng(seed).integers(lo, hi + 1, size=shape).astype(np.float32)
    return synth.f32_to_bf16_bits(v)


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("T,E,H", [(1, 896, 7168), (2, 896, 7168), (3, 896, 7168), (5, 896, 7168), (8, 896, 7168),
                                   (4, 7, 72), (6, 1001, 232), (17, 128, 1024), (64, 896, 7168), (100, 200, 512),
                                   (300, 896, 1024), (1020, 256, 7168),
                                   # plan branches at the full gate: 64-column tiles (T = 128), 128-column
                                   # tiles (T = 256); CTA pairs with a padding half and a split (T = 2048)
                                   (128, 896, 7168), (256, 896, 7168), (2048, 896, 1024)])
def test_integer_exact(moe, orc, algo, T, E, H):
    x, w = _ints(T, (T, H)), _ints(E + 1, (E, H))
    got = host(moe.router_logits(bf16_dev(x), bf16_dev(w), algo=ALGOS[algo]))
    exp, _ = orc.router_logits(x, w)
    np.testing.assert_array_equal(got.astype(np.float64), exp)


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("T,E,H", [(8, 896, 7168), (33, 96, 200), (64, 896, 7168), (257, 130, 2048), (5, 1, 64)])
def test_random_within_tolerance(moe, orc, algo, T, E, H):
    x = synth.normal_bf16(40 + T, 1, (T, H))
    w = synth.normal_bf16(40 + E, 2, (E, H), 0.02)
    got = host(moe.router_logits(bf16_dev(x), bf16_dev(w), algo=ALGOS[algo])).astype(np.float64)
    exp, ab = orc.router_logits(x, w)
    assert np.all(np.abs(got - exp) <= 1e-5 * ab)


@pytest.mark.parametrize("T", [1, 16, 64, 256, 1020, 2048, 4096])
def test_full_size_every_element(moe, orc, T):
    """The public call (its own plan at each T: 16-CTA clusters of narrow tiles, 64- and
    128-column tiles, 5-CTA clusters of 256-column tiles at T = 1020, CTA pairs) at the
    full decode shapes (896 x 7168 gate): every logit against FP64."""
    x = synth.hidden_rows(T)
    w = synth.router_weight()
    got = host(moe.router_logits(bf16_dev(x), bf16_dev(w))).astype(np.float64)
    exp, ab = orc.router_logits(x, w)
    bad = np.argwhere(np.abs(got - exp) > 1e-5 * ab)
    assert bad.size == 0, f"{len(bad)} logits out of tolerance, first at (t, e) = {tuple(bad[0])}"


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("T", [1020, 2048, 4096])
def test_full_size_sampled(moe, orc, algo, T):
    """Each kernel family forced at the full decode shapes: 3000 sampled outputs against
    FP64 (a quick check; the public call is compared element by element above)."""
    x = synth.hidden_rows(T)
    w = synth.router_weight()
    got = host(moe.router_logits(bf16_dev(x), bf16_dev(w), algo=ALGOS[algo])).astype(np.float64)
    rng = np.random.default_rng(T)
    t = rng.integers(0, T, 3000).astype(np.int32)
    e = rng.integers(0, 896, 3000).astype(np.int32)
    t[:10] = T - 1  # the ragged last token tile
    exp, ab = orc.router_logits_sampled(x, w, t, e)
    assert np.all(np.abs(got[t, e] - exp) <= 1e-5 * ab)


@pytest.mark.parametrize("algo", list(ALGOS))
def test_deterministic(moe, algo):
    x = bf16_dev(synth.hidden_rows(300))
    w = bf16_dev(synth.router_weight())
    a = moe.router_logits(x, w, algo=ALGOS[algo])
    b = moe.router_logits(x, w, algo=ALGOS[algo])
    assert torch.equal(a, b)
    assert moe.device_error(clear=True) == 0

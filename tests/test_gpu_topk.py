"""Sigmoid + bias top-K on the GPU against the oracle (which consumes the same
logits): ids, FP32 and BF16 weights bit for bit (DEP page, EpMoeLayer.topk; wide
page, WideRoute an exact top-16 with renormalised weights)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_bits, dev, host

pytestmark = pytest.mark.gpu


def _compare(moe, orc, logits, bias, K, renorm=True, scale=1.0):
    ids, w, wb = moe.topk_route(dev(logits), None if bias is None else dev(bias), K, renorm, scale)
    torch.cuda.synchronize()
    eids, ew, ewb = orc.topk_route(logits, bias, K, renorm, scale)
    np.testing.assert_array_equal(host(ids), eids)
    # a NaN weight (a token with NaN scores among its picks) may carry any NaN payload;
    # every other weight bit for bit
    gw, gb = host(w), bf16_bits(wb)
    nan = np.isnan(ew)
    np.testing.assert_array_equal(np.isnan(gw), nan)
    np.testing.assert_array_equal(gw.view(np.uint32)[~nan], ew.view(np.uint32)[~nan])
    np.testing.assert_array_equal((gb & 0x7FFF) > 0x7F80, nan)
    np.testing.assert_array_equal(gb[~nan], ewb[~nan])


@pytest.mark.parametrize("T", [1, 8, 64, 1020, 4096])
def test_decode_shapes(moe, orc, T):
    logits = synth.normal_f32(20 + T, 1, (T, 896), 1.7)
    _compare(moe, orc, logits, synth.correction_bias(), 16)


def test_skew_bias(moe, orc):
    logits = synth.normal_f32(21, 1, (512, 896), 1.7)
    _compare(moe, orc, logits, synth.skew_bias(), 16)


@pytest.mark.parametrize("E,K", [(1, 1), (16, 16), (33, 4), (127, 16), (128, 32), (129, 8), (1000, 16), (1024, 32), (896, 1),
                                 (1025, 16), (2048, 32), (4096, 16)])
@pytest.mark.parametrize("T", [45, 300])
def test_expert_counts(moe, orc, E, K, T):
    """T = 45 takes the CTA-per-token body; T = 300 the warp-per-token body where it
    applies (E % 4 == 0 and E <= 1024), else the CTA body; E > 1024 up to 4096."""
    logits = synth.normal_f32(22 + E, 1, (T, E), 2.0)
    _compare(moe, orc, logits, synth.normal_f32(22 + E, 3, (E,), 0.05), K)


@pytest.mark.parametrize("renorm,scale,bias", [(False, 1.0, True), (True, 2.5, True), (False, 0.5, False), (True, 1.0, False)])
@pytest.mark.parametrize("T", [77, 300])
def test_flags(moe, orc, renorm, scale, bias, T):
    logits = synth.normal_f32(23, 1, (T, 896), 1.7)
    _compare(moe, orc, logits, synth.correction_bias() if bias else None, 16, renorm, scale)


@pytest.mark.parametrize("T", [64, 256])
def test_heavy_ties_fallback(moe, orc, T):
    """Saturated sigmoids (exactly 0 or 1) and a coarse bias grid: many equal keys, more
    than 64 candidates above the bound, so the token takes the argmax-rounds path (CTA
    body at T = 64, warp body at T = 256)."""
    rng = np.random.default_rng(24)
    logits = rng.choice(np.array([-100.0, 20.0, 0.0], np.float32), size=(T, 896)).astype(np.float32)
    bias = (rng.integers(-2, 3, 896) / 16.0).astype(np.float32)
    _compare(moe, orc, logits, bias, 16)
    _compare(moe, orc, np.zeros((T, 896), np.float32), None, 16)  # every key equal


@pytest.mark.parametrize("T", [32, 256])
def test_special_values(moe, orc, T):
    """Infinities, the sigmoid's clamp points, subnormals and NaN logits (a token whose
    scores are mostly NaN has fewer numbers than candidates: the all-exact path)."""
    rng = np.random.default_rng(25)
    logits = rng.normal(0, 30, (T, 256)).astype(np.float32)
    logits[:, ::7] = np.float32(np.inf)
    logits[:, 3::11] = -np.float32(np.inf)
    logits[:, 5::13] = 17.5
    logits[:, 6::17] = -88.5
    logits[:, 1::19] = 1e-40  # subnormal input
    logits[1, ::3] = np.float32(np.nan)
    logits[2, :250] = np.float32(np.nan)  # 6 numbers for K = 16: NaN keys rank last
    logits[3, 7] = np.float32(np.nan)
    _compare(moe, orc, logits, synth.normal_f32(25, 3, (256,), 0.01), 16)


@pytest.mark.slow
def test_sigmoid_exhaustive(moe, orc):
    """The specified sigmoid, GPU against oracle, for every FP32 bit pattern (E = K = 1,
    no renormalisation: the weight is the score)."""
    chunk = 1 << 26
    threads = os.cpu_count() or 4
    for start in range(0, 1 << 32, chunk):
        u = (np.arange(start, start + chunk, dtype=np.uint64)).astype(np.uint32)
        x = u.view(np.float32).reshape(chunk, 1)
        _, w, _ = moe.topk_route(dev(x), None, 1, False, 1.0, want_bf16=False)
        got = host(w).reshape(-1)
        parts = np.array_split(x.reshape(-1), threads)
        with ThreadPoolExecutor(threads) as ex:
            exp = np.concatenate(list(ex.map(orc.sigmoid, parts)))
        same = (got.view(np.uint32) == exp.view(np.uint32)) | (np.isnan(got) & np.isnan(exp))
        assert same.all(), f"mismatch at 0x{int(u[~same][0]):08x}"


@pytest.mark.parametrize("T,rows", [(1020, 1020), (8, 8), (37, 5), (3, 0)])
def test_fused_route_quantize(moe, orc, T, rows):
    """moe_topk_route_quantize == moe_topk_route + mxfp8_quantize_rows, bit for bit."""
    logits = synth.normal_f32(26 + T, 1, (T, 896), 1.7)
    bias = synth.correction_bias()
    latent = synth.latent_rows(max(rows, 1))[:rows]
    from gpu_helpers import bf16_dev
    ids, w, wb, q, sc = moe.topk_route_quantize(dev(logits), dev(bias), 16, bf16_dev(latent))
    torch.cuda.synchronize()
    eids, ew, ewb = orc.topk_route(logits, bias, 16)
    np.testing.assert_array_equal(host(ids), eids)
    np.testing.assert_array_equal(host(w).view(np.uint32), ew.view(np.uint32))
    np.testing.assert_array_equal(bf16_bits(wb), ewb)
    if rows:
        eq, es = orc.mxfp8_quantize(latent)
        np.testing.assert_array_equal(host(q), eq)
        np.testing.assert_array_equal(host(sc), es)

"""The whole routing-and-combine step on one stream (router -> top-16 with the MXFP8
latent in the same launch -> lists -> Finalize, programmatic dependent launches between
the kernels) against the oracle, at the decode shapes: every logit within tolerance, everything else bit for
bit, with the oracle's top-k consuming the GPU's logits."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_bits, bf16_dev, dev, host

pytestmark = pytest.mark.gpu


def _check_chain(moe, orc, T, skew=False, graph=False):
    d = synth.chain_inputs(T, skew=skew)
    x, w, bias, latent, rows = bf16_dev(d["x"]), bf16_dev(d["w"]), dev(d["bias"]), bf16_dev(d["latent"]), bf16_dev(d["rows"])
    rf = moe.RouteFinalize(T, synth.H, synth.L, synth.E, synth.K)
    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            rf.run(x, w, bias, latent, rows)  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rf.run(x, w, bias, latent, rows)
        rf.out.zero_()
        g.replay()
    else:
        rf.run(x, w, bias, latent, rows)
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 0
    logits = host(rf.logits)
    # R1: every logit against FP64 (the oracle splits the tokens over the host cores)
    exp, ab = orc.router_logits(d["x"], d["w"])
    err = np.abs(logits.astype(np.float64) - exp)
    bad = np.argwhere(err > 1e-5 * ab)
    assert bad.size == 0, f"{len(bad)} logits out of tolerance, first at (t, e) = {tuple(bad[0])}"
    # R2 top-16 from the GPU's logits
    ids, wf, wb = orc.topk_route(logits, d["bias"], synth.K)
    np.testing.assert_array_equal(host(rf.ids), ids)
    np.testing.assert_array_equal(host(rf.weights).view(np.uint32), wf.view(np.uint32))
    np.testing.assert_array_equal(bf16_bits(rf.weights_bf16), wb)
    # R3 lists
    off, pairs = orc.routing_lists(ids, synth.E)
    np.testing.assert_array_equal(host(rf.offsets), off)
    np.testing.assert_array_equal(host(rf.pairs), pairs)
    # R4 MXFP8
    q, sc = orc.mxfp8_quantize(d["latent"])
    np.testing.assert_array_equal(host(rf.q), q)
    np.testing.assert_array_equal(host(rf.scales), sc)
    # R5 Finalize with the BF16 weights (the wide path's Finalize input)
    np.testing.assert_array_equal(bf16_bits(rf.out), orc.finalize(d["rows"], wb, T, synth.K))


def test_tiny(moe, orc):
    _check_chain(moe, orc, 8)


def test_narrow(moe, orc):
    _check_chain(moe, orc, 64)


def test_wide(moe, orc):
    _check_chain(moe, orc, 1020)


@pytest.mark.parametrize("T", [1, 16, 64, 256, 1020, 4096])
def test_skew_sweep(moe, orc, T):
    """The skew sweep's token counts, Zipf(1.1) expert popularity."""
    _check_chain(moe, orc, T, skew=True)


def test_wide_in_cuda_graph(moe, orc):
    _check_chain(moe, orc, 1020, graph=True)


@pytest.mark.parametrize("T", [1, 4, 5, 8, 64, 100, 256, 1020, 2048, 4096])
def test_one_call_equals_four_calls(moe, T):
    """moe_route_finalize == the four calls it stands for, every output bit for bit --
    including the logits, which the one call's top-K launch sums from the router's
    split-K partials (every router plan: 16 splits of narrow tiles, 64- and 128-column
    tiles, 5-CTA clusters, CTA pairs with and without splits)."""
    d = synth.chain_inputs(T, seed=3)
    x, w, bias, latent, rows = bf16_dev(d["x"]), bf16_dev(d["w"]), dev(d["bias"]), bf16_dev(d["latent"]), bf16_dev(d["rows"])
    one = moe.RouteFinalize(T, synth.H, synth.L, synth.E, synth.K)
    one.run(x, w, bias, latent, rows)
    logits = moe.router_logits(x, w)
    ids, wf, wb, q, sc = moe.topk_route_quantize(logits, bias, synth.K, latent)
    off, pairs = moe.build_routing_lists(ids, synth.E)
    out = moe.finalize(rows, wb, T, synth.K)
    torch.cuda.synchronize()
    for name, b in (("logits", logits), ("ids", ids), ("weights", wf), ("weights_bf16", wb), ("offsets", off),
                    ("pairs", pairs), ("q", q), ("scales", sc), ("out", out)):
        a = getattr(one, name)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name


@pytest.mark.parametrize("T,H,L,E,K", [(37, 512, 256, 100, 8), (300, 1024, 512, 1000, 16), (9, 256, 64, 40, 3),
                                       (130, 768, 128, 2048, 16),
                                       # the lists CTAs stage the slot map in chunks (more blocks than fit)
                                       (1100, 512, 256, 100, 8), (400, 256, 64, 40, 3),
                                       # more chunks than their counts leave room for: the lists kernel
                                       (16300, 128, 64, 96, 8)])
def test_one_call_other_shapes(moe, orc, T, H, L, E, K):
    """The one-call step at shapes other than the decode layer's -- a last expert range
    of the lists shorter than 32 experts, K of 8, 3 and 16, E up to 2048 (the CTA-per-
    token top-K and the separate lists kernel), slot maps staged in several chunks, a
    batch too large for the lists CTAs (the separate lists kernel) -- equals the four
    calls bit for bit, and its lists the oracle's."""
    x = synth.normal_bf16(50 + T, 1, (T, H))
    w = synth.normal_bf16(50 + E, 2, (E, H), 0.02)
    bias = synth.normal_f32(50 + E, 3, (E,), 0.01)
    latent = synth.normal_bf16(50 + T, 5, (T, L))
    rows = synth.normal_bf16(50 + T, 4, (T * K, L))
    xd, wd, bd, ld, rd = bf16_dev(x), bf16_dev(w), dev(bias), bf16_dev(latent), bf16_dev(rows)
    one = moe.RouteFinalize(T, H, L, E, K)
    one.run(xd, wd, bd, ld, rd)
    logits = moe.router_logits(xd, wd)
    ids, wf, wb, q, sc = moe.topk_route_quantize(logits, bd, K, ld)
    off, pairs = moe.build_routing_lists(ids, E)
    out = moe.finalize(rd, wb, T, K)
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 0
    for name, b in (("logits", logits), ("ids", ids), ("weights", wf), ("weights_bf16", wb), ("offsets", off),
                    ("pairs", pairs), ("q", q), ("scales", sc), ("out", out)):
        a = getattr(one, name)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    eoff, epairs = orc.routing_lists(host(one.ids), E)
    np.testing.assert_array_equal(host(one.offsets), eoff)
    np.testing.assert_array_equal(host(one.pairs), epairs)

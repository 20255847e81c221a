"""Finalize with the RMSNorm epilogue on the GPU (ep page: rms_norm of the routed
latent, eps 1e-5; wide page: Finalize and the latent's RMSNorm): the routed latent bit
for bit against the oracle's Finalize, the normalised output a BF16 rounding of a value
within 2^-16 relative of the oracle's FP64 RMSNorm of that routed latent."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_bits, bf16_dev, dev

pytestmark = pytest.mark.gpu


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _check(moe, orc, rows, w, T, K, g, eps=1e-5, row_index=None, scale=1.0):
    wd = bf16_dev(w) if w.dtype == np.uint16 else dev(w)
    routed, out = moe.finalize_rmsnorm(bf16_dev(rows), wd, T, K, bf16_dev(g), eps=eps,
                                       row_index=None if row_index is None else dev(row_index), scale=scale)
    torch.cuda.synchronize()
    exp_routed = orc.finalize(rows, w, T, K, row_index=row_index, scale=scale)
    np.testing.assert_array_equal(bf16_bits(routed), exp_routed)
    lo, hi = orc.rmsnorm_bounds(orc.rmsnorm(exp_routed, g, eps))
    got = _f(bf16_bits(out))
    assert np.all(_f(lo) <= got) and np.all(got <= _f(hi))
    assert moe.device_error(clear=True) == 0
    return routed, out


def _weights(T, K, seed=0):
    u = synth.rng(seed, synth.WEIGHTS).random((T, K)).astype(np.float32)
    return synth.f32_to_bf16_bits(u / u.sum(1, keepdims=True))


@pytest.mark.parametrize("T", [1, 8, 64, 1020])
def test_decode_shapes(moe, orc, T):
    """The latent 3584, top-16 rows of the decode batches, BF16 weights, eps 1e-5."""
    _check(moe, orc, synth.expert_rows(T), _weights(T, 16), T, 16, synth.norm_weight())


@pytest.mark.parametrize("T,K,H,wdt,eps", [(37, 16, 3584, "f32", 1e-5), (5, 3, 256, "bf16", 0.0),
                                           (9, 32, 1024, "f32", 1e-6), (4, 8, 8192, "bf16", 1e-5),
                                           (3, 16, 7168, "bf16", 1e-5), (400, 12, 3584, "bf16", 1e-5)])
def test_shapes_and_chunks(moe, orc, T, K, H, wdt, eps):
    """Ragged T, other K and widths; H = 7168 and 8192 take the rows in chunks, and so
    does a batch of more tokens than two CTAs per SM hold at once (three CTAs per SM,
    chunks of ten rows)."""
    rows = synth.normal_bf16(21 + H, 4, (T * K, H))
    w = synth.normal_bf16(21, 7, (T, K), 0.25) if wdt == "bf16" else synth.normal_f32(21, 7, (T, K), 0.25)
    g = synth.norm_weight(l=H)
    _check(moe, orc, rows, w, T, K, g, eps=eps)


def test_gathered_rows_with_minus_one_and_scale(moe, orc):
    """The GLM finalize page's shape: T = 512, K = 8, hidden 7168, permuted indices with
    5 % -1, routed_scaling_factor 2.5."""
    d = synth.finalize_shared_inputs()
    _check(moe, orc, d["rows"], d["weights"], d["T"], d["K"], synth.norm_weight(l=7168), row_index=d["row_index"],
           scale=d["scale"])


def test_routed_matches_finalize_and_may_be_omitted(moe):
    T = 300
    rows = bf16_dev(synth.expert_rows(T))
    w = bf16_dev(_weights(T, 16))
    g = bf16_dev(synth.norm_weight())
    r1, o1 = moe.finalize_rmsnorm(rows, w, T, 16, g)
    _, o2 = moe.finalize_rmsnorm(rows, w, T, 16, g, want_routed=False)
    f = moe.finalize(rows, w, T, 16)
    assert torch.equal(r1.view(torch.int16), f.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_zero_rows_give_zero(moe):
    T, K, H = 4, 16, 3584
    rows = torch.zeros(T * K, H, dtype=torch.bfloat16, device="cuda")
    w = bf16_dev(_weights(T, K))
    _, out = moe.finalize_rmsnorm(rows, w, T, K, bf16_dev(synth.norm_weight()))
    assert torch.count_nonzero(out.float()) == 0

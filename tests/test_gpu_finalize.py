"""Finalize on the GPU against the oracle, bit for bit (wide page, class Finalize;
GLM-5-next finalize page, _QuadFinalizePublishDeviceKernel)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_bits, bf16_dev, dev
from helpers import f32_from_bits, golden_lines

pytestmark = pytest.mark.gpu


def _run(moe, rows, w, T, K, row_index=None, shared=None, scale=1.0):
    wd = bf16_dev(w) if w.dtype == np.uint16 else dev(w)
    out = moe.finalize(bf16_dev(rows), wd, T, K, row_index=None if row_index is None else dev(row_index),
                       shared=None if shared is None else bf16_dev(shared), scale=scale)
    torch.cuda.synchronize()
    return bf16_bits(out)


@pytest.mark.parametrize("T,K,H,wdt", [
    (8, 16, 3584, "bf16"),     # tiny decode batch
    (64, 16, 3584, "bf16"),    # narrow
    (37, 16, 3584, "f32"),     # ragged token count
    (5, 16, 8, "bf16"),        # one fragment per token
    (3, 12, 64, "f32"),        # runtime-K path with a tail chunk
    (4, 32, 256, "bf16"),      # K = 32
    (6, 1, 24, "f32"),
    (9, 8, 7168, "bf16"),      # the K = 8 path
])
def test_plain_parity(moe, orc, T, K, H, wdt):
    rows = synth.normal_bf16(11, 4, (T * K, H))
    w = synth.normal_bf16(11, 7, (T, K), 0.25) if wdt == "bf16" else synth.normal_f32(11, 7, (T, K), 0.25)
    np.testing.assert_array_equal(_run(moe, rows, w, T, K), orc.finalize(rows, w, T, K))


def test_wide_full_size(moe, orc):
    """T = 1020 (204 requests x 5 speculative tokens), K = 16, latent 3584: every output."""
    T = 1020
    rows = synth.expert_rows(T)
    u = synth.rng(0, synth.WEIGHTS).random((T, 16)).astype(np.float32)
    w = synth.f32_to_bf16_bits(u / u.sum(1, keepdims=True))
    np.testing.assert_array_equal(_run(moe, rows, w, T, 16), orc.finalize(rows, w, T, 16))


def test_shared_variant_full_size(moe, orc):
    """T = 512, K = 8, hidden 7168, permuted indices with 5 % -1, BF16 weights,
    routed_scaling_factor 2.5, shared expert rows added: every output."""
    d = synth.finalize_shared_inputs()
    got = _run(moe, d["rows"], d["weights"], d["T"], d["K"], d["row_index"], d["shared"], d["scale"])
    exp = orc.finalize(d["rows"], d["weights"], d["T"], d["K"], row_index=d["row_index"], shared=d["shared"], scale=d["scale"])
    np.testing.assert_array_equal(got, exp)


@pytest.mark.parametrize("gather,shared,scale,wdt", [
    (True, False, 1.0, "f32"), (True, True, 1.0, "bf16"), (False, True, 2.5, "f32"), (True, True, 0.75, "f32"),
    (False, False, 3.0, "bf16"),
])
def test_variant_matrix(moe, orc, gather, shared, scale, wdt):
    T, K, H, n = 19, 16, 512, 400
    rows = synth.normal_bf16(12, 4, (n, H))
    rng = np.random.default_rng(12)
    idx = rng.integers(-1, n, (T, K)).astype(np.int32) if gather else None
    if not gather:
        rows = rows[: T * K]
    w = synth.normal_bf16(12, 7, (T, K), 0.3) if wdt == "bf16" else synth.normal_f32(12, 7, (T, K), 0.3)
    sh = synth.normal_bf16(12, 8, (T, H)) if shared else None
    got = _run(moe, rows, w, T, K, idx, sh, scale)
    np.testing.assert_array_equal(got, orc.finalize(rows, w, T, K, row_index=idx, shared=sh, scale=scale))


@pytest.mark.parametrize("row", list(golden_lines("finalize_closed_forms.txt")), ids=lambda r: r[0])
def test_golden_on_gpu(moe, row):
    name, wbits, rbits, exp = row
    w = np.array([f32_from_bits(int(v, 16)) for v in wbits.split(",")], np.float32)[None, :]
    K = w.shape[1]
    rows = np.repeat(np.array([int(v, 16) for v in rbits.split(",")], np.uint16).reshape(K, 1), 16, axis=1)
    assert np.all(_run(moe, rows, w, 1, K) == int(exp, 16))


def test_all_minus_one_is_shared(moe):
    T, K, H = 4, 8, 64
    sh = synth.normal_bf16(13, 8, (T, H))
    got = _run(moe, synth.normal_bf16(13, 4, (8, H)), np.ones((T, K), np.float32), T, K,
               np.full((T, K), -1, np.int32), sh, 2.5)
    np.testing.assert_array_equal(got, sh)


def test_zero_tokens_is_a_noop(moe):
    out = moe.finalize(bf16_dev(np.zeros((16, 64), np.uint16)), dev(np.zeros((0, 16), np.float32)), 0, 16)
    assert out.shape == (0, 64)


def test_bad_index_sets_error_and_skips(moe, orc):
    moe.device_error(clear=True)
    T, K, H, n = 3, 4, 32, 10
    rows = synth.normal_bf16(14, 4, (n, H))
    idx = np.array([[0, 1, 2, 3], [4, 99, 5, -1], [-7, 6, 7, 8]], np.int32)
    w = synth.normal_f32(14, 7, (T, K))
    got = _run(moe, rows, w, T, K, idx)
    assert moe.device_error(clear=True) & moe.DEVERR_ROW_INDEX
    fixed = np.where((idx < -1) | (idx >= n), -1, idx).astype(np.int32)
    np.testing.assert_array_equal(got, orc.finalize(rows, w, T, K, row_index=fixed))
    assert moe.device_error(clear=True) == 0


def test_deterministic(moe):
    T, K, H = 64, 16, 3584
    rows = bf16_dev(synth.normal_bf16(15, 4, (T * K, H)))
    w = bf16_dev(synth.normal_bf16(15, 7, (T, K), 0.25))
    a = moe.finalize(rows, w, T, K)
    b = moe.finalize(rows, w, T, K)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))

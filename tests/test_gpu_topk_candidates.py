"""The top-K candidate search (approximate keys, exact refinement): the bound it
relies on, and parity with the oracle on near-tied keys that the approximate keys
cannot order (each candidate path: up to 32 and up to 64 candidates ranked over
shuffles, the all-exact fallback)."""
import os
import subprocess

import numpy as np
import pytest
import torch

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_approx_sigmoid_bound(tmp_path):
    """Every FP32 input: |approx - spec| < kApproxErr, NaN in the same places."""
    exe = tmp_path / "bound"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O3",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "latent_moe_decode_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cuda", "approx_sigmoid_bound.cu"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=300).stdout.split()
    err, bound, nan_mismatch = float(out[0]), float(out[1]), int(out[2])
    assert nan_mismatch == 0
    assert 0 < err < bound, (err, bound)


@pytest.mark.parametrize("step_exp", [-11, -13, -15, -20])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("T", [64, 256])
def test_near_ties(moe, orc, step_exp, with_bias, T):
    """Logits on a ladder 0.5 + i * 2^step_exp (shuffled over the experts): neighbouring
    scores differ by about 0.24 * 2^step_exp, near or below the approximation's error, so
    many experts fall inside the candidate margin (about 2^-10): 2^-11 gives ~25
    candidates (ranked over shuffles), 2^-13 ~50 (two per lane), 2^-15 and 2^-20 more
    than 64 (exact keys for all, argmax rounds). T = 64 takes the CTA-per-token body,
    T = 256 the warp-per-token body."""
    E, K = 896, 16
    rng = np.random.default_rng(100 - step_exp)
    lad = (0.5 + np.arange(E, dtype=np.float64) * 2.0 ** step_exp).astype(np.float32)
    logits = np.stack([lad[rng.permutation(E)] for _ in range(T)])
    bias = (np.full(E, 0.01, np.float32) if with_bias else None)
    ids, w, wb = moe.topk_route(dev(logits), None if bias is None else dev(bias), K)
    torch.cuda.synchronize()
    eids, ew, ewb = orc.topk_route(logits, bias, K)
    np.testing.assert_array_equal(host(ids), eids)
    np.testing.assert_array_equal(host(w).view(np.uint32), ew.view(np.uint32))

"""The allocation-free router entry point, moe_router_logits_noalloc, called through
the C ABI, against the regular moe_router_logits on the same inputs.

It exists for callers that cannot allocate device memory when they compute the
router logits (an engine whose memory pool owns the device after start-up, a plug-in
given only its inputs and outputs): it keeps the split-K partials in an array the
library reserves itself. Calls in a row with different shapes check that what the
previous call left in that shared array never leaks into a result. Kept in a file of
its own, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_dev

pytestmark = pytest.mark.gpu


def _noalloc(moe, x, w):
    T, H = x.shape
    E = w.shape[0]
    out = torch.empty(T, E, dtype=torch.float32, device=x.device)
    st = moe.load().moe_router_logits_noalloc(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(out.data_ptr()), T, H, E,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, moe.load().moe_status_string(st)
    return out


def test_noalloc_matches_router_logits(moe):
    """Calls in a row over every plan shape the router takes at the decode widths --
    T = 1, 8, 16, 64 (narrow tiles, up to 16 splits in a cluster), 256 (128-column
    tiles), 1020 (256-column tiles in 5-CTA clusters) -- each bit-identical to the
    regular entry point, so nothing an earlier call left in the shared array leaks in."""
    torch.backends.cuda.matmul.allow_tf32 = False  # the tolerance bound below in full FP32
    w = bf16_dev(synth.router_weight())
    for T, seed in ((1, 11), (8, 12), (64, 13), (1020, 14), (16, 15), (256, 16), (1020, 17)):
        x = bf16_dev(synth.hidden_rows(T, seed=seed))
        got = _noalloc(moe, x, w)
        ref = moe.router_logits(x, w)  # the regular entry point, caller-owned workspace
        torch.cuda.synchronize()
        bound = 1e-5 * (x.float().abs() @ w.float().abs().t())
        assert torch.all((got - ref).abs() <= bound), f"T={T}"
        assert torch.equal(got, ref), f"T={T}: not bit-identical"
    assert moe.device_error(clear=True) == 0


@pytest.mark.parametrize("T", [1, 4, 5, 16, 64, 256, 1020, 4096])
def test_noalloc_fits_every_decode_width(moe, T):
    """With the 896 x 7168 gate the array holds the partials of every token count the
    decode step uses (the call returns OK, not MOE_ERR_CAPACITY)."""
    w = bf16_dev(synth.router_weight())
    x = bf16_dev(synth.hidden_rows(T, seed=20 + T))
    got = _noalloc(moe, x, w)
    torch.cuda.synchronize()
    assert torch.equal(got, moe.router_logits(x, w)), f"T={T}"


def test_noalloc_rejects_bad_arguments(moe):
    lib = moe.load()
    x = bf16_dev(np.zeros((8, 64), np.uint16))
    w = bf16_dev(np.zeros((16, 64), np.uint16))
    out = torch.empty(8, 16, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moe_router_logits_noalloc(p(x), p(w), p(out), 0, 64, 16, s) == moe.ERR_INVALID_ARGUMENT
    assert lib.moe_router_logits_noalloc(p(x), p(w), p(out), 8, 63, 16, s) == moe.ERR_INVALID_ARGUMENT
    assert lib.moe_router_logits_noalloc(ctypes.c_void_p(x.data_ptr() + 2), p(w), p(out), 8, 64, 16, s) == moe.ERR_ALIGNMENT
    # T * E above 2^40 is refused before any plan or launch, as by moe_router_logits
    assert lib.moe_router_logits_noalloc(p(x), p(w), p(out), 1 << 30, 64, 1 << 11, s) == moe.ERR_CAPACITY

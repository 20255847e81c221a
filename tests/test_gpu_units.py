"""Unit windows on the GPU against the oracle, bit for bit (wide page, module
docstring: the grouped engine's units built from the routing lists, every touched
expert once per 8 of its tokens), on lists the GPU built from top-16-shaped ids."""
import numpy as np
import pytest
import torch

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def _ids(seed, T, K, E):
    rng = np.random.default_rng(seed)
    logp = -1.1 * np.log(np.arange(1, E + 1))  # Zipf(1.1) loads: heavy experts and empty ones
    return np.argsort(-(logp[None, :] + rng.gumbel(size=(T, E))), axis=1)[:, :K].astype(np.int32)


@pytest.mark.parametrize("T,K,E,W", [(8, 16, 896, 8), (64, 16, 896, 8), (1020, 16, 896, 8), (4096, 16, 896, 8),
                                     (1020, 16, 896, 1), (1020, 16, 896, 32), (500, 8, 1024, 8), (300, 1, 1, 8),
                                     (50, 4, 17, 3), (0, 16, 896, 8)])
def test_parity(moe, orc, T, K, E, W):
    ids = _ids(T + E + W, T, K, E) if T else np.zeros((0, K), np.int32)
    off, _ = moe.build_routing_lists(dev(ids), E)
    cap = moe.unit_windows_capacity(T, K, E, W)
    uo, ue, us, ul = moe.unit_windows(off, W, max_units=max(cap, 1))
    torch.cuda.synchronize()
    eo, ee, es, el = orc.unit_windows(host(off), W)
    n = int(eo[-1])
    assert n <= cap
    np.testing.assert_array_equal(host(uo), eo)
    np.testing.assert_array_equal(host(ue)[:n], ee)
    np.testing.assert_array_equal(host(us)[:n], es)
    np.testing.assert_array_equal(host(ul)[:n], el)
    assert moe.device_error(clear=True) == 0


def test_too_small_capacity_sets_error(moe, orc):
    moe.device_error(clear=True)
    off = dev(np.array([0, 0, 17, 18, 26, 26], np.int32))
    sentinel = -7
    ue, us, ul = (torch.full((5,), sentinel, dtype=torch.int32, device="cuda") for _ in range(3))
    uo, ue, us, ul = moe.unit_windows(off, 8, max_units=3, unit_expert=ue, unit_start=us, unit_len=ul)
    assert moe.device_error(clear=True) & moe.DEVERR_CAPACITY
    eo, ee, es, el = orc.unit_windows(np.array([0, 0, 17, 18, 26, 26], np.int32), 8)
    np.testing.assert_array_equal(host(uo), eo)  # the offsets are complete
    assert host(ue)[:3].tolist() == ee[:3].tolist() and host(ue)[3:].tolist() == [sentinel] * 2

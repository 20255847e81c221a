"""Routing lists on the GPU against the oracle, bit for bit (wide page, WideRoute:
pair code t*K + k appended to its expert's list; here CSR in token order)."""
import numpy as np
import pytest
import torch

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def _ids(seed, T, K, E, skew=False):
    rng = np.random.default_rng(seed)
    if T == 0:
        return np.zeros((0, K), np.int32)
    if skew:  # Zipf(1.1) popularity through Gumbel top-k (distinct per row)
        logp = -1.1 * np.log(np.arange(1, E + 1))
        g = logp[None, :] + rng.gumbel(size=(T, E))
        return np.argsort(-g, axis=1)[:, :K].astype(np.int32)
    return np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)


@pytest.mark.parametrize("T,K,E,skew", [
    (1, 16, 896, False), (8, 16, 896, False), (64, 16, 896, False), (1020, 16, 896, False),
    (1024, 16, 896, True), (1025, 16, 896, False), (4096, 16, 896, True), (5000, 8, 300, False),
    (100, 32, 1024, False), (300, 1, 1, False), (50, 4, 17, True), (0, 16, 896, False),
])
def test_parity(moe, orc, T, K, E, skew):
    ids = _ids(T + K + E, T, K, E, skew)
    off, pairs = moe.build_routing_lists(dev(ids), E)
    torch.cuda.synchronize()
    eoff, epairs = orc.routing_lists(ids, E)
    np.testing.assert_array_equal(host(off), eoff)
    np.testing.assert_array_equal(host(pairs), epairs)


@pytest.mark.parametrize("T,K,E,hi", [(100, 16, 896, 1), (300, 16, 896, 4), (2000, 16, 64, 40), (700, 8, 33, 33)])
def test_parity_repeated_ids(moe, orc, T, K, E, hi):
    """Ids drawn with repeats from [0, hi): whole warps of equal ids, which the
    placement ranks as one group (the pages do not forbid repeats within a token)."""
    ids = np.random.default_rng(T + hi).integers(0, hi, size=(T, K)).astype(np.int32)
    off, pairs = moe.build_routing_lists(dev(ids), E)
    torch.cuda.synchronize()
    eoff, epairs = orc.routing_lists(ids, E)
    np.testing.assert_array_equal(host(off), eoff)
    np.testing.assert_array_equal(host(pairs), epairs)


def test_bad_id_sets_error(moe):
    moe.device_error(clear=True)
    ids = np.array([[0, 1], [2, 9], [-1, 3]], np.int32)
    off, pairs = moe.build_routing_lists(dev(ids), 5)
    assert moe.device_error(clear=True) & moe.DEVERR_EXPERT_ID
    o = host(off)
    assert o[-1] == 4  # the two bad pairs were dropped
    assert host(pairs)[:4].tolist() == [0, 1, 2, 5]

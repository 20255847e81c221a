"""GPU-test helpers: move numpy test data (BF16 as uint16 bits) to CUDA tensors and
back. Test-only; shares nothing with the oracle or the library."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


@pytest.fixture(scope="session")
def moe():
    require_gpu()
    import latent_moe_decode_gb300 as m

    m.build.build()
    m.load()
    m.device_error(clear=True)
    return m

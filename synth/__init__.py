"""Seeded synthetic inputs shaped like the pages' decode batches.

Shared by the tests, the smoke check and the benchmark. Holds none of the method's
arithmetic: it only draws random tensors and stores them in the formats the path
consumes (BF16 as raw ``uint16`` bits, FP32, int32).

Every tensor is drawn from its own counter-based stream: a Philox-4x64 generator
keyed by (seed, tensor id), so a tensor does not depend on which others were drawn
or in what order. Normal draws are rounded FP64 -> FP32 -> BF16 (nearest even).

Shapes (the Kimi-K3 latent-MoE layer of the wide decode page): hidden H = 7168,
latent L = 3584, E = 896 routed experts, top-k K = 16.
"""
from __future__ import annotations

import numpy as np

H, L, E, K = 7168, 3584, 896, 16

# tensor ids of the counter-based streams
X, W, BIAS, ROWS, LATENT, PERM, WEIGHTS, SHARED, SKEW, W_DOWN, NORM = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11

# Zipf-skew temperature: bias_e = -1.1 * SKEW_TAU * ln(rank_e). Calibrated once by
# tests/golden/calibrate_skew.py (oracle top-16 over seed-0 inputs at T=4096) so
# that the log-log slope of the sorted expert loads is -1.1 +- 0.05.
SKEW_TAU = 0.0201


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed), int(tensor_id)]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 array -> BF16 bits (round to nearest even; inputs here are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, tensor_id: int, shape, std: float = 1.0) -> np.ndarray:
    g = rng(seed, tensor_id)
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    chunk = 1 << 24
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        v = g.standard_normal(m) * std
        out[i : i + m] = f32_to_bf16_bits(v.astype(np.float32))
    return out.reshape(shape)


def normal_f32(seed: int, tensor_id: int, shape, std: float = 1.0) -> np.ndarray:
    g = rng(seed, tensor_id)
    return (g.standard_normal(int(np.prod(shape))) * std).astype(np.float32).reshape(shape)


# ---------------------------------------------------------------------------
# The routing chain: router -> top-16 -> lists, MXFP8 of the latent, Finalize.

def hidden_rows(T: int, seed: int = 0, h: int = H) -> np.ndarray:
    """x: BF16 [T, h] ~ N(0, 1)."""
    return normal_bf16(seed, X, (T, h), 1.0)


def router_weight(seed: int = 0, e: int = E, h: int = H) -> np.ndarray:
    """gate: BF16 [e, h] ~ N(0, 0.02)."""
    return normal_bf16(seed, W, (e, h), 0.02)


def latent_down_weight(seed: int = 0, l: int = L, h: int = H) -> np.ndarray:
    """latent down projection: BF16 [l, h] ~ N(0, 0.02) (the router weight's scale;
    the pages give no initialisation)."""
    return normal_bf16(seed, W_DOWN, (l, h), 0.02)


def norm_weight(seed: int = 0, l: int = L) -> np.ndarray:
    """RMSNorm weight: BF16 [l] ~ 1 + N(0, 0.1) (near one, as a trained norm)."""
    return f32_to_bf16_bits((1.0 + rng(seed, NORM).standard_normal(l) * 0.1).astype(np.float32))


def correction_bias(seed: int = 0, e: int = E) -> np.ndarray:
    """e_score_correction_bias: FP32 [e] ~ N(0, 0.01)."""
    return normal_f32(seed, BIAS, (e,), 0.01)


def skew_bias(seed: int = 0, e: int = E, tau: float = SKEW_TAU) -> np.ndarray:
    """Zipf-popularity bias: -1.1 * tau * ln(rank), ranks a seeded permutation of 1..e."""
    ranks = rng(seed, SKEW).permutation(e) + 1
    return (-1.1 * tau * np.log(ranks.astype(np.float64))).astype(np.float32)


def expert_rows(T: int, seed: int = 0, k: int = K, l: int = L) -> np.ndarray:
    """The experts' expanded output rows: BF16 [T*k, l] ~ N(0, 1); row t*k + j is
    (token t, slot j)."""
    return normal_bf16(seed, ROWS, (T * k, l), 1.0)


def latent_rows(T: int, seed: int = 0, l: int = L) -> np.ndarray:
    """Latent rows to quantise: BF16 [T, l] ~ N(0, 1)."""
    return normal_bf16(seed, LATENT, (T, l), 1.0)


def chain_inputs(T: int, seed: int = 0, skew: bool = False) -> dict:
    return {
        "x": hidden_rows(T, seed),
        "w": router_weight(seed),
        "bias": skew_bias(seed) if skew else correction_bias(seed),
        "rows": expert_rows(T, seed),
        "latent": latent_rows(T, seed),
    }


# ---------------------------------------------------------------------------
# Finalize with the shared expert (the GLM-5-next finalize page's kernel shape).

def finalize_shared_inputs(T: int = 512, k: int = 8, h: int = H, n_rows: int = 4096,
                           minus_one_frac: float = 0.05, seed: int = 0) -> dict:
    """routed rows BF16 [n_rows, h] ~ N(0,1); permuted_indices int32 [T*k] a seeded
    permutation of 0..n_rows-1 (T*k == n_rows) with round(frac * T*k) seeded
    positions set to -1; weights U(0,1) per (t, slot) divided by the token's
    sequential FP32 sum, rounded to BF16; shared BF16 [T, h] ~ N(0,1)."""
    assert T * k == n_rows
    g = rng(seed, PERM)
    perm = g.permutation(n_rows).astype(np.int32)
    n_neg = int(round(minus_one_frac * n_rows))
    perm[g.choice(n_rows, size=n_neg, replace=False)] = -1
    u = rng(seed, WEIGHTS).random((T, k)).astype(np.float32)
    s = np.zeros(T, np.float32)
    for j in range(k):
        s = (s + u[:, j]).astype(np.float32)
    wts = f32_to_bf16_bits((u / s[:, None]).astype(np.float32))
    return {
        "rows": normal_bf16(seed, ROWS, (n_rows, h), 1.0),
        "row_index": perm.reshape(T, k),
        "weights": wts,
        "shared": normal_bf16(seed, SHARED, (T, h), 1.0),
        "scale": 2.5,
        "T": T,
        "K": k,
        "H": h,
    }


# The benchmark configurations (sizes of the pages' decode batches).
CONFIGS = {
    "tiny": dict(T=8),            # one small decode batch
    "narrow": dict(T=64),         # the prepared-batch ceiling of the narrow path
    "wide": dict(T=1020),         # 204 verify requests x 5 speculative tokens
    "skew": dict(T=(1, 16, 64, 256, 1020, 4096)),
}

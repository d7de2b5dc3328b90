"""Seeded synthetic inputs shared by the oracle side and the CUDA side of a test.

Holds none of the method's arithmetic: only random activation vectors and
token lists drawn with numpy's seeded generator.  Model weights and the KV
prefill are not drawn here; each side generates those itself from (seed, uid)
with its own implementation of the counter-based generator.
"""
import numpy as np


def activation(n: int, seed: int, std: float = 1.0) -> np.ndarray:
    """fp32 vector ~ N(0, std^2), the GEMV input x."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n) * std).astype(np.float32)


def dyadic_activation(n: int, seed: int, lo: int = -8, hi: int = 8, shift: int = 3) -> np.ndarray:
    """Small dyadic rationals k / 2^shift: sums of products with dyadic weights are exact in fp64."""
    rng = np.random.default_rng(seed)
    return (rng.integers(lo, hi + 1, n).astype(np.float64) / (1 << shift)).astype(np.float32)


def f16_cache(n_kv: int, max_ctx: int, head_dim: int, seed: int) -> np.ndarray:
    """f16 bits (uint16) of N(0,1) draws, shaped [n_kv][max_ctx][head_dim]: a K or V cache."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n_kv, max_ctx, head_dim)).astype(np.float16).view(np.uint16)

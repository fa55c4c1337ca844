"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no rotation, no quantisation, no packing).  Both the CUDA
path and the CPU oracle receive the exact arrays it returns.

Distributions follow the 27B-class workloads the pages talk about
(hidden 5120, FFN 27648 -- zwxr.cn/news/303439, sec. on the model topology):
  weights      ~ N(0, 0.02) with a fixed fraction of entries (chosen without
               replacement) multiplied by 20 ("outliers")
  activations  ~ N(0, 1) with a few whole channels (columns) multiplied by 30
Generator: numpy PCG64 via ``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to fp32 values."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(N: int, K: int, seed: int, *, dtype: str = "bf16", std: float = 0.02,
            outlier_frac: float = 0.001, outlier_mult: float = 20.0) -> np.ndarray:
    """W [N][K]: float32 array (dtype="f32") or uint16 bf16 bits (dtype="bf16")."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)
    n_out = int(round(outlier_frac * N * K))
    if n_out:
        idx = rng.choice(N * K, size=n_out, replace=False)
        w.reshape(-1)[idx] *= np.float32(outlier_mult)
    if dtype == "f32":
        return w
    if dtype == "bf16":
        return f32_to_bf16_bits(w)
    raise ValueError(dtype)


def activations(M: int, K: int, seed: int, *, n_outlier_channels: int = 4,
                outlier_mult: float = 30.0) -> np.ndarray:
    """x [M][K] as uint16 bf16 bits (N(0,1), a few channels scaled up)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if n_outlier_channels:
        ch = rng.choice(K, size=min(n_outlier_channels, K), replace=False)
        x[:, ch] *= np.float32(outlier_mult)
    return f32_to_bf16_bits(x)


def tiny_config():
    """The small end-to-end case: one 256x256 linear, fp32 weights with 0.5%
    outliers x20 (exactly 328 entries), bf16 activations, batch 1, seed 0."""
    W = weights(256, 256, 0, dtype="f32", outlier_frac=0.005)
    x = activations(1, 256, 1, n_outlier_channels=0)
    return W, x

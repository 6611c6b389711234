"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers and casts them; it holds none of the attention's
arithmetic.  Values are drawn in float64 from numpy's PCG64 stream seeded with
SeedSequence([seed, config, layer, tensor_id]), cast to float32 and, for bf16 inputs,
rounded to bfloat16 (round-to-nearest-even, done by torch's cast).

The pages train and evaluate on FineWeb-Edu and Wikipedia text, which are not available
here; i.i.d. N(0, 1) activations shaped like the pages' 60M model (16 layers, 8 heads of
64 = hidden 512, training length 1024, evaluation length 4096) stand in for them.
"""
from __future__ import annotations

import numpy as np
import torch

SEED = 20261202
TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_DO, TENSOR_ALPHA = 0, 1, 2, 3, 4

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def rng(config: int, layer: int, tensor_id: int, seed: int = SEED) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, config, layer, tensor_id]))


def normal(shape, config: int, layer: int, tensor_id: int, dtype: str = "f32",
           seed: int = SEED) -> torch.Tensor:
    """N(0,1) tensor (CPU, `dtype`), drawn in float64, cast to float32, then to dtype."""
    x = rng(config, layer, tensor_id, seed).standard_normal(size=tuple(shape))
    t = torch.from_numpy(x.astype(np.float32))
    return t.to(TORCH_DTYPES[dtype])


def qkv(B: int, H: int, N: int, D: int, config: int, layer: int, dtype: str = "f32",
        seed: int = SEED):
    """(q, k, v) CPU tensors of layout [B, H, N, D]."""
    shape = (B, H, N, D)
    return tuple(normal(shape, config, layer, t, dtype, seed)
                 for t in (TENSOR_Q, TENSOR_K, TENSOR_V))


def upstream_grad(B: int, H: int, N: int, D: int, config: int, layer: int,
                  dtype: str = "f32", seed: int = SEED) -> torch.Tensor:
    return normal((B, H, N, D), config, layer, TENSOR_DO, dtype, seed)


def learned_alpha(n_layers: int, config: int, lo: float = 0.9, hi: float = 1.1,
                  seed: int = SEED) -> np.ndarray:
    """Per-layer alpha drawn U[lo, hi] and rounded to float32 (a learned parameter is
    stored as float32).  Returned as float64 values that are exactly float32."""
    a = rng(config, 0, TENSOR_ALPHA, seed).uniform(lo, hi, size=n_layers)
    return a.astype(np.float32).astype(np.float64)


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a CPU tensor (bf16 and f32 both embed exactly in float64)."""
    return t.detach().to(torch.float64).cpu().numpy()

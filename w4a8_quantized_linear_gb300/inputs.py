"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle
checks.  This module holds no arithmetic of the quantized linear itself: it
only draws activations and full-precision weights with the shapes and value
distributions of the workloads (the pages measure on real Qwen3 / Llama3
layers and wikitext2, which are not available; these stand in for them).

Recipe
------
* Random numbers: numpy ``Generator(PCG64(seed))``; one seed per tensor:
  layer i of a workload draws its activations x with ``base_seed + 2 i`` and
  its weights W with ``base_seed + 2 i + 1`` (tensor index 0, 1, 2, 3, ... in
  the order x, W, x2, W2, ...).
* Activations x [M, K]: fp32 N(0, 1); ``floor(K / 100)`` outlier channels
  (1 % of K, sampled without replacement from the same generator) are scaled
  by 20; the result is rounded to fp16 (or, for the bf16 entry points, to
  bf16).
* Weights W [N, K]: fp32 N(0, 0.02).
"""
from __future__ import annotations

import numpy as np

OUTLIER_SCALE = 20.0
WEIGHT_SIGMA = 0.02


def activations(M: int, K: int, seed: int = 0) -> np.ndarray:
    """fp16 [M, K] ~ N(0,1) with floor(K/100) outlier channels scaled x20."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = K // 100
    if n_out:
        cols = rng.choice(K, size=n_out, replace=False)
        x[:, cols] *= np.float32(OUTLIER_SCALE)
    return x.astype(np.float16)


def activations_bf16(M: int, K: int, seed: int = 0) -> np.ndarray:
    """The draws of :func:`activations`, rounded to bf16 (nearest, ties to
    even) instead of fp16, as uint16 bit patterns [M, K] (numpy has no bf16
    type; the upper half of each fp32, rounded)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = K // 100
    if n_out:
        cols = rng.choice(K, size=n_out, replace=False)
        x[:, cols] *= np.float32(OUTLIER_SCALE)
    b = x.view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def weights(N: int, K: int, seed: int = 1) -> np.ndarray:
    """fp32 [N, K] ~ N(0, 0.02)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(WEIGHT_SIGMA)
    return w


def layer(M: int, N: int, K: int, base_seed: int = 0, index: int = 0):
    """(x fp16 [M,K], W fp32 [N,K]) for the index-th layer of a workload."""
    return (activations(M, K, base_seed + 2 * index),
            weights(N, K, base_seed + 2 * index + 1))


# Workload shapes (N x K) of the benchmark and the parity tests.
SWEEP_SHAPES = [(10240, 2560), (2560, 10240)]
SWEEP_M = [1, 16, 128, 1024, 4096, 8192]
# Qwen3-2B-shaped decoder layer (hidden 2048, 8 KV heads x 128, MLP 6144).
QWEN3_2B = {"q": (2048, 2048), "k": (1024, 2048), "v": (1024, 2048),
            "o": (2048, 2048), "gate": (6144, 2048), "up": (6144, 2048),
            "down": (2048, 6144)}
QWEN3_2B_M = [1334, 2393, 3455]
# Qwen3-8B-shaped decoder layer (hidden 4096, 8 KV heads x 128, MLP 12288).
QWEN3_8B = {"q": (4096, 4096), "k": (1024, 4096), "v": (1024, 4096),
            "o": (4096, 4096), "gate": (12288, 4096), "up": (12288, 4096),
            "down": (4096, 12288)}
QWEN3_8B_M = [4096, 1]

"""Seeded synthetic inputs shared by the CPU oracle, the tests and the bench.

This module only draws random numbers and lays them out; it holds none of
the quantisation or GEMM arithmetic.  Every tensor is produced in float32
from a numpy ``Generator(PCG64(seed))`` in a fixed draw order and then
rounded to BF16 (round-to-nearest-even), returned as raw ``uint16`` bit
patterns so that the CPU oracle and the GPU path start from the very same
bytes.

Distributions follow the workloads of the linear layer described on the
pages: activations and gradients are N(0, 1) with a Bernoulli fraction of
outliers scaled by a constant (activations "often contain significant
outliers", Unified FP8 review, "FP8 Quantization"), weights are N(0, std)
("near Gaussian", same section).  MoE routing for the grouped GEMM uses
top-k over N(0, 1) logits plus a Zipf-shaped expert bias.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "activations",
    "weights",
    "moe_routing",
]


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return uint16 bits.

    Inputs must be finite (the generators never produce inf/NaN).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations(shape, seed: int, outlier_frac: float = 0.01, outlier_mult: float = 50.0) -> np.ndarray:
    """N(0,1) values; a Bernoulli(outlier_frac) subset multiplied by outlier_mult.

    Draw order: all normals, then all uniforms for the outlier mask.
    Returns BF16 bits (uint16) of the given shape.
    """
    g = rng(seed)
    n = int(np.prod(shape))
    z = g.standard_normal(n, dtype=np.float32)
    if outlier_frac > 0.0:
        u = g.random(n, dtype=np.float32)
        z = np.where(u < np.float32(outlier_frac), z * np.float32(outlier_mult), z)
    return f32_to_bf16_bits(z).reshape(shape)


def weights(shape, seed: int, std: float = 0.02) -> np.ndarray:
    """N(0, std) values as BF16 bits."""
    g = rng(seed)
    n = int(np.prod(shape))
    z = g.standard_normal(n, dtype=np.float32) * np.float32(std)
    return f32_to_bf16_bits(z).reshape(shape)


def moe_routing(tokens: int, experts: int, top_k: int, seed: int, zipf_s: float = 1.1):
    """Top-k expert routing with a Zipf-shaped popularity bias.

    logits[t, e] = N(0,1) + b_e with b_e = -zipf_s * ln(rank_e), where the
    ranks are a seeded permutation of 1..experts.  Softmax is monotone, so
    the top-k of the softmax equals the top-k of the logits; ties go to the
    lower expert index.  Returns (token_index, offsets): token_index lists,
    expert by expert and in ascending token order, the token feeding each
    routed row; offsets[e] .. offsets[e+1] is expert e's row range.
    """
    g = rng(seed)
    logits = g.standard_normal((tokens, experts), dtype=np.float32)
    ranks = g.permutation(experts) + 1
    bias = (-zipf_s * np.log(ranks.astype(np.float64))).astype(np.float32)
    logits = logits + bias[None, :]
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    expert_of = order.reshape(-1)
    token_of = np.repeat(np.arange(tokens, dtype=np.int64), top_k)
    perm = np.lexsort((token_of, expert_of))
    token_index = token_of[perm]
    counts = np.bincount(expert_of, minlength=experts).astype(np.int64)
    offsets = np.zeros(experts + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    return token_index, offsets

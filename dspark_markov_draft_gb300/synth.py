"""Seeded synthetic inputs for the Markov draft walk.

This module only draws random inputs; it holds none of the walk's arithmetic.
Both the CUDA path (tests, bench) and the CPU oracle read the tensors it makes,
so the two sides always see identical bytes.

Value distributions follow the workloads the walk is benchmarked on:

* ``W1``   [V, R] bf16, N(0, 1)
* ``W2``   [V, R] bf16, N(0, 1/R) (so one bias value has std about 1 at R = 256)
* ``base`` [bs, K, V] bf16, N(0, 3^2); optionally one +8 peak per (row, position)
  at a uniformly drawn vocabulary index, added in fp32 before the bf16 rounding
* ``prev`` [bs] int32, uniform in [0, V)
* ``seeds`` [bs] uint64, ``seed_base + b`` (per-request seeds 0..bs-1 by default)

Random draws use numpy's PCG64 generator; bf16 values are produced by torch's
round-to-nearest-even conversion from fp32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

RANK = 256


@dataclass
class WalkInputs:
    V: int
    R: int
    bs: int
    K: int
    w1: torch.Tensor  # [V, R] bf16 (CPU)
    w2: torch.Tensor  # [V, R] bf16 (CPU)
    base: torch.Tensor  # [bs, K, V] bf16 (CPU)
    prev: torch.Tensor  # [bs] int32 (CPU)
    seeds: torch.Tensor  # [bs] uint64 stored as int64 bit patterns (CPU)

    @staticmethod
    def bits(t: torch.Tensor) -> np.ndarray:
        """The raw uint16 bit pattern of a bf16 tensor as a numpy array."""
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x).to(torch.bfloat16)


def weights(V: int, R: int = RANK, seed: int = 0):
    """(W1, W2) as bf16 CPU tensors: W1 ~ N(0,1), W2 ~ N(0, 1/R)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w1 = _normal_bf16(rng, (V, R), 1.0)
    w2 = _normal_bf16(rng, (V, R), 1.0 / np.sqrt(R))
    return w1, w2


def base_logits(bs: int, K: int, V: int, seed: int = 1, peak: float | None = None,
                std: float = 3.0) -> torch.Tensor:
    """bf16 [bs, K, V] base logits ~ N(0, std^2), optionally with one +peak per row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(size=(bs, K, V), dtype=np.float32)
    x *= np.float32(std)
    if peak is not None:
        idx = rng.integers(0, V, size=(bs, K))
        b_ix, k_ix = np.meshgrid(np.arange(bs), np.arange(K), indexing="ij")
        x[b_ix, k_ix, idx] += np.float32(peak)
    return torch.from_numpy(x).to(torch.bfloat16)


def prev_tokens(bs: int, V: int, seed: int = 2) -> torch.Tensor:
    rng = np.random.Generator(np.random.PCG64(seed))
    return torch.from_numpy(rng.integers(0, V, size=bs).astype(np.int32))


def seeds(bs: int, seed_base: int = 0) -> torch.Tensor:
    return torch.arange(seed_base, seed_base + bs, dtype=torch.int64)


def make(V: int, bs: int, K: int, R: int = RANK, seed: int = 0, peak: float | None = None,
         seed_base: int = 0) -> WalkInputs:
    """One full input set for a walk of `bs` rows and `K` draft positions."""
    w1, w2 = weights(V, R, seed)
    base = base_logits(bs, K, V, seed + 1, peak)
    prev = prev_tokens(bs, V, seed + 2)
    return WalkInputs(V, R, bs, K, w1, w2, base, prev, seeds(bs, seed_base))


# The benchmark workloads: (name, V, K, batch sizes, W2 format, mode, temperature, top-k, extras)
WORKLOADS = {
    "v129280_k5_bf16_greedy": dict(V=129280, K=5, bs=(1,), w2="bf16", mode="greedy", T=1.0,
                                   top_k=0, peak=None, draft_logits=False),
    "v151936_k7_int8": dict(V=151936, K=7, bs=(1, 16, 64), w2="int8", mode=("greedy", "prob"),
                            T=1.0, top_k=0, peak=8.0, draft_logits=False),
    "v151936_k16_bf16_prob_logits": dict(V=151936, K=16, bs=(1, 64), w2="bf16", mode="prob",
                                         T=0.7, top_k=0, peak=8.0, draft_logits=True),
    "v248320_k16_int8_greedy": dict(V=248320, K=16, bs=(1, 16, 64), w2="int8", mode="greedy",
                                    T=1.0, top_k=0, peak=None, draft_logits=False),
    "v151936_k7_topk": dict(V=151936, K=7, bs=(64,), w2="bf16", mode="prob", T=1.0,
                            top_k=(512, 4096), peak=None, draft_logits=False),
}


def lmhead(M: int, d: int, V: int, seed: int = 0, std: float = 3.0):
    """Synthetic drafter LM head: hidden states [M, d] ~ N(0, 1) and LM-head rows [V, d]
    ~ N(0, std^2 / d), both bf16, so that the logits are about N(0, std^2) like the base
    logits of the walk's workloads."""
    g = torch.Generator().manual_seed(seed)
    hidden = torch.randn(M, d, generator=g).to(torch.bfloat16)
    head = (torch.randn(V, d, generator=g) * (std / d ** 0.5)).to(torch.bfloat16)
    return hidden, head

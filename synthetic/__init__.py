"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it draws seeded random numbers,
rounds them to the storage type, draws the kept mask units, and names the
workload shapes.  Both the oracle side and the GPU side receive exactly these
arrays, so neither side generates its own inputs.

bf16 tensors are carried as ``numpy.uint16`` arrays of bf16 bit patterns
(numpy has no bf16 type); ``bf16_bits_to_f32`` widens them exactly.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """Independent generator per (seed, stream) pair."""
    return np.random.default_rng([int(seed), int(stream)])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def normal(shape, seed: int, stream: int = 0, std: float = 1.0,
           dtype: str = "bf16") -> np.ndarray:
    """N(0, std^2) samples of `shape`; dtype 'f32' (float32) or 'bf16' (uint16 bits)."""
    x = rng(seed, stream).standard_normal(size=tuple(shape), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def keep_units(B: int, n_units: int, n_keep: int, seed: int,
               stream: int = 99) -> np.ndarray:
    """Kept mask-unit ids [B, n_keep] int32: the first n_keep of a seeded
    per-sample permutation of range(n_units), sorted ascending (the order in
    which boolean-mask indexing visits kept units)."""
    g = rng(seed, stream)
    out = np.empty((B, n_keep), dtype=np.int32)
    for b in range(B):
        out[b] = np.sort(g.permutation(n_units)[:n_keep])
    return out


# --------------------------------------------------------------------------
# Workload shapes (the pages' workloads; all values synthetic).
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class IHAShape:
    B: int
    N: int
    H: int
    P: int
    d: int

    @property
    def HP(self) -> int:
        return self.H * self.P


# Tiny IHA layer forward, fp32, non-causal.
TINY = IHAShape(B=1, N=128, H=4, P=2, d=32)
# LLaMA-2.4B layer shape (hidden 2560 = 20 heads x 128), P = 4.
LLAMA_PREMIX = IHAShape(B=1, N=8192, H=20, P=4, d=128)
# Pseudo-head attention, causal sliding window: 80 pseudo-heads, N = 4096.
LLAMA_WINDOW = IHAShape(B=1, N=4096, H=20, P=4, d=128)
WINDOW_KEYS = 1024          # W = WSL + 1 keys including the diagonal
# Long context layer forward with RoPE (base 10000) and causal attention.
LONG_CTX = IHAShape(B=2, N=16384, H=20, P=4, d=128)
ROPE_BASE = 10000.0


@dataclass(frozen=True)
class MaskUnitShape:
    B: int = 128
    grid_h: int = 56
    grid_w: int = 56
    mu_h: int = 8
    mu_w: int = 8
    n_keep: int = 20
    C: int = 96

    @property
    def n_units(self) -> int:
        return (self.grid_h // self.mu_h) * (self.grid_w // self.mu_w)

    @property
    def unit_tokens(self) -> int:
        return self.mu_h * self.mu_w


# Hiera-Base MAE stage 1: 224x224 -> 56x56 tokens, 8x8 mask units, mask
# ratio 0.6 keeps 20 of 49 units, embed dim 96 (one head of width 96).
HIERA_MU = MaskUnitShape()


@dataclass(frozen=True)
class QPoolShape:
    B: int = 128
    n_units: int = 20       # kept mask units per sample (the MAE keeps 20 of 49)
    T: int = 64             # tokens per unit entering the block (stage-1 resolution)
    q_stride: int = 4       # 2 x 2 spatial pooling, flattened
    heads: int = 2
    head_dim: int = 96      # dim_out 192 of Hiera-Base stage 2

    @property
    def Tq(self) -> int:
        return self.T // self.q_stride


# Hiera-Base MAE, first block of stage 2: mask-unit attention whose queries
# are max-pooled 4:1 (q_stride = 4) over the 64 tokens of each kept unit.
HIERA_QPOOL = QPoolShape()


def premix_weight(H: int, P: int, seed: int, stream: int) -> np.ndarray:
    """W[H, P, H] float32 ~ N(0, 1/H)."""
    return normal((H, P, H), seed, stream, std=1.0 / math.sqrt(H), dtype="f32")

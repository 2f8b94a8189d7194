"""Seeded synthetic inputs for the 4-bit weight-quantized linear.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic, so the CPU oracle's tests and the CUDA path's tests can both take their
inputs from it.

Distributions (Llama-shaped synthetic workloads; there are no trained weights here):
  x      ~ N(0, 1) float32, [M, K] row-major
  qweight  uniform bytes, [N, ceil(K/2)] uint8 -- two independent uniform nibbles per
           byte, i.e. uniform codes 0..15 (signed value code - 8); for odd K the last
           byte's high nibble is padding and is random too (it must never be read)
  scales ~ U(0.005, 0.02), [ceil(K/group_size), N]; float16 scales are drawn in float32
           and rounded to nearest-even by numpy, so both sides read the same bits
  bias   ~ N(0, 0.1) float32, [N], or None
The generator is numpy PCG64(seed).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np


@dataclass
class Case:
    M: int
    N: int
    K: int
    group_size: int
    x: np.ndarray            # float32 [M, K]
    qweight: np.ndarray      # uint8 [N, ceil(K/2)]
    scales: np.ndarray       # float32 or float16 [ceil(K/gs), N]
    bias: Optional[np.ndarray]  # float32 [N] or None

    @property
    def scale_f16(self) -> bool:
        return self.scales.dtype == np.float16


def packed_row_bytes(K: int) -> int:
    return (K + 1) // 2


def num_groups(K: int, group_size: int) -> int:
    return -(-K // group_size)


def make_case(M: int, N: int, K: int, group_size: int, scale_f16: bool = False,
              bias: bool = False, seed: int = 0) -> Case:
    """Random case with the distributions in the module docstring."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K), dtype=np.float32)
    qweight = rng.integers(0, 256, size=(N, packed_row_bytes(K)), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, size=(num_groups(K, group_size), N)).astype(np.float32)
    scales = s.astype(np.float16) if scale_f16 else s
    b = rng.normal(0.0, 0.1, size=N).astype(np.float32) if bias else None
    return Case(M, N, K, group_size, x, qweight, scales, b)


def make_dyadic_case(M: int, N: int, K: int, group_size: int, scale_f16: bool = False,
                     bias: bool = False, seed: int = 0) -> Case:
    """Inputs on which every fp32 / tf32 / bf16 path is exact.

    x in {-2, -1.5, ..., 2} (halves), scales in {1/8, 1/4, 1/2, 1}, bias in multiples
    of 1/8 within [-4, 4].  Each product x * (q - 8) * s is a multiple of 1/16 bounded
    by 16, so every partial sum of up to 2^19 terms stays an exactly representable
    float32; any correct summation order gives the same bits.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    x = (rng.integers(-4, 5, size=(M, K)).astype(np.float32) * np.float32(0.5))
    qweight = rng.integers(0, 256, size=(N, packed_row_bytes(K)), dtype=np.uint8)
    e = rng.integers(-3, 1, size=(num_groups(K, group_size), N))
    s = np.ldexp(np.ones_like(e, dtype=np.float32), e).astype(np.float32)
    scales = s.astype(np.float16) if scale_f16 else s
    b = (rng.integers(-32, 33, size=N).astype(np.float32) / np.float32(8)) if bias else None
    return Case(M, N, K, group_size, x, qweight, scales, b)


def fill_codes(N: int, K: int, code: int) -> np.ndarray:
    """A packed weight whose every nibble (padding included) holds ``code``."""
    return np.full((N, packed_row_bytes(K)), (code << 4) | code, dtype=np.uint8)


@dataclass
class BackwardCase:
    """Seeded inputs of the input gradient d_x = d_out @ dequant(W)."""
    M: int
    N: int
    K: int
    group_size: int
    d_out: np.ndarray    # float32 [M, N]
    qweight: np.ndarray  # uint8 [N, ceil(K/2)]
    scales: np.ndarray   # float32 or float16 [ceil(K/gs), N]

    @property
    def scale_f16(self) -> bool:
        return self.scales.dtype == np.float16


def make_backward_case(M: int, N: int, K: int, group_size: int, scale_f16: bool = False,
                       seed: int = 0, dyadic: bool = False) -> BackwardCase:
    """d_out ~ N(0,1) (or halves in [-2, 2] with power-of-two scales when dyadic, so that
    every fp32 summation order is exact), uniform packed bytes, scales U(0.005, 0.02)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if dyadic:
        d_out = rng.integers(-4, 5, size=(M, N)).astype(np.float32) * np.float32(0.5)
        e = rng.integers(-3, 1, size=(num_groups(K, group_size), N))
        s = np.ldexp(np.ones_like(e, dtype=np.float32), e).astype(np.float32)
    else:
        d_out = rng.standard_normal((M, N)).astype(np.float32)
        s = rng.uniform(0.005, 0.02, size=(num_groups(K, group_size), N)).astype(np.float32)
    qweight = rng.integers(0, 256, size=(N, packed_row_bytes(K)), dtype=np.uint8)
    return BackwardCase(M, N, K, group_size, d_out, qweight,
                        s.astype(np.float16) if scale_f16 else s)


@dataclass
class RequantCase:
    """Seeded inputs of the re-quantisation of fp32 latents with frozen scales."""
    N: int
    K: int
    group_size: int
    latent: np.ndarray   # float32 [N, K]
    scales: np.ndarray   # float32 or float16 [ceil(K/gs), N]

    @property
    def scale_f16(self) -> bool:
        return self.scales.dtype == np.float16


def make_requant_case(N: int, K: int, group_size: int, scale_f16: bool = False,
                      seed: int = 0, specials: bool = False) -> RequantCase:
    """latent ~ N(0, 0.05) (quotients spread over the code range, some clamped), scales
    U(0.005, 0.02).  With specials: one group column of zero scales, NaN and +-Inf
    latents, and latents that are exact half-integer multiples of a power-of-two scale
    (round-to-even ties)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    G = num_groups(K, group_size)
    latent = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    s = rng.uniform(0.005, 0.02, size=(G, N)).astype(np.float32)
    if specials:
        s[rng.integers(0, G), :] = 0.0
        flat = latent.reshape(-1)
        idx = rng.choice(flat.size, size=min(flat.size, 6), replace=False)
        flat[idx[:2]] = np.nan
        flat[idx[2:4]] = np.inf
        flat[idx[4:]] = -np.inf
        n_tie = rng.integers(0, N)
        g_tie = rng.integers(0, G)
        s[g_tie, n_tie] = np.float32(0.015625)
        k0, k1 = g_tie * group_size, min(K, (g_tie + 1) * group_size)
        halves = rng.integers(-17, 16, size=k1 - k0).astype(np.float32) + np.float32(0.5)
        latent[n_tie, k0:k1] = halves * np.float32(0.015625)
    return RequantCase(N, K, group_size, latent, s.astype(np.float16) if scale_f16 else s)

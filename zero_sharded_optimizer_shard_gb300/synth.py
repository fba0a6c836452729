"""Seeded, counter-based synthetic inputs (host side).

This module only draws numbers; it holds none of the optimizer's arithmetic.
Its device twin (csrc/synth.cu, built as its own library) implements the same
definition independently, so any element of any synthetic tensor can be
regenerated on the host from its coordinates alone.

Definition
----------
mix64(z) is the SplitMix64 output function (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014; the public
splitmix64.c reference by S. Vigna):

    z ^= z >> 30; z *= 0xbf58476d1ce4e5b9
    z ^= z >> 27; z *= 0x94d049bb133111eb
    z ^= z >> 31                                   (all mod 2**64)

With GOLDEN = 0x9e3779b97f4a7c15 (the SplitMix64 increment):

    k0  = mix64(seed + GOLDEN * (stream + 1))
    k1  = mix64(k0   + GOLDEN * (step   + 1))
    key = mix64(k1   + GOLDEN * (rank   + 1))
    draw(key, index, j) = mix64(key + GOLDEN * (8 * index + j + 1)),  j = 0..7

Normal(0, sigma) by Irwin-Hall(12): draws j = 0..5 each give two 24-bit
uniforms (bits 40..63 and 8..31); their integer sum s is exact.  Then
    x = (f32(s) * 2**-24 - 6.0f) * f32(sigma_eff)
with each operation one IEEE binary32 operation rounded to nearest-even.
sigma_eff = outlier_sigma when (draw j=6 >> 32) < floor(outlier_p * 2**32),
else sigma.  A bf16 sample is the upper 16 bits of x (truncation).
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)
_MASK24 = np.uint64(0xFFFFFF)


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def _u64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.uint64)


def key(seed: int, stream: int, step: int, rank: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k0 = mix64(_u64([seed]) + GOLDEN * _u64([stream + 1]))
        k1 = mix64(k0 + GOLDEN * _u64([step + 1]))
        k2 = mix64(k1 + GOLDEN * _u64([rank + 1]))
    return k2[0]


def draw(k: np.uint64, index: np.ndarray, j: int) -> np.ndarray:
    index = _u64(index)
    with np.errstate(over="ignore"):
        return mix64(k + GOLDEN * (index * np.uint64(8) + np.uint64(j + 1)))


def uniform_u64(seed: int, stream: int, step: int, rank: int, index) -> np.ndarray:
    """Raw 64-bit draw j=7 at the given coordinates (used for list shapes)."""
    return draw(key(seed, stream, step, rank), _u64(index), 7)


def normal_f32(seed: int, stream: int, step: int, rank: int, index,
               sigma: float, outlier_p: float = 0.0, outlier_sigma: float = 0.0) -> np.ndarray:
    """fp32 Irwin-Hall(12) normal samples at flat indices `index`."""
    k = key(seed, stream, step, rank)
    index = _u64(np.atleast_1d(index))
    s = np.zeros(index.shape, dtype=np.uint64)
    for j in range(6):
        d = draw(k, index, j)
        s += (d >> np.uint64(40)) & _MASK24
        s += (d >> np.uint64(8)) & _MASK24
    x = s.astype(np.int64).astype(np.float32)
    x = x * np.float32(2.0 ** -24)
    x = x - np.float32(6.0)
    sig = np.full(index.shape, np.float32(sigma), dtype=np.float32)
    if outlier_p > 0.0:
        thr = np.uint64(int(outlier_p * 2.0 ** 32))
        out = (draw(k, index, 6) >> np.uint64(32)) < thr
        sig[out] = np.float32(outlier_sigma)
    return (x * sig).astype(np.float32)


def normal_bf16(seed: int, stream: int, step: int, rank: int, index,
                sigma: float, outlier_p: float = 0.0, outlier_sigma: float = 0.0) -> np.ndarray:
    """bf16 samples (uint16 bit patterns): upper half of the fp32 sample."""
    x = normal_f32(seed, stream, step, rank, index, sigma, outlier_p, outlier_sigma)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)

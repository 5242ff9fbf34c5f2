"""Seeded synthetic inputs shared by the CUDA path, the oracle checks and the bench.

This module holds no convolution arithmetic. It turns (seed, count, distribution,
dtype) into raw 16-bit words, nothing more; callers decide the tensor shapes.

Generator (fixed, documented so any consumer can reproduce it):

* splitmix64: state_i = seed + (i + 1) * 0x9E3779B97F4A7C15 (mod 2^64), then the
  standard splitmix64 finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9,
  xor-shift 27, multiply 0x94D049BB133111EB, xor-shift 31).
* uniform in [0, 1): the top 53 bits of the finalised word times 2^-53.
* uniform[a, b]: a + (b - a) * u.
* normal(mean, std): Box-Muller on consecutive pairs (u1 = word 2j, u2 = word
  2j + 1): mean + std * sqrt(-2 ln(1 - u1)) * cos(2 pi u2) for element 2j and
  the sine branch for element 2j + 1.
* integers in {lo..hi}: lo + floor(u * (hi - lo + 1)).
* rounding to the storage dtype: float64 -> float32 (round to nearest even),
  then float32 -> bf16 by round-to-nearest-even on the bit pattern, or
  float32 -> fp16 by numpy's round-to-nearest-even cast.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """n finalised splitmix64 words for the given seed (uint64 array)."""
    with np.errstate(over="ignore"):
        i = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, n: int) -> np.ndarray:
    w = splitmix64(seed, n)
    return (w >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def values(seed: int, n: int, dist: str = "uniform", a: float = -1.0, b: float = 1.0) -> np.ndarray:
    """float64 values. dist: 'uniform' (a, b), 'normal' (a = mean, b = std),
    'int' (integers a..b inclusive)."""
    if dist == "uniform":
        return a + (b - a) * uniform01(seed, n)
    if dist == "normal":
        m = n + (n & 1)
        u = uniform01(seed, m)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        out = np.empty(m, dtype=np.float64)
        out[0::2] = r * np.cos(2.0 * np.pi * u2)
        out[1::2] = r * np.sin(2.0 * np.pi * u2)
        return a + b * out[:n]
    if dist == "int":
        lo, hi = int(a), int(b)
        u = uniform01(seed, n)
        return lo + np.floor(u * (hi - lo + 1))
    raise ValueError(f"unknown distribution {dist!r}")


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); returns uint16 words."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    out = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(v, dtype=np.float32))
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def to_bits(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the 16-bit storage dtype ('bf16' or 'fp16')."""
    f32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(f32)
    if dtype == "fp16":
        return f32.astype(np.float16).view(np.uint16)
    raise ValueError(f"unsupported storage dtype {dtype!r}")


def tensor_bits(seed: int, n: int, dtype: str, dist: str = "uniform", a: float = -1.0,
                b: float = 1.0) -> np.ndarray:
    """n seeded values rounded to dtype, as uint16 words."""
    return to_bits(values(seed, n, dist, a, b), dtype)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode 16-bit words to float32 (exact for both bf16 and fp16)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    raise ValueError(f"unsupported storage dtype {dtype!r}")

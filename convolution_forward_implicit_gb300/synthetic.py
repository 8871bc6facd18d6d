"""Seeded synthetic inputs shared by the tests, the benchmark and the checker.

This module draws numbers and rounds them to the storage type; it holds none of
the convolution's arithmetic.  Both the CUDA path and the CPU oracle receive
exactly the arrays produced here.

Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used in counter form: output ``i`` of a stream
with seed ``s`` is ``mix(s + (i + 1) * GAMMA)``.  Uniforms take the top 53 bits.
Normals come from the Box-Muller transform (Box and Muller, 1958), one pair of
uniforms per pair of normals.

Values are drawn in float64, rounded once to float32, and for bf16 tensors
rounded once more from float32 to bf16 with round-to-nearest-even.  bf16 arrays
are carried as ``uint16`` bit patterns.

Seeds: the stream of tensor ``t`` (x=0, w=1, bias=2) of workload ``i`` uses seed
``BASE_SEED + 1000 * i + t``.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

TENSOR_X, TENSOR_W, TENSOR_BIAS = 0, 1, 2


def stream_seed(workload_index: int, tensor_id: int) -> int:
    return BASE_SEED + 1000 * int(workload_index) + int(tensor_id)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream ``seed``."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, count: int) -> np.ndarray:
    """``count`` float64 uniforms in [0, 1) from the top 53 bits."""
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _CHUNK):
        n = min(_CHUNK, count - s)
        out[s:s + n] = (splitmix64(seed, s, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return out


def normal(seed: int, count: int) -> np.ndarray:
    """``count`` float64 N(0,1) values by Box-Muller on consecutive uniform pairs."""
    pairs = (count + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float64)
    for s in range(0, pairs, _CHUNK):
        n = min(_CHUNK, pairs - s)
        u = (splitmix64(seed, 2 * s, 2 * n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))          # 1 - u1 lies in (0, 1]
        th = 2.0 * np.pi * u2
        out[2 * s:2 * (s + n):2] = r * np.cos(th)
        out[2 * s + 1:2 * (s + n):2] = r * np.sin(th)
    return out[:count]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(v64: np.ndarray, dtype: str) -> np.ndarray:
    """float64 draw -> float32 -> (bf16 bits).  dtype is 'f32' or 'bf16'."""
    f = v64.astype(np.float32)
    if dtype == "f32":
        return f
    if dtype == "bf16":
        return f32_to_bf16_bits(f)
    raise ValueError(dtype)


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """The exact value of a stored tensor as float32 (every bf16 value is a float32 value)."""
    return bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def gen_normal(seed: int, shape, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    return to_storage(normal(seed, n), dtype).reshape(shape)


def gen_uniform_pm(seed: int, shape, bound: float, dtype: str) -> np.ndarray:
    """U(-bound, +bound)."""
    n = int(np.prod(shape))
    return to_storage(bound * (2.0 * uniform01(seed, n) - 1.0), dtype).reshape(shape)


def gen_int(seed: int, shape, lo: int, hi: int, dtype: str) -> np.ndarray:
    """Integers uniform in [lo, hi] stored in ``dtype`` (exact in f32 and bf16 for small ranges)."""
    n = int(np.prod(shape))
    u = uniform01(seed, n)
    v = np.floor(lo + u * (hi - lo + 1)).clip(lo, hi)
    return to_storage(v, dtype).reshape(shape)

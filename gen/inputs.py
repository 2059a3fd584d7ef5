"""Seeded synthetic inputs shared by the oracle, the tests and the bench.

This module draws random numbers and rounds them to bfloat16; it contains none of the
attention arithmetic.  Both sides of every parity check (the float64 CPU oracle and the
CUDA path) consume the exact same bf16 bit patterns produced here.

Generator (published definitions, restated):

* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014; the 64-bit finaliser popularised by Vigna): the i-th output of stream
  ``seed`` is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)`` with the two xor-shift-multiply
  rounds below.  It is counter based, so any element can be generated independently and
  chunking does not change the values.
* uniform in (0, 1]: ``((z >> 11) + 1) * 2**-53``.
* Box-Muller (1958): a pair (u1, u2) gives ``r*cos(2*pi*u2)`` and ``r*sin(2*pi*u2)`` with
  ``r = sqrt(-2 ln u1)``; element 2p takes the cosine of pair p and element 2p+1 the sine.
* bfloat16 rounding: round-to-nearest-even from the float64 sample directly (no detour
  through float32, so there is no double rounding).
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per generation chunk (bounds host memory for 67M-element tensors)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the splitmix64 stream ``seed`` (uint64)."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Uniform float64 samples in (0, 1] from splitmix64 outputs ``start..start+count-1``."""
    z = splitmix64(seed, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal_f64(seed: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """``n`` samples of N(0, sigma^2) in float64 (Box-Muller over splitmix64 uniforms)."""
    out = np.empty(n, dtype=np.float64)
    for e0 in range(0, n, _CHUNK):
        e1 = min(n, e0 + _CHUNK)          # e0 is even because _CHUNK is even
        npairs = (e1 - e0 + 1) // 2
        u = uniform01(seed, e0, 2 * npairs)  # pair p uses uniforms 2p and 2p+1 of the stream
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = (2.0 * np.pi) * u2
        pair = np.empty(2 * npairs, dtype=np.float64)
        pair[0::2] = r * np.cos(th)
        pair[1::2] = r * np.sin(th)
        out[e0:e1] = sigma * pair[: e1 - e0]
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (round to nearest, ties to even); uint16 bit patterns.

    Works on the float64 bit pattern: keep 7 of the 52 fraction bits with RNE, then the value
    is exactly a float32 whose top 16 bits are the bf16 pattern.  Values below the smallest
    normal bf16 go through float32 (they do not occur for these distributions).
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    drop = np.uint64(45)
    with np.errstate(over="ignore"):
        lsb = (b >> drop) & np.uint64(1)
        r = (b + (np.uint64((1 << 44) - 1) + lsb)) >> drop << drop
    y = r.view(np.float64).astype(np.float32)
    bits = (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    tiny = np.abs(x) < 2.0 ** -126
    if np.any(tiny):
        f = x[tiny].astype(np.float32).view(np.uint32)
        rr = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        bits[tiny] = rr.astype(np.uint16)
    return bits


def bf16_normal(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16, C order) of N(0, sigma^2) samples of the given shape."""
    n = int(np.prod(shape))
    return f64_to_bf16_bits(normal_f64(seed, n, sigma)).reshape(shape)


def uniform_int(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform on [lo, hi] (``lo + z mod (hi-lo+1)``; bias < 2^-52)."""
    z = splitmix64(seed, 0, n)
    return (np.int64(lo) + (z % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int64)


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    """int32 exclusive prefix sum [0, L0, L0+L1, ...] of the sequence lengths."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)

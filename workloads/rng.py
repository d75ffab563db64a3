"""Counter-based random numbers for the synthetic workloads.

Every random value is a pure function of (seed, stream name, flat index), so
any slice of any tensor (for example the rows of a few sequences) can be
regenerated on its own and equals the same slice of the full tensor.

The generator is SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used in counter mode: the
i-th output of a stream is the SplitMix64 finaliser applied to
``key + (i + 1) * 0x9E3779B97F4A7C15`` (mod 2**64).  Normal deviates use the
Box-Muller transform on two consecutive uniforms.

This module holds no arithmetic of the decoding method itself.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO_POW_M53 = 1.0 / 9007199254740992.0  # 2**-53


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _fnv1a64(text: str) -> int:
    """64-bit FNV-1a hash of a UTF-8 string (stable across runs and hosts)."""
    h = 0xCBF29CE484222325
    for byte in text.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, name: str) -> np.uint64:
    """Key of the named stream under ``seed``."""
    with np.errstate(over="ignore"):
        base = np.uint64(_fnv1a64(name)) ^ (np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * _GOLDEN)
        return _mix(np.array([base], dtype=np.uint64))[0]


def raw_u64(seed: int, name: str, start: int, stop: int) -> np.ndarray:
    """Outputs ``start .. stop-1`` of the named stream as uint64."""
    key = stream_key(seed, name)
    idx = np.arange(start, stop, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + (idx + np.uint64(1)) * _GOLDEN)


def uniform(seed: int, name: str, start: int, stop: int) -> np.ndarray:
    """Uniform float64 in the open interval (0, 1), 53-bit resolution."""
    r = raw_u64(seed, name, start, stop)
    # the top 53 bits fit an int64 exactly; int64 -> float64 is the fast path
    return ((r >> np.uint64(11)).view(np.int64).astype(np.float64) + 0.5) * _TWO_POW_M53


def _normal_serial(seed: int, name: str, start: int, stop: int) -> np.ndarray:
    u = uniform(seed, name, 2 * start, 2 * stop)
    u1 = u[0::2]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


_CHUNK = 1 << 18


def normal(seed: int, name: str, start: int, stop: int) -> np.ndarray:
    """Standard normal float64 deviates ``start .. stop-1`` (Box-Muller, cosine branch).

    Deviate i consumes uniforms 2i and 2i+1 of the stream.  Large ranges are
    cut into fixed chunks drawn on a thread pool; the values do not depend on
    the chunking.
    """
    n = stop - start
    if n <= 2 * _CHUNK:
        return _normal_serial(seed, name, start, stop)
    out = np.empty(n, dtype=np.float64)
    bounds = list(range(start, stop, _CHUNK)) + [stop]

    def work(i):
        lo, hi = bounds[i], bounds[i + 1]
        out[lo - start:hi - start] = _normal_serial(seed, name, lo, hi)

    with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(len(bounds) - 1)))
    return out


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  NaN is not expected in the
    synthetic inputs and is not handled specially.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        rounded = b + np.uint32(0x7FFF) + lsb
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_float(bits: np.ndarray, dtype=np.float64) -> np.ndarray:
    """Exact conversion of bfloat16 bit patterns (uint16) to float32/float64."""
    f32 = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    return f32.astype(dtype)

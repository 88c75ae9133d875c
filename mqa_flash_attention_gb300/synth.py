"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws numbers.  It holds none of the attention arithmetic:
no scores, no softmax, no masking.  Everything is plain numpy on the host, so the
same seed gives the same bytes on any machine (x86 or Arm) and with any numpy
version, because the generator is written out here instead of taken from
``numpy.random``:

* ``splitmix64`` (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) used as a counter-based generator: draw ``i`` of
  stream ``s`` is ``mix64(key(seed, s) + (i + 1) * GOLDEN)``;
* 53-bit uniforms ``(x >> 11) * 2**-53``;
* Box-Muller (Box and Muller, "A note on the generation of random normal
  deviates", 1958) for N(0, 1), rounded to fp16 with round-to-nearest-even.

Sub-streams: every tensor of a workload has its own stream id, so the K rows do
not change when T changes, for instance.
"""

from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids of the tensors of one attention call.
STREAM_Q = 1
STREAM_K_RAW = 2
STREAM_V_RAW = 3
STREAM_K_COMP = 4
STREAM_V_COMP = 5
STREAM_IDX = 6
STREAM_MASK = 7
STREAM_IDX_Q = 8      # indexer query vectors
STREAM_IDX_K = 9      # indexer compressed rows
STREAM_IDX_W = 10     # indexer head weights
STREAM_CMP_KV = 11    # compressor input rows
STREAM_CMP_S = 12     # compressor score rows


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    base = np.array([(int(seed) & 0xFFFFFFFF) | ((int(stream) & 0xFFFFFFFF) << 32)], dtype=np.uint64)
    return _mix64(base)[0]


def uint64_stream(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+n-1`` of the counter-based splitmix64 stream."""
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix64(_key(seed, stream) + ctr * GOLDEN)


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    x = uint64_stream(seed, stream, n, offset)
    return (x >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """N(0, 1) doubles by Box-Muller over pairs of uniforms."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    u1 = 1.0 - u[0::2]          # (0, 1]: log is finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def normal_f32(seed: int, stream: int, shape) -> np.ndarray:
    """N(0, 1) rounded to fp32, C-contiguous."""
    n = int(np.prod(shape))
    return normal_f64(seed, stream, n).astype(np.float32).reshape(shape)


def normal_f16(seed: int, stream: int, shape) -> np.ndarray:
    """N(0, 1) rounded to fp16 (round-to-nearest-even), C-contiguous."""
    n = int(np.prod(shape))
    return normal_f64(seed, stream, n).astype(np.float16).reshape(shape)


def sample_without_replacement(seed: int, stream: int, row: int, population: int, k: int) -> np.ndarray:
    """``k`` distinct integers drawn uniformly from ``[0, population)``, sorted.

    Each candidate gets an independent 64-bit key from its own counter range
    (``row * 2**32 + candidate``); the ``k`` smallest keys win.  That is a
    uniformly random ``k``-subset (ties have probability ~2**-64 and break by
    candidate number)."""
    if k > population:
        raise ValueError(f"cannot draw {k} distinct values from {population}")
    keys = uint64_stream(seed, stream, population, offset=row << 32)
    order = np.lexsort((np.arange(population), keys))
    return np.sort(order[:k]).astype(np.int32)

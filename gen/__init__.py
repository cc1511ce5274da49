"""Seeded synthetic inputs for the FP32 SGEMM workloads.

This module is the one piece that both the CPU oracle's tests and the GPU path's
tests and benchmark use.  It draws random matrices and nothing else: it holds no
part of the matrix product.

Generator
---------
SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used as a counter-based generator: output ``i``
(``i = 0, 1, ...``) of the stream whose state starts at ``s`` is
``mix64(s + (i + 1) * GAMMA)``, which is exactly the ``i``-th value the
sequential SplitMix64 returns when seeded with ``s``.

A stream is keyed by ``(seed, stream_id)`` through the start state
``s = seed * 256 + stream_id``.  Matrices are filled in row-major order,
element ``(r, c)`` of an ``rows x cols`` matrix taking draw ``r * cols + c``
(or draws ``2(r*cols+c)`` and ``2(r*cols+c)+1`` for the normal distribution).

Distributions
-------------
* ``uniform``: ``u = (x >> 11) * 2**-53`` in [0, 1); value ``2u - 1`` (exact in
  FP64), rounded to FP32: the interval [-1, 1].
* ``normal``: Box-Muller on two draws, ``u1 = ((x1 >> 11) + 1) * 2**-53`` in
  (0, 1] and ``u2 = (x2 >> 11) * 2**-53``; value
  ``sqrt(-2 ln u1) * cos(2 pi u2)`` in FP64, rounded to FP32.
* ``int``: ``((x >> 32) * 9) >> 32`` in {0..8}, minus 4: small integers in
  [-4, 4], stored as FP32.
"""

from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_MUL1 = 0xBF58476D1CE4E5B9
_MUL2 = 0x94D049BB133111EB

#: Stream ids for the two operands and their small-integer copies.
STREAM_A = 0
STREAM_B = 1
STREAM_A_INT = 2
STREAM_B_INT = 3

_CHUNK = 1 << 22
_U64 = np.uint64


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> _U64(30))) * _U64(_MUL1)
    z = (z ^ (z >> _U64(27))) * _U64(_MUL2)
    return z ^ (z >> _U64(31))


def stream_state(seed: int, stream_id: int) -> int:
    """Start state of the stream keyed by ``(seed, stream_id)``."""
    if seed < 0 or not (0 <= stream_id < 256):
        raise ValueError("seed must be >= 0 and stream_id in [0, 256)")
    return (seed * 256 + stream_id) & 0xFFFFFFFFFFFFFFFF


def draws(state: int, start: int, count: int) -> np.ndarray:
    """Raw uint64 outputs ``start .. start+count-1`` of the stream at ``state``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _U64(state) + idx * _U64(GAMMA)
    return mix64(z)


def _unit53(x: np.ndarray) -> np.ndarray:
    return (x >> _U64(11)).astype(np.float64) * (2.0 ** -53)


def _fill(out: np.ndarray, state: int, dist: str) -> None:
    flat = out.reshape(-1)
    n = flat.size
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        cnt = hi - lo
        if dist == "uniform":
            u = _unit53(draws(state, lo, cnt))
            flat[lo:hi] = (2.0 * u - 1.0).astype(np.float32)
        elif dist == "normal":
            x = draws(state, 2 * lo, 2 * cnt)
            u1 = _unit53(x[0::2]) + 2.0 ** -53
            u2 = _unit53(x[1::2])
            flat[lo:hi] = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)).astype(np.float32)
        elif dist == "int":
            x = draws(state, lo, cnt)
            v = ((x >> _U64(32)) * _U64(9)) >> _U64(32)
            flat[lo:hi] = v.astype(np.float32) - np.float32(4.0)
        else:
            raise ValueError(f"unknown distribution {dist!r}")


def matrix(seed: int, stream_id: int, rows: int, cols: int, dist: str = "uniform") -> np.ndarray:
    """A ``rows x cols`` row-major float32 matrix drawn from stream ``(seed, stream_id)``."""
    if rows < 0 or cols < 0:
        raise ValueError("negative matrix extent")
    out = np.empty((rows, cols), dtype=np.float32)
    if out.size:
        _fill(out, stream_state(seed, stream_id), dist)
    return out


def operands(M: int, N: int, K: int, seed: int, dist: str = "uniform", integer_copy: bool = False):
    """The pair (A, B) of an SGEMM problem: A is M x K, B is K x N, both row-major FP32.

    ``integer_copy`` selects the independent small-integer streams instead of
    ``dist`` (the integer copy of a workload is a separate draw, not a rounding
    of the real-valued one).
    """
    if integer_copy:
        return (matrix(seed, STREAM_A_INT, M, K, "int"),
                matrix(seed, STREAM_B_INT, K, N, "int"))
    return matrix(seed, STREAM_A, M, K, dist), matrix(seed, STREAM_B, K, N, dist)


def strided(mat: np.ndarray, ld: int, fill: float = np.nan) -> np.ndarray:
    """Copy ``mat`` into a row-major buffer with leading dimension ``ld >= cols``.

    The returned array has shape ``(rows, ld)``; columns ``cols..ld-1`` hold
    ``fill`` (NaN by default, so that a kernel reading the gap shows up).
    """
    rows, cols = mat.shape
    if ld < cols:
        raise ValueError("leading dimension smaller than the row length")
    buf = np.full((rows, max(ld, 1)), fill, dtype=np.float32)
    buf[:, :cols] = mat
    return buf


#: The synthetic workloads, by name: the five of the pages' examples, one larger square product
#: and one long-K product with few output tiles.
#: Each entry: (M, N, K, dist, seed).
WORKLOADS = {
    "tiny_6x6x9": (6, 6, 9, "uniform", 0),
    "square_1024": (1024, 1024, 1024, "uniform", 1),
    "square_8192": (8192, 8192, 8192, "normal", 2),
    "ragged_3001x4999x2047": (3001, 4999, 2047, "uniform", 3),
    "skinny_16384x16384x32": (16384, 16384, 32, "uniform", 4),
    # not one of the pages' examples: the headline's square product at twice
    # the size, where the FP32 kernel's L2 reuse is tested hardest
    "square_16384": (16384, 16384, 16384, "normal", 5),
    # not one of the pages' examples: four output tiles over a long K, the
    # load imbalance that tiling alone leaves (few tiles for many SMs)
    "longk_256x256x65536": (256, 256, 65536, "uniform", 6),
}

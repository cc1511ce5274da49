"""Counting side of the oracle: a CPU simulator of the pages' SGEMM kernels
(test infrastructure only; no GPU code uses it).

It enumerates the threads of the naive kernel, the shared-memory tiled kernel
and the 2-D register-tiled kernel as the pages describe them, and counts the
loads each thread issues from global memory and from shared memory, plus the
multiply-adds.  A separate bank model gives the conflict degree of one warp-wide
shared-memory access.

Sources
-------
* Naive kernel: one thread per output element, each reading one A and one B
  element per trip of its K-long loop ("SGEMM: Shared Memory Tiling
  Visualizer", "Why exactly 2 x M x N x K for the naive approach?";
  "Shared Memory Tiling", "The naive kernel").
* Tiled kernel: a TILE x TILE thread block loads one A element and one B element
  per thread per tile step, zero-filling out-of-range slots, then each thread
  reads a row of the A tile and a column of the B tile from shared memory
  ("SGEMM: Shared Memory Tiling Visualizer", tiled kernel listing;
  "Memory hierarchy -- visual walkthrough", Steps 3-4).
* 2-D register tiling: per inner step each thread loads TM values of A and TN of
  B into registers and does TM x TN multiply-adds ("SGEMM: 2D Register Tiling
  Visualizer", listing and "Why 2D Register Tiling Dominates").
* Banks: 32 banks of 4-byte words; a warp access is serialised by the largest
  number of distinct words that fall in one bank, identical words being a
  broadcast ("Memory hierarchy -- visual walkthrough", Step 6;
  "SGEMM: Shared Memory Tiling Visualizer", "Why no padding?").

Readings where the pages leave a step open
-----------------------------------------
* The tile loop runs ceil(K / TILE) times (the visualizer listing writes
  ``ceil(K / 2)`` with integer operands; the intended count is the ceiling).
* The undefined ``tileColA`` / ``tileRowB`` are ``tileIdx*TILE + tx`` and
  ``tileIdx*TILE + ty``.
* A zero-filled (masked) slot issues no global load and is not counted.
* Counts are in elements; bytes are four times as many (FP32).
* Register reads are counted as two per multiply-add; no page prints a value
  for them, so that count is parity unpinned.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BANKS = 32


@dataclass(frozen=True)
class Counts:
    threads: int            # threads that compute an in-range output element
    launched_threads: int   # threads launched (including padding threads)
    global_reads: int       # global-memory element loads issued
    shared_reads: int       # shared-memory element reads
    fma: int                # multiply-adds on in-range output elements
    tile_steps: int = 0     # steps of the tile loop (0 for the naive kernel)
    padded_slots: int = 0   # tile slots zero-filled instead of loaded

    @property
    def reads_per_thread(self) -> float:
        return self.global_reads / self.threads if self.threads else 0.0


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def naive(M: int, N: int, K: int) -> Counts:
    """The naive kernel: each in-range thread runs K trips, loading A and B once each."""
    rows = np.arange(M, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64)
    # one thread per output element; each trip of its loop loads one A, one B
    trips = np.full((rows.size, cols.size), K, dtype=np.int64) if M and N else np.zeros((0, 0), np.int64)
    loads_per_thread = 2 * trips
    threads = int(trips.size)
    return Counts(threads=threads, launched_threads=threads,
                  global_reads=int(loads_per_thread.sum()), shared_reads=0,
                  fma=int(trips.sum()))


def tiled(M: int, N: int, K: int, T: int) -> Counts:
    """The shared-memory tiled kernel with TILE = T and zero-filled edges.

    The grid is ceil(N/T) x ceil(M/T) blocks of T x T threads.  At each tile step
    a thread (tx, ty) of the block at (bx, by) loads A[row][step*T + tx] if that
    slot is inside A and B[step*T + ty][col] if that slot is inside B
    (row = by*T + ty, col = bx*T + tx), then reads T values of each tile.
    """
    if T < 1:
        raise ValueError("tile size must be >= 1")
    gm, gn = _ceil_div(M, T), _ceil_div(N, T)
    steps = _ceil_div(K, T)
    row = np.arange(gm * T, dtype=np.int64)     # globalRow over the whole grid
    col = np.arange(gn * T, dtype=np.int64)     # globalCol over the whole grid
    tx, ty = col % T, row % T
    launched = row.size * col.size
    a_loads = b_loads = 0
    for step in range(steps):
        a_issue = np.logical_and.outer(row < M, step * T + tx < K)
        b_issue = np.logical_and.outer(step * T + ty < K, col < N)
        a_loads += int(np.count_nonzero(a_issue))
        b_loads += int(np.count_nonzero(b_issue))
    shared = launched * steps * 2 * T
    inside = int(np.count_nonzero(np.logical_and.outer(row < M, col < N)))
    padded = 2 * launched * steps - (a_loads + b_loads)
    return Counts(threads=inside, launched_threads=launched,
                  global_reads=a_loads + b_loads, shared_reads=shared,
                  fma=inside * K, tile_steps=steps, padded_slots=padded)


def register_tiled(M: int, N: int, K: int, BM: int, BN: int, BK: int, TM: int, TN: int) -> Counts:
    """The 2-D register-tiled kernel: BM x BN output blocks, BK-deep tile steps,
    each of the (BM/TM)*(BN/TN) threads owning a TM x TN block of outputs.

    Per tile step the block loads the in-range part of a BM x BK slab of A and a
    BK x BN slab of B; per inner step (dotIdx) each thread reads TM values of the
    A slab and TN values of the B slab and does TM*TN multiply-adds.
    """
    if BM % TM or BN % TN:
        raise ValueError("thread tile must divide the block tile")
    gm, gn = _ceil_div(M, BM), _ceil_div(N, BN)
    steps = _ceil_div(K, BK)
    threads_per_block = (BM // TM) * (BN // TN)
    blocks = gm * gn
    g_reads = 0
    for by in range(gm):
        rows_in = min(BM, M - by * BM)
        for bx in range(gn):
            cols_in = min(BN, N - bx * BN)
            for step in range(steps):
                k_in = min(BK, K - step * BK)
                g_reads += rows_in * k_in + k_in * cols_in
    shared = blocks * threads_per_block * steps * BK * (TM + TN)
    return Counts(threads=M * N, launched_threads=blocks * threads_per_block,
                  global_reads=g_reads, shared_reads=shared, fma=M * N * K,
                  tile_steps=steps)


def inner_step_ratio(TM: int, TN: int):
    """(shared-memory reads, multiply-adds) of one thread in one inner step."""
    reads = 0
    fmas = 0
    for _ in range(TM):   # regM[i] = As[...]
        reads += 1
    for _ in range(TN):   # regN[j] = Bs[...]
        reads += 1
    for _ in range(TM):
        for _ in range(TN):
            fmas += 1
    return reads, fmas


def register_reads(counts: Counts) -> int:
    """Register operand reads under the two-per-multiply-add convention (unpinned)."""
    return 2 * counts.fma


def bank_degree(word_addresses, banks: int = BANKS) -> int:
    """Serialisation degree S of one warp access to shared memory.

    ``word_addresses`` are the 4-byte word indices the threads touch.  S is the
    largest number of distinct words that map to one bank (word mod banks);
    threads touching the same word share one access.
    """
    words = np.unique(np.asarray(word_addresses, dtype=np.int64))
    if words.size == 0:
        return 0
    per_bank = np.bincount(words % banks, minlength=banks)
    return int(per_bank.max())


def tile_word(row: int, col: int, row_words: int) -> int:
    """Word index of element [row][col] of a shared tile with rows of ``row_words`` words."""
    return row * row_words + col


def smem_bytes(T: int, pad: int = 0, arrays: int = 2, elem_bytes: int = 4) -> int:
    """Shared memory of ``arrays`` T x (T + pad) FP32 tiles."""
    return arrays * T * (T + pad) * elem_bytes


def intensity(flops: float, elements_read: float, elem_bytes: int = 4) -> float:
    """FLOPs per byte read from global memory."""
    return flops / (elements_read * elem_bytes)

"""Pins of the counting simulator against every figure the pages print
(fixtures in tests/golden/pages_figures.json, each with its citation), plus
invariants the pages state in words."""

import json
import os

import numpy as np
import pytest

from oracle import tilesim

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def _model(e):
    if e["model"] == "naive":
        return tilesim.naive(e["M"], e["N"], e["K"])
    return tilesim.tiled(e["M"], e["N"], e["K"], e["T"])


@pytest.mark.parametrize("e", GOLDEN["read_counts"], ids=lambda e: e["id"])
def test_read_counts(e):
    c = _model(e)
    for key in ("global_reads", "threads", "tile_steps", "reads_per_thread"):
        if key in e:
            assert getattr(c, key) == e[key], (key, e["cite"])
    if "printed" in e:   # "2.15 B": the count to three significant digits
        assert f"{c.global_reads / 1e9:.2f} B" == e["printed"]


@pytest.mark.parametrize("e", GOLDEN["speedup"], ids=lambda e: e["id"])
def test_speedup(e):
    n, T = e["N"], e["T"]
    assert tilesim.naive(n, n, n).global_reads / tilesim.tiled(n, n, n, T).global_reads == e["ratio"]


def _bank_access(e):
    w = e["row_words"]
    if e["access"] == "column":      # thread i reads tile[i][c]
        return [tilesim.tile_word(i, 5, w) for i in range(32)]
    if e["access"] == "broadcast":   # every thread reads tileA[ty][k]
        return [tilesim.tile_word(3, 7, w)] * 32
    return [tilesim.tile_word(7, tx, w) for tx in range(32)]   # tileB[k][tx]


@pytest.mark.parametrize("e", GOLDEN["banks"], ids=lambda e: e["id"])
def test_bank_degrees(e):
    assert tilesim.bank_degree(_bank_access(e)) == e["degree"]


@pytest.mark.parametrize("e", GOLDEN["inner_step_ratios"], ids=lambda e: e["id"])
def test_inner_step_ratios(e):
    assert tilesim.inner_step_ratio(e["TM"], e["TN"]) == (e["shared_reads"], e["fma"])


@pytest.mark.parametrize("e", GOLDEN["smem_bytes"], ids=lambda e: e["id"])
def test_smem_bytes(e):
    assert tilesim.smem_bytes(e["T"], e["pad"]) == e["bytes"]


@pytest.mark.parametrize("e", GOLDEN["intensity"], ids=lambda e: e["id"])
def test_intensity(e):
    n = e["N"]
    c = _model(dict(e, M=n, K=n))
    assert tilesim.intensity(2 * c.fma, c.global_reads) == e["flop_per_byte"]


# ------------------------------------------------------------- stated invariants

@pytest.mark.parametrize("M,N,K,T", [(6, 6, 9, 3), (4, 4, 8, 2), (6, 6, 9, 2), (32, 48, 64, 16)])
def test_divisible_shapes_follow_the_closed_form(M, N, K, T):
    # every T-divisible M and N gives exactly 2MNK/T reads (the clean law)
    c = tilesim.tiled(M, N, K, T)
    assert c.global_reads * T == 2 * M * N * K


def test_masked_tails_issue_only_in_range_loads():
    M, N, K, T = 5, 7, 9, 4
    c = tilesim.tiled(M, N, K, T)
    # each A element is loaded once per block column, each B element once per block row
    assert c.global_reads == M * K * 2 + K * N * 2
    assert c.padded_slots == 2 * c.launched_threads * c.tile_steps - c.global_reads
    assert c.padded_slots > 0


def test_tile_of_one_is_naive():
    for (M, N, K) in [(5, 7, 3), (16, 16, 16)]:
        assert tilesim.tiled(M, N, K, 1).global_reads == tilesim.naive(M, N, K).global_reads


def test_naive_per_thread_derivation():
    # threads = M*N, reads per thread = 2K, total = 2MNK (the four-step derivation)
    c = tilesim.naive(3, 4, 5)
    assert (c.threads, c.reads_per_thread, c.global_reads, c.fma) == (12, 10, 120, 60)


def test_shared_reads_tiled():
    c = tilesim.tiled(4, 4, 8, 2)
    # each of 16 threads reads 2 values per k for 8 k
    assert c.shared_reads == 16 * 2 * 8


def test_padding_fixes_transposed_tile_store():
    # a warp storing 4 rows x 8 k of A into a k-major tile with rows of BM + pad words
    for pad, want in ((0, 8), (4, 1)):
        addr = [tilesim.tile_word(k, r, 128 + pad) for r in range(4) for k in range(8)]
        assert tilesim.bank_degree(addr) == want


def test_bank_degree_counts_distinct_words_only():
    assert tilesim.bank_degree([0, 0, 32, 32, 64]) == 3
    assert tilesim.bank_degree([]) == 0


# ------------------------------------------------- the 2-D model on ragged shapes
#
# "SGEMM: 2D Register Tiling Visualizer" (the listing; 'Why 2D Register Tiling
# Dominates'): per tile step a block loads the in-range part of a BM x BK slab
# of A and a BK x BN slab of B, and per inner step every launched thread reads
# TM values of A and TN of B from shared memory.  Over a grid of ceil(M/BM) x
# ceil(N/BN) blocks, each element of A is loaded once per block column and each
# element of B once per block row:  global reads = M K ceil(N/BN) + K N ceil(M/BM).

# (M, N, K, BM, BN, BK, TM, TN, global reads, shared reads), worked by hand:
#   (5, 7, 9) at 4/4/4/2/2: 2 x 2 blocks of 4 threads, 3 tile steps of 4 inner steps;
#     global 5*9*2 + 9*7*2 = 216; shared 16 threads * 12 inner steps * (2 + 2) = 768
#   (130, 67, 33) at 64/64/8/4/4: 3 x 2 blocks of 256 threads, 5 steps of 8;
#     global 130*33*2 + 33*67*3 = 8580 + 6633 = 15213; shared 1536 * 40 * 8 = 491520
#   (70, 45, 10) at 32/16/4/4/2: 3 x 3 blocks of 64 threads, 3 steps of 4;
#     global 70*10*3 + 10*45*3 = 2100 + 1350 = 3450; shared 576 * 12 * 6 = 41472
#   (8, 8, 8) at 4/4/4/2/2 (the visualizer's divisible block):
#     global 8*8*2 + 8*8*2 = 256 = 2MNK(1/BN + 1/BM)/2; shared 16 * 8 * 4 = 512 = MNK(1/TM + 1/TN)
REGISTER_CASES = [
    (5, 7, 9, 4, 4, 4, 2, 2, 216, 768),
    (130, 67, 33, 64, 64, 8, 4, 4, 15213, 491520),
    (70, 45, 10, 32, 16, 4, 4, 2, 3450, 41472),
    (8, 8, 8, 4, 4, 4, 2, 2, 256, 512),
]


def _cdiv(a, b):
    return -(-a // b)


def trace_register_tiled(A, B, BM, BN, BK, TM, TN):
    """Run the 2-D register-tiled kernel on real numbers, thread by thread as
    the listing does, counting every global load it issues (masked slots are
    zero-filled without a load) and every shared-memory read; returns
    (C, global loads, shared reads).  An independent route to the counts: it
    must also produce the product."""
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N), dtype=np.int64)
    g_loads = s_reads = 0
    for by in range(_cdiv(M, BM)):
        for bx in range(_cdiv(N, BN)):
            acc = np.zeros((BM, BN), dtype=np.int64)
            for step in range(_cdiv(K, BK)):
                As = np.zeros((BM, BK), dtype=np.int64)
                Bs = np.zeros((BK, BN), dtype=np.int64)
                for r in range(BM):
                    for c in range(BK):
                        gr, gc = by * BM + r, step * BK + c
                        if gr < M and gc < K:
                            As[r, c] = A[gr, gc]
                            g_loads += 1
                for r in range(BK):
                    for c in range(BN):
                        gr, gc = step * BK + r, bx * BN + c
                        if gr < K and gc < N:
                            Bs[r, c] = B[gr, gc]
                            g_loads += 1
                for ty in range(BM // TM):
                    for tx in range(BN // TN):
                        for dot in range(BK):
                            regM = [As[ty * TM + i, dot] for i in range(TM)]
                            regN = [Bs[dot, tx * TN + j] for j in range(TN)]
                            s_reads += TM + TN
                            for i in range(TM):
                                for j in range(TN):
                                    acc[ty * TM + i, tx * TN + j] += regM[i] * regN[j]
            rows, cols = min(BM, M - by * BM), min(BN, N - bx * BN)
            C[by * BM: by * BM + rows, bx * BN: bx * BN + cols] = acc[:rows, :cols]
    return C, g_loads, s_reads


def register_pin_failures(fn):
    """Which pins a 2-D counting model ``fn`` (tilesim.register_tiled's
    signature) fails: the hand-worked counts, the closed form for global reads,
    the launched-thread count for shared reads, and the multiply-add count."""
    bad = []
    for (M, N, K, BM, BN, BK, TM, TN, g, s) in REGISTER_CASES:
        c = fn(M, N, K, BM, BN, BK, TM, TN)
        tag = f"{M}x{N}x{K}@{BM}/{BN}/{BK}/{TM}/{TN}"
        if c.global_reads != g:
            bad.append(f"{tag}: global {c.global_reads} != {g}")
        if c.global_reads != M * K * _cdiv(N, BN) + K * N * _cdiv(M, BM):
            bad.append(f"{tag}: global reads off the closed form")
        if c.shared_reads != s:
            bad.append(f"{tag}: shared {c.shared_reads} != {s}")
        if c.fma != M * N * K or c.threads != M * N:
            bad.append(f"{tag}: multiply-adds or threads")
    return bad


def tiled_pin_failures(fn):
    """The same for a square-tile model ``fn`` (tilesim.tiled's signature)."""
    bad = []
    for (M, N, K, T) in [(5, 7, 9, 4), (6, 6, 9, 2), (33, 17, 40, 16), (4, 4, 8, 2)]:
        c = fn(M, N, K, T)
        if c.global_reads != M * K * _cdiv(N, T) + K * N * _cdiv(M, T):
            bad.append(f"{M}x{N}x{K}@{T}: global reads off the closed form")
        launched = _cdiv(M, T) * T * _cdiv(N, T) * T
        if c.shared_reads != 2 * launched * _cdiv(K, T) * T:
            bad.append(f"{M}x{N}x{K}@{T}: shared reads")
    if fn(4, 4, 8, 2).global_reads != 128:   # the pages' toy example
        bad.append("toy example")
    return bad


@pytest.mark.parametrize("case", REGISTER_CASES, ids=lambda c: "x".join(map(str, c[:3])))
def test_register_tiled_ragged_counts(case):
    M, N, K, BM, BN, BK, TM, TN, g, s = case
    c = tilesim.register_tiled(M, N, K, BM, BN, BK, TM, TN)
    assert (c.global_reads, c.shared_reads) == (g, s)
    assert c.global_reads == M * K * _cdiv(N, BN) + K * N * _cdiv(M, BM)
    assert c.launched_threads == _cdiv(M, BM) * _cdiv(N, BN) * (BM // TM) * (BN // TN)
    assert c.tile_steps == _cdiv(K, BK)


@pytest.mark.parametrize("case", REGISTER_CASES,
                         ids=lambda c: "x".join(map(str, c[:3])))
def test_register_tiled_counts_match_a_traced_run(case):
    # execute the kernel on small integers: it must produce A B exactly, and the
    # loads it issued must be the counts the model gives
    M, N, K, BM, BN, BK, TM, TN, _, _ = case
    rng = np.random.default_rng(M * 1000 + N)
    A = rng.integers(-4, 5, (M, K))
    B = rng.integers(-4, 5, (K, N))
    C, g, s = trace_register_tiled(A, B, BM, BN, BK, TM, TN)
    assert np.array_equal(C, A @ B)
    c = tilesim.register_tiled(M, N, K, BM, BN, BK, TM, TN)
    assert (c.global_reads, c.shared_reads) == (g, s)


def test_register_tiled_divisible_closed_forms():
    # divisible shapes: global reads 2MNK(1/BM + 1/BN)/2, shared MNK(1/TM + 1/TN)
    M, N, K, BM, BN, BK, TM, TN = 128, 64, 32, 32, 16, 8, 4, 2
    c = tilesim.register_tiled(M, N, K, BM, BN, BK, TM, TN)
    assert c.global_reads * BM * BN == M * N * K * (BM + BN)
    assert c.shared_reads * TM * TN == M * N * K * (TM + TN)
    assert tilesim.register_reads(c) == 2 * c.fma


def test_the_real_simulator_passes_every_pin():
    assert register_pin_failures(tilesim.register_tiled) == []
    assert tiled_pin_failures(tilesim.tiled) == []


# ---------------------------------------------- planted mistakes (on the CPU)
#
# Each copy below carries one plausible slip in the simulator's edge handling;
# the pins above must catch every one of them.

def _register_variant(slip):
    def fn(M, N, K, BM, BN, BK, TM, TN):
        gm, gn, steps = _cdiv(M, BM), _cdiv(N, BN), _cdiv(K, BK)
        threads_per_block = (BM // TM) * (BN // TN)
        g = 0
        for by in range(gm):
            rows_in = BM if slip == "full_rows" else min(BM, M - by * BM)
            for bx in range(gn):
                cols_in = BN if slip == "full_cols" else min(BN, N - bx * BN)
                for step in range(steps):
                    k_in = BK if slip == "full_k" else min(BK, K - step * BK)
                    if slip == "a_only":
                        g += rows_in * k_in
                    else:
                        g += rows_in * k_in + k_in * cols_in
        blocks = gm * gn
        if slip == "in_range_threads":
            shared = (M * N // (TM * TN)) * steps * BK * (TM + TN)
        elif slip == "k_not_padded":
            shared = blocks * threads_per_block * K * (TM + TN)
        else:
            shared = blocks * threads_per_block * steps * BK * (TM + TN)
        return tilesim.Counts(threads=M * N, launched_threads=blocks * threads_per_block, global_reads=g,
                              shared_reads=shared, fma=M * N * K, tile_steps=steps)
    return fn


def _tiled_counting_zero_fill(M, N, K, T):
    # counts every tile slot, zero-filled or not, as a global read
    c = tilesim.tiled(M, N, K, T)
    return tilesim.Counts(threads=c.threads, launched_threads=c.launched_threads,
                          global_reads=c.global_reads + c.padded_slots, shared_reads=c.shared_reads,
                          fma=c.fma, tile_steps=c.tile_steps, padded_slots=0)


def _tiled_floor_steps(M, N, K, T):
    # the visualizer's integer division taken literally: K // T tile steps
    gm, gn = _cdiv(M, T), _cdiv(N, T)
    steps = K // T
    launched = gm * T * gn * T
    g = 0
    for step in range(steps):
        k_in = min(T, K - step * T)
        g += M * k_in * gn + k_in * N * gm
    return tilesim.Counts(threads=M * N, launched_threads=launched, global_reads=g,
                          shared_reads=launched * steps * 2 * T, fma=M * N * K, tile_steps=steps)


@pytest.mark.parametrize("slip", ["full_rows", "full_cols", "full_k", "a_only", "in_range_threads",
                                  "k_not_padded"])
def test_planted_register_tiled_slip_is_caught(slip):
    assert register_pin_failures(_register_variant(slip)), f"no pin catches the slip {slip!r}"


def test_planted_register_tiled_variant_is_faithful_without_a_slip():
    # the harness that plants the slips is itself the model when no slip is planted
    assert register_pin_failures(_register_variant(None)) == []


@pytest.mark.parametrize("variant", [_tiled_counting_zero_fill, _tiled_floor_steps], ids=lambda f: f.__name__)
def test_planted_tiled_slip_is_caught(variant):
    assert tiled_pin_failures(variant), f"no pin catches {variant.__name__}"

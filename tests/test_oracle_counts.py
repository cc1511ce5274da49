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


def test_register_tiled_model():
    # the 2D visualizer's block: BM=BN=BK=4, TM=TN=2 on 8 x 8 matrices, 4 threads per block
    c = tilesim.register_tiled(8, 8, 8, 4, 4, 4, 2, 2)
    assert c.launched_threads == 4 * 4
    assert c.fma == 8 * 8 * 8
    assert c.shared_reads == 16 * 2 * 4 * (2 + 2)
    assert c.global_reads == 8 * 8 * 2 + 8 * 8 * 2
    # shared reads : multiply-adds = (TM+TN) : TM*TN
    assert c.shared_reads * 2 * 2 == c.fma * (2 + 2)
    assert tilesim.register_reads(c) == 2 * c.fma


def test_padding_fixes_transposed_tile_store():
    # a warp storing 4 rows x 8 k of A into a k-major tile with rows of BM + pad words
    for pad, want in ((0, 8), (4, 1)):
        addr = [tilesim.tile_word(k, r, 128 + pad) for r in range(4) for k in range(8)]
        assert tilesim.bank_degree(addr) == want


def test_bank_degree_counts_distinct_words_only():
    assert tilesim.bank_degree([0, 0, 32, 32, 64]) == 3
    assert tilesim.bank_degree([]) == 0


def test_planted_mistake_in_simulator_is_caught():
    # a simulator that forgets the mask (counts zero-filled slots) misses the pin
    c = tilesim.tiled(5, 7, 9, 4)
    assert c.global_reads + c.padded_slots != c.global_reads
    # counting per launched thread instead of in-range threads breaks the naive pin
    assert tilesim.naive(1024, 1024, 1024).threads == 1048576

"""The phased TMA kernel: operands whose rows are only 4-byte aligned (leading
dimensions that are not multiples of 4 floats, bases off 16-byte boundaries)
are read through four tensor maps each -- rows s, s + 4, ... of one residue s
-- in boxes 4 floats wider than the tile, and every row is shifted left by its
phase's offset in shared memory before the FMAs.  Checked against the FP64
oracle within 2 K u sum|a||b| (exactly on small integers) for every offset
pattern of both operands, on the 128 x 128 tile (plain grids and cluster
splits) and the 128 x 64 narrow tile, with ragged edges, split-K and the
bounded waits; the canaries in the row gaps and in front of the operands must
never reach C."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, _device_buffer, check_entries, check_full, check_rows, run_sgemm

pytestmark = pytest.mark.gpu

FORCE_PHASED = 2048
ALL_TILES = 256
NO_NARROW = 1024     # keep products with few tiles on the 128 x 128 tile
NO_SPLIT = 1 << 4


def forced(cs):
    return (cs << 4) | ALL_TILES


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    sg.sgemm_test_switches(0, 2_000_000_000)
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


# every residue of the base offset and of the leading dimension (mod 4 floats)
# of each operand: the four phases then take every pattern of shifts
@pytest.mark.parametrize("a_off,lda_pad", [(0, 1), (1, 0), (2, 3), (3, 2), (1, 1), (3, 3)])
@pytest.mark.parametrize("b_off,ldb_pad", [(0, 0), (0, 1), (2, 2), (3, 1)])
def test_every_shift_pattern(sg, a_off, lda_pad, b_off, ldb_pad):
    M, N, K = 261, 259, 101          # two and a bit tiles each way, a partial last k-step
    sg.sgemm_test_switches(NO_NARROW)
    A, B = gen.operands(M, N, K, seed=400 + 7 * a_off + lda_pad)
    C = run_sgemm(sg, A, B, lda=K + lda_pad, ldb=N + ldb_pad, a_off=a_off, b_off=b_off)
    check_full(C, A, B)
    Ai, Bi = gen.operands(M, N, K, seed=401, integer_copy=True)
    C = run_sgemm(sg, Ai, Bi, lda=K + lda_pad, ldb=N + ldb_pad, a_off=a_off, b_off=b_off, c_off=1)
    check_full(C, Ai, Bi, exact=True)


@pytest.mark.parametrize("M,N,K", [(4, 4, 4), (5, 7, 4), (4, 300, 37), (300, 4, 5), (127, 129, 31), (128, 128, 32),
                                   (129, 1, 1000), (7, 513, 65)])
def test_small_and_edge_shapes(sg, M, N, K):
    sg.sgemm_test_switches(NO_NARROW)
    A, B = gen.operands(M, N, K, seed=410)
    check_full(run_sgemm(sg, A, B, lda=K + 1, ldb=N + 3, a_off=2, b_off=1), A, B)


@pytest.mark.parametrize("M,N,K", [(3, 100, 50), (100, 100, 3), (2, 2, 2)])
def test_fewer_than_four_rows_take_the_cp_async_kernel(sg, M, N, K):
    A, B = gen.operands(M, N, K, seed=411)
    check_full(run_sgemm(sg, A, B, lda=K + 1, ldb=N + 1, a_off=1), A, B)


def test_aligned_operands_through_the_phase_maps(sg):
    # a test-only switch routes 16-byte aligned operands here too (every shift 0)
    A, B = gen.operands(300, 520, 200, seed=412)
    sg.sgemm_test_switches(FORCE_PHASED | NO_NARROW)
    check_full(run_sgemm(sg, A, B), A, B)
    Ai, Bi = gen.operands(300, 520, 200, seed=412, integer_copy=True)
    check_full(run_sgemm(sg, Ai, Bi), Ai, Bi, exact=True)


@pytest.mark.parametrize("cs", [2, 4, 8])
def test_cluster_split(sg, cs):
    M, N, K = 300, 260, 777
    A, B = gen.operands(M, N, K, seed=420 + cs)
    sg.sgemm_test_switches(forced(cs))
    assert sg.sgemm_f32_plan(M, N, K, aligned=False)[2] == cs
    C1 = run_sgemm(sg, A, B, lda=K + 3, ldb=N + 1, a_off=1, b_off=3)
    check_full(C1, A, B)
    # the exchange adds in rank order: the same bits every run
    C2 = run_sgemm(sg, A, B, lda=K + 3, ldb=N + 1, a_off=1, b_off=3)
    assert np.array_equal(C1, C2)


def test_plain_waves_then_cluster_split(sg):
    """A plain grid of whole waves, then the last tiles split over clusters that
    start as the plain grid drains (the automatic plan on this shape)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles_n = 8
    tiles_m = sms // tiles_n + 1
    M, N, K = 128 * tiles_m - 5, 128 * tiles_n - 3, 1021
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K, aligned=False)
    assert cs > 1 and 0 < full < tiles and tn == 128
    A, B = gen.operands(M, N, K, seed=430)
    C = run_sgemm(sg, A, B, lda=K, ldb=N + 2, a_off=3)
    check_rows(C, A, B, [0, 1, 127, 128, M // 2, M - 129, M - 2, M - 1])
    cols = np.arange(N - 130, N)
    rows = np.arange(0, M, 11)
    check_entries(C, A, B, np.repeat(rows, cols.size), np.tile(cols, rows.size))


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_split_k(sg, splits):
    M, N, K = 200, 333, 900
    A, B = gen.operands(M, N, K, seed=440 + splits)
    check_full(run_sgemm(sg, A, B, lda=K + 1, ldb=N + 2, b_off=1, splits=splits), A, B)


@pytest.mark.parametrize("flags", [NO_SPLIT, 4 << 4 | ALL_TILES, 0], ids=["plain", "clusters", "narrow"])
def test_timeout_is_reported_and_nothing_is_written(sg, flags):
    """Copies never issued (a test-only switch): every block gives up after the
    wait limit, writes nothing, and the status reports it; the next product on
    the same buffers is correct."""
    import torch
    M, N, K = 256, 256, 512
    A, B = gen.operands(M, N, K, seed=450)
    dev = torch.device("cuda", 0)
    a_buf, pa = _device_buffer(A, K + 1, 1, torch, dev)
    b_buf, pb = _device_buffer(B, N + 3, 0, torch, dev)
    dC = torch.from_numpy(np.full((M, N), CANARY_BITS, np.int32).view(np.float32)).cuda()
    sg.sgemm_test_switches(flags | 1, 50_000_000)
    assert sg.sgemm_f32_plan(M, N, K, aligned=False)[3] == (64 if flags == 0 else 128)
    sg.sgemm_f32(M, N, K, pa, K + 1, pb, N + 3, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    sg.sgemm_test_switches(flags, 2_000_000_000)
    sg.sgemm_f32(M, N, K, pa, K + 1, pb, N + 3, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)


# ------------------------------------------------------------------ the narrow tile

def narrow_plan(sg, M, N, K):
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K, aligned=False)
    assert tn == 64 and full == 0 and cs in (2, 4, 8), (M, N, K, tiles, full, cs, tn)
    return cs


@pytest.mark.parametrize("M,N,K,lda_pad,ldb_pad,a_off", [(512, 512, 512, 1, 1, 0), (257, 130, 1000, 1, 3, 2),
                                                         (1000, 200, 777, 3, 1, 1), (129, 65, 2000, 2, 2, 3),
                                                         (300, 190, 999, 0, 2, 1), (1024, 1024, 1024, 1, 1, 0)])
def test_narrow_tile(sg, M, N, K, lda_pad, ldb_pad, a_off):
    narrow_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=460 + M % 31)
    check_full(run_sgemm(sg, A, B, lda=K + lda_pad, ldb=N + ldb_pad, a_off=a_off, c_off=1), A, B)


def test_narrow_tile_integers_exact_and_repeatable(sg):
    M, N, K = 384, 320, 1537
    narrow_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=470, integer_copy=True)
    c1 = run_sgemm(sg, A, B, lda=K + 2, ldb=N + 1, b_off=3)
    c2 = run_sgemm(sg, A, B, lda=K + 2, ldb=N + 1, b_off=3)
    check_full(c1, A, B, exact=True)
    assert np.array_equal(c1, c2)


def test_rows_more_than_2_gib_apart(sg):
    # lda = 2^29 + 1 floats: the phase maps' row pitch (16 lda bytes, 8 GiB) and
    # the offsets of A's rows exceed 32 bits; the product is still exact
    import torch
    from oracle import ref_gemm
    M, N, K = 4, 40, 9              # one row per phase of A: 6.4 GB of buffer
    lda, ldb = (1 << 29) + 1, N + 1
    A, B = gen.operands(M, N, K, seed=480, integer_copy=True)
    dA = torch.zeros((M - 1) * lda + K, device="cuda")
    dB = torch.zeros((K - 1) * ldb + N, device="cuda")
    for r in range(M):
        dA[r * lda: r * lda + K] = torch.from_numpy(A[r]).cuda()
    for r in range(K):
        dB[r * ldb: r * ldb + N] = torch.from_numpy(B[r]).cuda()
    assert sg.sgemm_f32_plan(M, N, K, aligned=False)[3] == 128
    C = torch.full((M, N), float("nan"), device="cuda")
    sg.sgemm_f32(M, N, K, dA, lda, dB, ldb, C, N)
    torch.cuda.synchronize()
    C64, _ = ref_gemm.gemm_f64(A, B)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), C64)
    del dA, dB

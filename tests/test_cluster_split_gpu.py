"""The TMA path's cluster split: tiles that would leave SMs idle (the tiles
beyond whole multiples of the SM count, or every tile of a small grid) are
each shared by a thread-block cluster of 2 to 8 blocks that take equal runs of
k-steps and add their partial sums through distributed shared memory in rank
order.  Checked against the FP64 oracle within 2 K u sum|a||b|, exactly on
small integers, bit for bit from run to run, with alpha/beta, with ragged
edges, with ranks that get no k-steps, with cluster sizes that do not divide
the per-thread rows evenly, with and without programmatic overlap; and the
bounded-wait path in cluster mode (no fault, no hang)."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, check_full, check_rows, run_sgemm

pytestmark = pytest.mark.gpu

NO_SPLIT = 1 << 4
ALL_TILES = 256
NO_OVERLAP = 512
NO_NARROW = 1024
OVERHEAD = 2.0       # k-steps a block spends outside its k-loop
# narrow-tile cost models, per path: (k-steps an SM advances per unit with
# three or more blocks resident, the fraction of that with two, units per
# round of blocks, blocks per SM)
NARROW_MODEL = {"tma": (4.4, 0.9, 1.25, 4), "cp": (5.9, 0.75, 1.5, 3)}


def forced(cs, all_tiles=True):
    return (cs << 4) | (ALL_TILES if all_tiles else 0)


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


def sm_time(L, w):
    return (L // 2) * (w + OVERHEAD) + (L % 2) * (0.5 * w + OVERHEAD)


def narrow_sm_time(model, L, w):
    steps, two, rnd, per_sm = model
    if L <= 1:
        return w / (0.5 * steps) + rnd
    if L == 2:
        return 2 * w / (two * steps) + rnd
    return L * w / steps + rnd * -(-L // per_sm)


def expected_plan(M, N, K, sms, narrow="tma", ksplit=False):
    """The automatic plan restated, as (tiles, full, cluster size, tile width):
    the 128 x 128 tiles beyond whole multiples of the SM count P (all of them
    when there are fewer than P) are split over the cluster size c = 2, 4 or 8
    that minimises the cost model (an SM runs blocks two at a time, each
    advancing a k-step per unit, or one alone at two per unit; each block
    spends OVERHEAD units outside its k-loop, hidden when it has a partner),
    ties to the larger c, keeping four 32-deep k-steps per block, if that beats
    the plain grid by 4 %.  With fewer tiles than P, 128 x 64 narrow tiles of
    the path (`narrow`: "tma", "cp" or None) in clusters of c = 2, 4 or 8 (the
    lowest estimate of that path's NARROW_MODEL, ties to the larger c) replace
    that when lower still; on the TMA path (`ksplit`), narrow tiles that fill
    at least 70 % of one round over the SMs with at most 48 k-steps take the
    k-split tile instead, one CTA per tile (cluster size 1, every tile full)."""
    P = sms
    tiles = -(-M // 128) * -(-N // 128)
    rem = tiles % P
    full = tiles - rem
    kt = -(-K // 32)
    cs = 1
    if rem:
        plain = sm_time(-(-tiles // P), kt)
        best = plain
        for c in (2, 4, 8):
            if kt < 4 * c:
                break
            t = sm_time(full // P, kt) + sm_time(-(-rem * c // P), -(-kt // c))
            if t <= best:
                best, cs = t, c
        if cs > 1 and best > 0.96 * plain:
            cs, best = 1, plain
        if narrow and tiles < P:
            ntiles = -(-M // 128) * -(-N // 64)
            if ksplit and ntiles <= P and 100 * ntiles >= 70 * P and kt <= 48:
                return (ntiles, ntiles, 1, 64)
            ncs, nbest = 0, 0.0
            for c in (2, 4, 8):
                if kt < 4 * c:
                    break
                t = narrow_sm_time(NARROW_MODEL[narrow], -(-ntiles * c // P), -(-kt // c))
                if ncs == 0 or t <= nbest:
                    ncs, nbest = c, t
            if ncs and nbest < best:
                return (ntiles, 0, ncs, 64)
    return (tiles, full if cs > 1 else tiles, cs, 128)


@pytest.mark.parametrize("cs", [2, 3, 4, 6, 8])
@pytest.mark.parametrize("M,N,K,seed", [(300, 200, 1000, 200), (129, 383, 517, 201), (640, 768, 4096, 202),
                                        (128, 128, 288, 203)])
def test_forced_split_matches_oracle(sg, cs, M, N, K, seed):
    A, B = gen.operands(M, N, K, seed=seed)
    sg.sgemm_test_switches(forced(cs))
    tiles, full, c, tn = sg.sgemm_f32_plan(M, N, K)
    assert (full, c, tn) == (0, cs, 128)
    check_full(run_sgemm(sg, A, B), A, B)
    assert sg.sgemm_device_status() == sg.SGEMM_OK


@pytest.mark.parametrize("cs", [2, 3, 5, 8])
def test_forced_split_integers_exact(sg, cs):
    A, B = gen.operands(256, 384, 1536, seed=204, integer_copy=True)
    sg.sgemm_test_switches(forced(cs))
    check_full(run_sgemm(sg, A, B), A, B, exact=True)


def test_ranks_without_k_steps(sg):
    # K = 100: 4 k-steps over 8 ranks, so ranks 4..7 contribute zeros
    A, B = gen.operands(200, 300, 100, seed=205)
    sg.sgemm_test_switches(forced(8))
    check_full(run_sgemm(sg, A, B), A, B)


@pytest.mark.parametrize("cs", [2, 8])
def test_bitwise_repeatable(sg, cs):
    import torch
    A, B = gen.operands(512, 640, 2048, seed=206)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    sg.sgemm_test_switches(forced(cs))
    c1 = sg.matmul(dA, dB)
    c2 = sg.matmul(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("overlap", [True, False])
def test_tail_split_after_full_waves(sg, overlap):
    # more tiles than one wave: a plain launch for the full waves, clusters for
    # the rest, with and without programmatic overlap of the two launches
    import torch
    sg.sgemm_test_switches(0 if overlap else NO_OVERLAP)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles_n = 8
    tiles_m = sms // tiles_n + 1              # one tile per SM, then a short tail
    M, N, K = 128 * tiles_m - 37, 128 * tiles_n - 4, 1000   # N % 4 == 0: the TMA path
    A, B = gen.operands(M, N, K, seed=207)
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K)
    assert (tiles, full, cs, tn) == expected_plan(M, N, K, sms, ksplit=True)
    assert cs > 1 and 0 < full < tiles and tn == 128
    C = run_sgemm(sg, A, B)
    rows = [0, 1, 127, 128, M - 129, M - 128, M - 2, M - 1] + list(np.random.default_rng(1).integers(0, M, 12))
    check_rows(C, A, B, rows)


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (8192, 8192, 8192), (3008, 5008, 2048), (256, 256, 96),
                                   (2048, 2048, 2048), (4096, 4096, 4096), (6144, 6144, 6144), (512, 512, 8192),
                                   (1536, 1536, 1536), (4955, 1020, 1024), (16384, 16384, 1024)])
def test_automatic_plan(sg, M, N, K):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sg.sgemm_f32_plan(M, N, K) == expected_plan(M, N, K, sms, ksplit=True)
    # operands the TMA cannot address directly: the phased TMA kernel, whose
    # narrow tile runs like the TMA kernel's (four CTAs per SM) and takes its model
    assert sg.sgemm_f32_plan(M, N, K, aligned=False) == expected_plan(M, N, K, sms, narrow="tma")
    # with every product on the cp.async-fed kernel: its narrow tile and model
    sg.sgemm_test_switches(2)
    assert sg.sgemm_f32_plan(M, N, K, aligned=False) == expected_plan(M, N, K, sms, narrow="cp")
    sg.sgemm_test_switches(NO_NARROW)
    assert sg.sgemm_f32_plan(M, N, K) == expected_plan(M, N, K, sms, narrow=None)
    assert sg.sgemm_f32_plan(M, N, K, aligned=False) == expected_plan(M, N, K, sms, narrow=None)


def test_square_768_uses_clusters_and_matches(sg):
    # (1024^3 takes the k-split tile, tested in test_ksplit_gpu.py)
    A, B = gen.operands(768, 768, 768, seed=1)
    assert sg.sgemm_f32_plan(768, 768, 768)[2] > 1
    check_full(run_sgemm(sg, A, B), A, B)


def test_no_split_switch(sg):
    sg.sgemm_test_switches(NO_SPLIT)
    tiles, full, cs, tn = sg.sgemm_f32_plan(1024, 1024, 1024)
    assert cs == 1 and full == tiles == 64 and tn == 128


@pytest.mark.parametrize("cs", [2, 4])
def test_alpha_beta_with_split(sg, cs):
    from oracle import ref_gemm, tolerance
    from test_gemm_general_gpu import run_gemm
    A = gen.matrix(208, gen.STREAM_A, 200, 700)
    B = gen.matrix(208, gen.STREAM_B, 700, 260)
    C0 = gen.matrix(209, gen.STREAM_A, 200, 260)
    sg.sgemm_test_switches(forced(cs))
    C = run_gemm(sg, 0, 0, 0, -0.75, A, B, 1.5, C0)
    C64, S, T = ref_gemm.gemm_general_f64(False, False, -0.75, A, B, 1.5, C0)
    assert tolerance.max_error_ratio_general(C, C64, S, T, 700, -0.75) <= 1.0


def test_timeout_in_cluster_mode(sg):
    """Copies never issued: every block of every cluster gives up after the wait
    limit, all blocks still meet at both cluster barriers, nothing is written,
    and the device stays usable."""
    import torch
    M, N, K = 256, 256, 512
    A, B = gen.operands(M, N, K, seed=210)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(np.full((M, N), CANARY_BITS, np.int32).view(np.float32)).cuda()
    sg.sgemm_test_switches(forced(4) | 1, 50_000_000)
    assert sg.sgemm_f32_plan(M, N, K)[2:] == (4, 128)
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    sg.sgemm_test_switches(forced(4))
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)


def test_timeout_with_plain_waves_and_tail(sg):
    """Both launches time out (copies never issued): the tail clusters wait for
    the plain grid before exiting; nothing is written and the device recovers."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles_n = 8
    tiles_m = sms // tiles_n + 1
    M, N, K = 128 * tiles_m, 128 * tiles_n, 1024
    sg.sgemm_test_switches(1, 50_000_000)
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K)
    assert cs > 1 and 0 < full < tiles and tn == 128
    dA = torch.zeros(M, K, device="cuda")
    dB = torch.zeros(K, N, device="cuda")
    dC = torch.from_numpy(np.full((M, N), CANARY_BITS, np.int32).view(np.float32)).cuda()
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    sg.sgemm_test_switches(0)
    A, B = gen.operands(M, N, K, seed=211)
    dA.copy_(torch.from_numpy(A))
    dB.copy_(torch.from_numpy(B))
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_rows(dC.cpu().numpy(), A, B, [0, 5, M - 200, M - 1])

"""The small-K tiles (K <= 64 on aligned operands: 128 x 64 tiles, one stage;
for K <= 32 with beta == 0 and a C the TMA can address, the tile whose C is
written by a TMA store) on large grids: against the FP64 oracle with ragged
edges and every K from 1 to 64 class, exactly on small integers, bit for bit
against the main tile fed by cp.async (the same per-element arithmetic), with
alpha/beta, and on the bounded-wait path with thousands of CTAs."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, check_full, check_rows, run_sgemm

pytestmark = pytest.mark.gpu

FORCE_CP_ASYNC = 2


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


def ld4(n):
    return (n + 3) // 4 * 4


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 32), (3001, 2500, 64), (1000, 777 * 4, 1), (4099, 1030, 33),
                                   (128, 64, 48), (130, 70, 17), (1000, 1030, 32), (257, 100, 32), (5, 36, 3)])
def test_matches_oracle(sg, M, N, K):
    # leading dimensions padded to 4 floats keep every case on the TMA path
    A, B = gen.operands(M, N, K, seed=300 + K)
    C = run_sgemm(sg, A, B, lda=ld4(K), ldb=ld4(N), ldc=ld4(N))
    if M * N <= 1_000_000:
        check_full(C, A, B)
    else:
        rows = [0, 1, 127, 128, M // 2, M - 2, M - 1] + list(np.random.default_rng(K).integers(0, M, 12))
        check_rows(C, A, B, rows)


def test_integers_exact(sg):
    A, B = gen.operands(1536, 2048, 64, seed=310, integer_copy=True)
    C = run_sgemm(sg, A, B)
    rows = [0, 5, 700, 1535]
    from oracle import ref_gemm
    C64, _ = ref_gemm.gemm_f64(np.ascontiguousarray(A[rows]), B)
    assert np.array_equal(C[rows].astype(np.float64), C64)


@pytest.mark.parametrize("K", [32, 64, 5])
def test_bitwise_equal_to_the_main_tile(sg, K):
    import torch
    A, B = gen.operands(2000, 3000, K, seed=311)
    dA = torch.zeros(2000, ld4(K), device="cuda")[:, :K]     # row pitch a multiple of 4 floats
    dA.copy_(torch.from_numpy(A))
    dB = torch.from_numpy(B).cuda()
    c1 = sg.matmul(dA, dB)
    sg.sgemm_test_switches(FORCE_CP_ASYNC)
    c2 = sg.matmul(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("K", [40, 32, 20])   # two k-steps; one k-step (the tile unrolled by four); one, ragged
def test_alpha_beta(sg, K):
    from oracle import ref_gemm, tolerance
    from test_gemm_general_gpu import run_gemm
    A = gen.matrix(312, gen.STREAM_A, 700, K)
    B = gen.matrix(312, gen.STREAM_B, K, 900)
    C0 = gen.matrix(313, gen.STREAM_A, 700, 900)
    C = run_gemm(sg, 0, 0, 0, 1.75, A, B, -0.5, C0)
    C64, S, T = ref_gemm.gemm_general_f64(False, False, 1.75, A, B, -0.5, C0)
    assert tolerance.max_error_ratio_general(C, C64, S, T, K, 1.75) <= 1.0


@pytest.mark.parametrize("K", [64, 32])   # the small-K tile, and its one-k-step form unrolled by four
def test_timeout_with_many_ctas(sg, K):
    import torch
    M, N = 2048, 4096
    A, B = gen.operands(M, N, K, seed=314)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(np.full((M, N), CANARY_BITS, np.int32).view(np.float32)).cuda()
    sg.sgemm_test_switches(1, 50_000_000)
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    sg.sgemm_test_switches(0)
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_rows(dC.cpu().numpy(), A, B, [0, 1000, M - 1])


@pytest.mark.parametrize("K", [32, 9])
def test_tma_store_tile_alpha_bitwise(sg, K):
    # beta == 0 with a 16-byte aligned C and N a multiple of 4 takes the
    # TMA-store tile; ldc = N + 1 takes the per-thread stores of the small-K tile: the same accumulators and
    # alpha * acc rounded once, so the same bits, zero signs included (rows of
    # zeros in A make products of exactly zero, times a negative alpha)
    import torch
    M, N = 1000, 1028
    A = gen.matrix(315, gen.STREAM_A, M, K)
    A[::7] = 0.0
    B = gen.matrix(315, gen.STREAM_B, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    out = {}
    for ldc in (N + 4, N + 1):   # N + 4: rows 16-byte aligned (1032); N + 1: not
        dC = torch.full((M, ldc), float("nan"), device="cuda")
        sg.sgemm_gemm(0, 0, 0, M, N, K, -1.5, dA, K, dB, N, 0.0, dC, ldc)
        assert sg.sgemm_device_status() == sg.SGEMM_OK
        c = dC.cpu().numpy()
        assert np.isnan(c[:, N:]).all(), "wrote past column N"
        out[ldc] = c[:, :N].copy()
    assert np.array_equal(out[N + 4].view(np.int32), out[N + 1].view(np.int32))
    assert np.signbit(out[N + 4][::7]).all()   # -1.5 * (+0) is -0
    from oracle import ref_gemm, tolerance
    C64, S, T = ref_gemm.gemm_general_f64(False, False, -1.5, A, B, 0.0, np.zeros((M, N), np.float32))
    assert tolerance.max_error_ratio_general(out[N + 4], C64, S, T, K, -1.5) <= 1.0

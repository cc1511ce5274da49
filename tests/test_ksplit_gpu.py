"""The k-split tile (ffma_tma_ksplit.cuh): one round of 128 x 64 tiles, one
CTA per tile of two warp groups, each taking one half of every 32-deep k-step,
their sums added in shared memory.  sgemm_f32 takes it for TMA-addressable products whose narrow
tiles fill 70-100 % of the SMs with at most 48 k-steps.  Against the FP64
oracle on every element with ragged edges, odd and partial k-step counts and
as few k-steps as stages; exactly on small integers; bit for bit from run to
run; with alpha/beta and with a C the 16-byte stores cannot take; and on the
bounded-wait path (no fault, no hang)."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, check_full, run_sgemm

pytestmark = pytest.mark.gpu


@pytest.fixture
def sg(cuda_device, lib):
    import torch

    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the shapes below are chosen for 152 SMs")
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


def ld4(n):
    return (n + 3) // 4 * 4


def ksplit_plan(sg, M, N, K):
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K)
    assert (full, cs, tn) == (tiles, 1, 64), (M, N, K, tiles, full, cs, tn)
    assert tiles == -(-M // 128) * -(-N // 64)


@pytest.mark.parametrize("M,N,K", [
    (1024, 1024, 1024),   # 128 tiles, 32 k-steps
    (1000, 1000, 1000),   # ragged rows, columns and last k-step
    (1024, 1216, 1024),   # exactly one tile per SM
    (960, 960, 960),      # 30 k-steps
    (1024, 1024, 992),    # 31 k-steps
    (1100, 900, 97),      # 4 k-steps, the last with one k-value (the second group's half of it all zeros)
    (1024, 1024, 65),     # 3 k-steps, as many as the stages (K <= 64 takes the small-K tiles)
    (1024, 1024, 1536),   # 48 k-steps, the most the plan gives it
])
def test_matches_oracle(sg, M, N, K):
    ksplit_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=700 + M % 97)
    C = run_sgemm(sg, A, B, lda=ld4(K), ldb=ld4(N), ldc=ld4(N))
    check_full(C, A, B)


def test_integers_exact(sg):
    M, N, K = 1024, 1000, 1500
    ksplit_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=710, integer_copy=True)
    check_full(run_sgemm(sg, A, B, lda=ld4(K)), A, B, exact=True)


def test_bitwise_repeatable(sg):
    import torch
    ksplit_plan(sg, 1024, 1024, 1024)
    A, B = gen.operands(1024, 1024, 1024, seed=711)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c1 = sg.matmul(dA, dB)
    c2 = sg.matmul(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_unaligned_c(sg):
    # a C whose rows are not 16-byte aligned: the epilogue's 4-byte stores,
    # with the canaries around C untouched (run_sgemm checks them)
    M, N, K = 1000, 1000, 1000
    ksplit_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=712)
    check_full(run_sgemm(sg, A, B, lda=ld4(K), ldb=ld4(N), ldc=N + 1, c_off=1), A, B)


def test_alpha_beta(sg):
    from oracle import ref_gemm, tolerance
    from test_gemm_general_gpu import run_gemm
    M, N, K = 1024, 1024, 1024
    ksplit_plan(sg, M, N, K)
    A = gen.matrix(713, gen.STREAM_A, M, K)
    B = gen.matrix(713, gen.STREAM_B, K, N)
    C0 = gen.matrix(714, gen.STREAM_A, M, N)
    C = run_gemm(sg, 0, 0, 0, -0.75, A, B, 1.5, C0)
    C64, S, T = ref_gemm.gemm_general_f64(False, False, -0.75, A, B, 1.5, C0)
    assert tolerance.max_error_ratio_general(C, C64, S, T, K, -0.75) <= 1.0


def test_against_the_cluster_plan(sg):
    # with the narrow tile switched off the product takes the 128 x 128 tile's
    # cluster plan: both within the bound, not bit for bit (the k-steps are
    # summed in different orders)
    M, N, K = 1024, 1024, 1024
    A, B = gen.operands(M, N, K, seed=715)
    c_ks = run_sgemm(sg, A, B)
    sg.sgemm_test_switches(1024)
    assert sg.sgemm_f32_plan(M, N, K)[3] == 128
    c_wide = run_sgemm(sg, A, B)
    check_full(c_ks, A, B)
    check_full(c_wide, A, B)


def test_timeout(sg):
    """Copies never issued: every CTA gives up after the wait limit, nothing is
    written, and the device stays usable."""
    import torch
    M, N, K = 1024, 1024, 1024
    ksplit_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=716)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(np.full((M, N), CANARY_BITS, np.int32).view(np.float32)).cuda()
    sg.sgemm_test_switches(1, 50_000_000)
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    sg.sgemm_test_switches(0)
    sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)

"""The narrow tiles (128 x 64 tiles, 8 x 8 packed per thread, every tile split
over a thread-block cluster; 2 stages and four CTAs per SM on the TMA kernel,
3 stages and three on the cp.async kernel), which sgemm_f32 takes when a
product has fewer 128 x 128 tiles than SMs and the plan's cost model prefers
them: against the FP64 oracle with ragged edges and a partial last k-step, on
both kernels with every copy width, exactly on small integers, bit for bit
from run to run, with alpha/beta, within the bound of the 128 x 128 tile's
result, and on the bounded-wait path (no fault, no hang)."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, check_full, check_rows, run_sgemm

pytestmark = pytest.mark.gpu

NO_NARROW = 1024
FORCE_CP = 2        # route every product to the cp.async-fed kernel (test-only)


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


def ld4(n):
    return (n + 3) // 4 * 4


def narrow_plan(sg, M, N, K, aligned=True):
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K, aligned)
    assert tn == 64 and full == 0 and cs in (2, 4, 8), (M, N, K, tiles, full, cs, tn)
    assert tiles == -(-M // 128) * -(-N // 64)
    return cs


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (512, 512, 4096), (768, 768, 768), (257, 130, 1000),
                                   (640, 640, 8192), (1000, 200, 777), (129, 65, 2000)])
def test_matches_oracle(sg, M, N, K):
    # leading dimensions padded to 4 floats keep every case on the TMA path
    narrow_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=600 + M % 97)
    C = run_sgemm(sg, A, B, lda=ld4(K), ldb=ld4(N), ldc=ld4(N))
    check_full(C, A, B)


@pytest.mark.parametrize("M,N,K", [(2048, 1024, 2048), (1000, 2000, 4096), (256, 8192, 2048), (4096, 512, 2048)])
def test_wide_grids_sampled(sg, M, N, K):
    narrow_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=610)
    C = run_sgemm(sg, A, B)
    rows = [0, 1, 127, 128, M // 2, M - 129, M - 2, M - 1] + list(np.random.default_rng(M).integers(0, M, 12))
    check_rows(C, A, B, rows)


def test_integers_exact(sg):
    narrow_plan(sg, 384, 320, 1536)
    A, B = gen.operands(384, 320, 1536, seed=620, integer_copy=True)
    check_full(run_sgemm(sg, A, B), A, B, exact=True)


def test_bitwise_repeatable(sg):
    import torch
    narrow_plan(sg, 768, 640, 3000)
    A, B = gen.operands(768, 640, 3000, seed=621)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c1 = sg.matmul(dA, dB)
    c2 = sg.matmul(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_against_the_wide_tile(sg):
    # the two tiles divide the k-steps differently, so they agree within the
    # bound, not bit for bit; switching the narrow tile off restores the wide one
    import torch
    M, N, K = 768, 1024, 2048
    narrow_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=622)
    c_narrow = run_sgemm(sg, A, B)
    sg.sgemm_test_switches(NO_NARROW)
    assert sg.sgemm_f32_plan(M, N, K)[3] == 128
    c_wide = run_sgemm(sg, A, B)
    check_full(c_narrow, A, B)
    check_full(c_wide, A, B)


def test_alpha_beta(sg):
    from oracle import ref_gemm, tolerance
    from test_gemm_general_gpu import run_gemm
    M, N, K = 300, 260, 1000
    narrow_plan(sg, M, N, K)
    A = gen.matrix(623, gen.STREAM_A, M, K)
    B = gen.matrix(623, gen.STREAM_B, K, N)
    C0 = gen.matrix(624, gen.STREAM_A, M, N)
    C = run_gemm(sg, 0, 0, 0, -0.75, A, B, 1.5, C0)
    C64, S, T = ref_gemm.gemm_general_f64(False, False, -0.75, A, B, 1.5, C0)
    assert tolerance.max_error_ratio_general(C, C64, S, T, K, -0.75) <= 1.0


def test_timeout(sg):
    """Copies never issued: every block of every narrow cluster gives up after
    the wait limit, nothing is written, and the device stays usable."""
    import torch
    M, N, K = 512, 512, 1024
    narrow_plan(sg, M, N, K)
    A, B = gen.operands(M, N, K, seed=625)
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


# ------------------------------------------------------------------ the cp.async kernel's narrow tile
# (operands that are not TMA-addressable take the phased TMA kernel's narrow
# tile by default, tested in test_phased_gpu.py; a test-only switch keeps these
# on the cp.async-fed kernel)

@pytest.mark.parametrize("M,N,K,pad_a,pad_b", [(512, 512, 512, 1, 1), (257, 130, 1000, 1, 3), (1000, 200, 777, 3, 1),
                                               (129, 65, 2000, 1, 1), (768, 640, 3000, 2, 2),
                                               (512, 256, 1024, 4, 1),   # A 16-byte copies, B 4-byte
                                               (512, 256, 1024, 1, 4),   # A 4-byte, B 16-byte
                                               (300, 190, 999, 4, 2)])   # A 16-byte, B 4-byte, ragged
def test_cp_matches_oracle(sg, M, N, K, pad_a, pad_b):
    # rows of A and B padded so that at least one operand is not TMA-addressable
    sg.sgemm_test_switches(FORCE_CP)
    narrow_plan(sg, M, N, K, aligned=False)
    A, B = gen.operands(M, N, K, seed=630 + M % 89)
    lda = ld4(K) + 4 if pad_a == 4 else K + pad_a      # pad 4: rows 16-byte aligned
    ldb = ld4(N) + 4 if pad_b == 4 else N + pad_b
    C = run_sgemm(sg, A, B, lda=lda, ldb=ldb, ldc=N + 1)
    check_full(C, A, B)


def test_cp_unaligned_base(sg):
    M, N, K = 384, 320, 1500
    sg.sgemm_test_switches(FORCE_CP)
    narrow_plan(sg, M, N, K, aligned=False)
    A, B = gen.operands(M, N, K, seed=640)
    check_full(run_sgemm(sg, A, B, a_off=1, b_off=2, c_off=3), A, B)


def test_cp_wide_grid_sampled(sg):
    M, N, K = 2048, 1024, 2048
    sg.sgemm_test_switches(FORCE_CP)
    narrow_plan(sg, M, N, K, aligned=False)
    A, B = gen.operands(M, N, K, seed=641)
    C = run_sgemm(sg, A, B, lda=K + 1, ldb=N + 1)
    rows = [0, 1, 127, 128, 1024, M - 129, M - 2, M - 1] + list(np.random.default_rng(7).integers(0, M, 12))
    check_rows(C, A, B, rows)


def test_cp_integers_exact_and_repeatable(sg):
    import torch
    M, N, K = 384, 320, 1537
    sg.sgemm_test_switches(FORCE_CP)
    narrow_plan(sg, M, N, K, aligned=False)
    A, B = gen.operands(M, N, K, seed=642, integer_copy=True)
    c1 = run_sgemm(sg, A, B)
    c2 = run_sgemm(sg, A, B)
    check_full(c1, A, B, exact=True)
    assert np.array_equal(c1, c2)

"""sgemm_gemm: C = alpha op(A) op(B) + beta C with transposes, on the FFMA and
3xTF32 algorithms, against the FP64 oracle of the same general form with the
bound 2 (K + 2) u (|alpha| sum|a||b| + |beta||c|)."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, GUARD, WS_GUARD, _device_buffer
from oracle import ref_gemm, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    return sg


def stored(M, N, K, ta, tb, seed, integer=False):
    dist = "int" if integer else "uniform"
    sa, sb = (gen.STREAM_A_INT, gen.STREAM_B_INT) if integer else (gen.STREAM_A, gen.STREAM_B)
    A = gen.matrix(seed, sa, K if ta else M, M if ta else K, dist)
    B = gen.matrix(seed, sb, N if tb else K, K if tb else N, dist)
    C0 = gen.matrix(seed + 1, sa, M, N, dist)
    return A, B, C0


def run_gemm(sg, algo, ta, tb, alpha, A, B, beta, C0, lda=None, ldb=None, ldc=None, a_off=0, c_off=0):
    """Run sgemm_gemm on canary-guarded buffers; C starts as C0."""
    import torch
    dev = torch.device("cuda", 0)
    M, N = C0.shape
    K = A.shape[0] if ta else A.shape[1]
    lda = lda or max(A.shape[1], 1)
    ldb = ldb or max(B.shape[1], 1)
    ldc = ldc or max(N, 1)
    a_buf, pa = _device_buffer(A, lda, a_off, torch, dev)
    b_buf, pb = _device_buffer(B, ldb, 0, torch, dev)
    c_buf, pc = _device_buffer(C0, ldc, c_off, torch, dev)
    need = sg.sgemm_gemm_workspace_size(algo, ta, tb, M, N, K)
    ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
    sg.sgemm_gemm(algo, ta, tb, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, ws.data_ptr() + 4 * WS_GUARD, need)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    w = ws.cpu().numpy()
    assert np.isnan(w[:WS_GUARD]).all() and np.isnan(w[-WS_GUARD:]).all()
    host = c_buf.cpu().numpy().view(np.int32)
    start = GUARD + c_off
    C = np.empty((M, N), np.float32)
    touched = np.zeros(host.size, bool)
    for r in range(M):
        C[r] = host[start + r * ldc: start + r * ldc + N].view(np.float32)
        touched[start + r * ldc: start + r * ldc + N] = True
    assert np.all(host[~touched] == CANARY_BITS), "wrote outside the M x N block of C"
    return C


def check_general(C, ta, tb, alpha, A, B, beta, C0):
    C64, S, T = ref_gemm.gemm_general_f64(ta, tb, alpha, A, B, beta, C0)
    K = A.shape[0] if ta else A.shape[1]
    r = tolerance.max_error_ratio_general(C, C64, S, T, K, alpha)
    assert r <= 1.0, f"error/bound {r:.3g}"


ALGOS = [0, 1]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("tb", [0, 1])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.5, 1.0), (2.5, -1.5)])
def test_transposes_alpha_beta(sg, algo, ta, tb, alpha, beta):
    M, N, K = 150, 133, 270
    A, B, C0 = stored(M, N, K, ta, tb, seed=100 + 2 * ta + tb)
    C = run_gemm(sg, algo, ta, tb, alpha, A, B, beta, C0)
    check_general(C, ta, tb, alpha, A, B, beta, C0)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_integers_exact(sg, algo, ta, tb):
    M, N, K = 70, 90, 300
    A, B, C0 = stored(M, N, K, ta, tb, seed=110, integer=True)
    C = run_gemm(sg, algo, ta, tb, 2.0, A, B, -1.0, C0)
    C64, _, _ = ref_gemm.gemm_general_f64(ta, tb, 2.0, A, B, -1.0, C0)
    assert np.array_equal(C.astype(np.float64), C64)


@pytest.mark.parametrize("algo", ALGOS)
def test_beta_zero_never_reads_c(sg, algo):
    M, N, K = 64, 80, 96
    A, B, _ = stored(M, N, K, 1, 0, seed=111)
    C0 = np.full((M, N), np.nan, np.float32)
    C = run_gemm(sg, algo, 1, 0, 1.5, A, B, 0.0, C0)
    assert np.isfinite(C).all()
    check_general(C, 1, 0, 1.5, A, B, 0.0, np.zeros((M, N), np.float32))


@pytest.mark.parametrize("algo", ALGOS)
def test_alpha_zero_and_k_zero_do_not_read_a_b(sg, algo):
    M, N, K = 40, 50, 60
    A = np.full((M, K), np.nan, np.float32)
    B = np.full((K, N), np.nan, np.float32)
    C0 = gen.matrix(112, gen.STREAM_A, M, N)
    C = run_gemm(sg, algo, 0, 0, 0.0, A, B, -2.0, C0)
    assert np.array_equal(C, (np.float32(-2.0) * C0).astype(np.float32))
    Z = run_gemm(sg, algo, 0, 0, 3.0, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), 0.5, C0)
    assert np.array_equal(Z, (np.float32(0.5) * C0).astype(np.float32))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("ta,tb", [(1, 1), (0, 1)])
def test_strides_and_offsets(sg, algo, ta, tb):
    M, N, K = 97, 61, 130
    A, B, C0 = stored(M, N, K, ta, tb, seed=113)
    C = run_gemm(sg, algo, ta, tb, 0.75, A, B, 0.25, C0, lda=A.shape[1] + 3, ldb=B.shape[1] + 5, ldc=N + 2,
                 a_off=1, c_off=3)
    check_general(C, ta, tb, 0.75, A, B, 0.25, C0)


def test_plain_case_is_bitwise_sgemm_f32(sg):
    # alpha = 1, beta = 0, no transposes on the FFMA algorithm is exactly sgemm_f32
    import torch
    A, B = gen.operands(300, 264, 200, seed=114)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c1 = torch.empty(300, 264, device="cuda")
    c2 = torch.full((300, 264), float("nan"), device="cuda")
    sg.sgemm_f32(300, 264, 200, dA, 200, dB, 264, c1, 264)
    sg.sgemm_gemm(0, 0, 0, 300, 264, 200, 1.0, dA, 200, dB, 264, 0.0, c2, 264)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_square_1024_transposed_both(sg):
    A, B, C0 = stored(1024, 1024, 1024, 1, 1, seed=115)
    for algo in ALGOS:
        C = run_gemm(sg, algo, 1, 1, 1.0, A, B, 1.0, C0)
        check_general(C, 1, 1, 1.0, A, B, 1.0, C0)


def test_cp_async_path_with_alpha_beta(sg):
    # force the cp.async kernel (test-only switch) on the FFMA algorithm
    A, B, C0 = stored(130, 140, 150, 0, 0, seed=116)
    sg.sgemm_test_switches(2, 2_000_000_000)
    try:
        C = run_gemm(sg, 0, 0, 0, -1.25, A, B, 0.5, C0)
    finally:
        sg.sgemm_test_switches(0, 2_000_000_000)
    check_general(C, 0, 0, -1.25, A, B, 0.5, C0)


def test_bad_arguments(sg):
    import torch
    x = torch.zeros(4096, device="cuda")
    y = torch.zeros(4096, device="cuda")
    z = torch.zeros(4096, device="cuda")
    with pytest.raises(sg.SgemmError):          # bad algo
        sg.sgemm_gemm(7, 0, 0, 8, 8, 8, 1.0, x, 8, y, 8, 0.0, z, 8)
    with pytest.raises(sg.SgemmError):          # transposed A needs lda >= M
        sg.sgemm_gemm(0, 1, 0, 16, 8, 8, 1.0, x, 8, y, 8, 0.0, z, 8)
    with pytest.raises(sg.SgemmError):          # transposes on FFMA need a workspace
        sg.sgemm_gemm(0, 1, 0, 8, 8, 8, 1.0, x, 8, y, 8, 0.0, z, 8)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.75, 1.5)])
@pytest.mark.parametrize("M,N,K", [(190, 170, 150), (3, 170, 150), (190, 170, 2)])
@pytest.mark.parametrize("a_off,lda_pad,ldb_pad", [(1, 0, 0), (0, 1, 0), (0, 0, 3), (2, 5, 1)])
def test_unaligned_operands(sg, M, N, K, a_off, lda_pad, ldb_pad, alpha, beta):
    # FFMA form with unaligned A or B: read in place through phase maps, or
    # (M or K below 4) repacked into the workspace; the product must not
    # change, only its kernel
    A, B, C0 = stored(M, N, K, 0, 0, seed=117)
    C = run_gemm(sg, 0, 0, 0, alpha, A, B, beta, C0, lda=K + lda_pad, ldb=N + ldb_pad, a_off=a_off)
    check_general(C, 0, 0, alpha, A, B, beta, C0)


def test_unaligned_operands_need_no_workspace(sg):
    import torch
    M, N, K = 260, 300, 333
    A, B, C0 = stored(M, N, K, 0, 0, seed=118)
    dA = torch.zeros(M * (K + 1) + 1, device="cuda")
    dB = torch.zeros(K * (N + 3), device="cuda")
    for r in range(M):
        dA[1 + r * (K + 1): 1 + r * (K + 1) + K] = torch.from_numpy(A[r]).cuda()
    for r in range(K):
        dB[r * (N + 3): r * (N + 3) + N] = torch.from_numpy(B[r]).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    sg.sgemm_gemm(0, 0, 0, M, N, K, 0.5, dA.data_ptr() + 4, K + 1, dB, N + 3, 0.0, dC, N, None, 0)
    torch.cuda.synchronize()
    check_general(dC.cpu().numpy(), 0, 0, 0.5, A, B, 0.0, C0)


def test_ragged_workload_through_sgemm_gemm(sg):
    import torch
    M, N, K, dist, seed = gen.WORKLOADS["ragged_3001x4999x2047"]
    A, B = gen.operands(M, N, K, seed=seed, dist=dist)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    need = sg.sgemm_gemm_workspace_size(0, 0, 0, M, N, K)
    ws = torch.empty(need // 4, device="cuda")
    sg.sgemm_gemm(0, 0, 0, M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, ws, need)
    torch.cuda.synchronize()
    C = dC.cpu().numpy()
    from helpers import check_rows
    check_rows(C, A, B, [0, 1, 127, 128, 2999, 3000] + list(np.random.default_rng(8).integers(0, M, 20)))

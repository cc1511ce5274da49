"""Parity of the 3xTF32 tensor-core product (sgemm_f32_3xtf32) with the FP64
oracle under the same bound as the FP32 kernels, |C - C64| <= 2 K u sum|a||b|,
and exactly for small integers; plus workspace handling and the bounded-wait
timeout path of the tcgen05 kernel."""

import numpy as np
import pytest

import gen
from helpers import (CANARY_BITS, GUARD, WS_GUARD, _device_buffer, check_entries, check_full,
                     check_full_blocked, check_rows, workload_operands)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    return sg


def run_x3(sg, A, B, lda=None, ldb=None, ldc=None, a_off=0, b_off=0, c_off=0):
    """C = A * B through sgemm_f32_3xtf32 with canaries around C and the workspace."""
    import torch
    dev = torch.device("cuda", 0)
    M, K = A.shape
    N = B.shape[1]
    lda, ldb, ldc = lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1)
    a_buf, pa = _device_buffer(A, lda, a_off, torch, dev)
    b_buf, pb = _device_buffer(B, ldb, b_off, torch, dev)
    c_buf, pc = _device_buffer(np.zeros((M, 0), np.float32), ldc, c_off, torch, dev)
    need = sg.sgemm_f32_3xtf32_workspace_size(M, N, K)
    ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
    sg.sgemm_f32_3xtf32(M, N, K, pa, lda, pb, ldb, pc, ldc, ws.data_ptr() + 4 * WS_GUARD, need)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    w = ws.cpu().numpy()
    assert np.isnan(w[:WS_GUARD]).all() and np.isnan(w[-WS_GUARD:]).all(), "wrote outside the workspace"
    host = c_buf.cpu().numpy().view(np.int32)
    start = GUARD + c_off
    C = np.empty((M, N), np.float32)
    touched = np.zeros(host.size, bool)
    for r in range(M):
        C[r] = host[start + r * ldc: start + r * ldc + N].view(np.float32)
        touched[start + r * ldc: start + r * ldc + N] = True
    assert np.all(host[~touched] == CANARY_BITS), "wrote outside the M x N block of C"
    return C


def test_one_tile(sg):
    A, B = gen.operands(128, 256, 32, seed=70)
    check_full(run_x3(sg, A, B), A, B)


def test_integer_exact(sg):
    A = gen.matrix(71, gen.STREAM_A_INT, 300, 1000, "int")
    B = gen.matrix(71, gen.STREAM_B_INT, 1000, 257, "int")
    check_full(run_x3(sg, A, B), A, B, exact=True)


def test_tiny_6x6x9(sg):
    A, B = gen.operands(6, 6, 9, seed=0)
    check_full(run_x3(sg, A, B), A, B)
    Ai, Bi = gen.operands(6, 6, 9, seed=0, integer_copy=True)
    check_full(run_x3(sg, Ai, Bi), Ai, Bi, exact=True)


def test_square_1024(sg):
    A, B = gen.operands(1024, 1024, 1024, seed=1)
    check_full(run_x3(sg, A, B), A, B)


def test_identity_exact_on_tf32_values(sg):
    # an identity times a matrix of TF32-representable values is exact
    A = gen.matrix(72, gen.STREAM_A_INT, 200, 160, "int") / np.float32(8)
    I = np.eye(160, dtype=np.float32)
    assert np.array_equal(run_x3(sg, A.astype(np.float32), I), A)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 33), (129, 257, 31), (200, 300, 100), (130, 513, 257),
                                   (256, 256, 512)])
def test_ragged_shapes(sg, M, N, K):
    A, B = gen.operands(M, N, K, seed=73)
    check_full(run_x3(sg, A, B), A, B)


def test_strides_and_unaligned_pointers(sg):
    A, B = gen.operands(150, 140, 100, seed=74)
    check_full(run_x3(sg, A, B, lda=103, ldb=141, ldc=147, a_off=1, b_off=3, c_off=2), A, B)


def test_deterministic(sg):
    A, B = gen.operands(333, 444, 555, seed=75)
    assert np.array_equal(run_x3(sg, A, B), run_x3(sg, A, B))


def _device_x3(sg, A, B):
    import torch
    C = sg.matmul_3xtf32(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    return C.cpu().numpy()


def test_ragged_3001x4999x2047_full(sg):
    M, N, K, dist, seed = gen.WORKLOADS["ragged_3001x4999x2047"]
    A, B = workload_operands("ragged_3001x4999x2047")
    C = _device_x3(sg, A, B)
    check_rows(C, A, B, [0, 1, 127, 128, 2999, 3000] + list(np.random.default_rng(3).integers(0, M, 20)))
    check_full_blocked(C, A, B, key="ragged_3001x4999x2047")


def test_square_8192_full(sg):
    M, N, K, dist, seed = gen.WORKLOADS["square_8192"]
    A, B = workload_operands("square_8192")
    C = _device_x3(sg, A, B)
    assert np.isfinite(C).all()
    check_rows(C, A, B, [0, 127, 128, 4095, 8191])
    rng = np.random.default_rng(6)
    check_entries(C, A, B, rng.integers(0, M, 2000), rng.integers(0, N, 2000))
    check_full_blocked(C, A, B, key="square_8192")


def test_skinny_full(sg):
    M, N, K, dist, seed = gen.WORKLOADS["skinny_16384x16384x32"]
    A, B = workload_operands("skinny_16384x16384x32")
    C = _device_x3(sg, A, B)
    check_rows(C, A, B, [0, 16383] + list(np.random.default_rng(7).integers(0, M, 10)))
    check_full_blocked(C, A, B, key="skinny_16384x16384x32")


def test_timeout_path(sg):
    import torch
    A, B = gen.operands(128, 256, 64, seed=76)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(np.full((128, 256), CANARY_BITS, np.int32).view(np.float32)).cuda()
    need = sg.sgemm_f32_3xtf32_workspace_size(128, 256, 64)
    ws = torch.empty(need // 4, device="cuda")
    try:
        sg.sgemm_test_switches(1, 50_000_000)
        sg.sgemm_f32_3xtf32(128, 256, 64, dA, 64, dB, 256, dC, 256, ws, need)
        assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
        assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    finally:
        sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_f32_3xtf32(128, 256, 64, dA, 64, dB, 256, dC, 256, ws, need)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)


# ---------------------------------------------------------------- split-K for small grids

def _operand_bytes(M, N, K):
    kpad = (K + 3) // 4 * 4
    return (4 * kpad * (2 * M + 2 * N) + 255) // 256 * 256


from test_plan_model import x3_expected_layout as _expected_layout  # noqa: E402


@pytest.mark.parametrize("M,N,K,seed", [(256, 256, 4096, 80), (1024, 1024, 1024, 81), (300, 200, 1000, 82),
                                        (129, 500, 777, 83)])
def test_divided_products(sg, M, N, K, seed):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    width, splits = _expected_layout(M, N, K, sms)
    assert splits > 1
    assert sg.sgemm_f32_3xtf32_plan_model(M, N, K, sms) == (width, splits)
    ldp = (N + 3) // 4 * 4
    assert sg.sgemm_f32_3xtf32_workspace_size(M, N, K) == _operand_bytes(M, N, K) + splits * M * ldp * 4
    A, B = gen.operands(M, N, K, seed=seed)
    check_full(run_x3(sg, A, B), A, B)


def test_divided_product_integers_and_repeatability(sg):
    import torch
    A = gen.matrix(84, gen.STREAM_A_INT, 512, 2048, "int")
    B = gen.matrix(84, gen.STREAM_B_INT, 2048, 300, "int")
    C = run_x3(sg, A, B)
    check_full(C, A, B, exact=True)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c1 = sg.matmul_3xtf32(dA, dB)
    c2 = sg.matmul_3xtf32(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_divided_product_alpha_beta(sg):
    from oracle import ref_gemm, tolerance
    from test_gemm_general_gpu import run_gemm
    A = gen.matrix(85, gen.STREAM_A, 3000, 400)      # stored K x M: op(A) = A^T is 400 x 3000
    B = gen.matrix(85, gen.STREAM_B, 3000, 300)
    C0 = gen.matrix(86, gen.STREAM_A, 400, 300)
    C = run_gemm(sg, 1, 1, 0, -1.5, A, B, 0.75, C0)
    C64, S, T = ref_gemm.gemm_general_f64(True, False, -1.5, A, B, 0.75, C0)
    assert tolerance.max_error_ratio_general(C, C64, S, T, 3000, -1.5) <= 1.0


def test_divided_product_timeout_reports(sg):
    import torch
    M, N, K = 256, 256, 2048
    A, B = gen.operands(M, N, K, seed=87)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.empty(M, N, device="cuda")
    need = sg.sgemm_f32_3xtf32_workspace_size(M, N, K)
    assert need > _operand_bytes(M, N, K)
    ws = torch.empty(need // 4, device="cuda")
    try:
        sg.sgemm_test_switches(1, 50_000_000)
        sg.sgemm_f32_3xtf32(M, N, K, dA, K, dB, N, dC, N, ws, need)
        assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    finally:
        sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_f32_3xtf32(M, N, K, dA, K, dB, N, dC, N, ws, need)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)


# One shape per tile width: 10 rows of tiles (M = 1279, a ragged last row) and
# N chosen so that the width rule picks each of 208 .. 128 on 152 SMs; K = 40
# ends in a half k-step.  Each is checked on every element, once with C rows
# 16-byte aligned (quad stores) and once with ldc = N + 1 (scalar stores).
WIDTH_SHAPES = {208: 2881, 192: 2641, 176: 2401, 160: 2161, 144: 1921, 128: 1000}


@pytest.mark.parametrize("width", sorted(WIDTH_SHAPES))
@pytest.mark.parametrize("odd_ldc", [False, True])
def test_every_tile_width(sg, width, odd_ldc):
    import torch
    M, N, K = 1279, WIDTH_SHAPES[width], 40
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip(f"widths mapped for 152 SMs, this device has {sms}")
    assert sg.sgemm_f32_3xtf32_plan_model(M, N, K, sms) == (width, 1)
    A, B = gen.operands(M, N, K, seed=90 + width)
    check_full(run_x3(sg, A, B, ldc=N + 1 if odd_ldc else None), A, B)


def test_narrow_width_integers_exact_and_alpha_beta(sg):
    import torch
    dev = torch.device("cuda", 0)
    M, N, K = 1279, WIDTH_SHAPES[208], 40
    Ai = gen.matrix(91, gen.STREAM_A_INT, M, K, "int")
    Bi = gen.matrix(91, gen.STREAM_B_INT, K, N, "int")
    check_full(run_x3(sg, Ai, Bi), Ai, Bi, exact=True)
    # C = 2 A B - 3 C0 on the 3xTF32 algorithm: integers stay exact
    C0 = gen.matrix(92, gen.STREAM_A_INT, M, N, "int")
    a, b, c = (torch.from_numpy(x).to(dev) for x in (Ai, Bi, C0))
    need = sg.sgemm_gemm_workspace_size(1, 0, 0, M, N, K)
    ws = torch.empty(max(need // 4, 1), device=dev)
    sg.sgemm_gemm(1, 0, 0, M, N, K, 2.0, a, K, b, N, -3.0, c, N, ws, need)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    want = 2.0 * (Ai.astype(np.float64) @ Bi.astype(np.float64)) - 3.0 * C0.astype(np.float64)
    assert np.array_equal(c.cpu().numpy().astype(np.float64), want)

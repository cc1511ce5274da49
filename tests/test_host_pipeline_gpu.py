"""sgemm_f32_host: host-memory operands, copies overlapped with the product
over row panels (the first panel's product block by block over the column
blocks of B).  Within the oracle's bound for any panel count, ragged shapes and
strides; and equal bit for bit to sgemm_f32 when the cluster split is off on
both sides (same kernels, same per-element arithmetic)."""

import numpy as np
import pytest

import gen
from helpers import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    return sg


def host_product(sg, A, B, panels, lda=None, ldb=None, ldc=None):
    import torch
    M, K = A.shape
    N = B.shape[1]
    lda, ldb, ldc = lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1)
    hA = torch.zeros(M, lda).pin_memory()
    hA[:, :K] = torch.from_numpy(A)
    hB = torch.zeros(K, ldb).pin_memory()
    hB[:, :N] = torch.from_numpy(B)
    hC = torch.full((M, ldc), float("nan")).pin_memory()
    need = sg.sgemm_f32_host_workspace_size(M, N, K, panels)
    ws = torch.empty(max(need // 4, 4), device="cuda")
    s0, s1, s2 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sg.sgemm_f32_host(M, N, K, hA, lda, hB, ldb, hC, ldc, panels, ws, need, s0, s1, s2)
    s0.synchronize()
    C = hC.numpy()
    assert np.isnan(C[:, N:]).all(), "wrote into the row gap of C"
    return C[:, :N].copy()


def device_product(sg, A, B):
    import torch
    C = sg.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    return C.cpu().numpy()


NO_SPLIT = 1 << 4


@pytest.mark.parametrize("panels", [1, 2, 3, 8])
def test_equals_sgemm_f32(sg, panels):
    A, B = gen.operands(1000, 520, 300, seed=120)
    check_full(host_product(sg, A, B, panels), A, B)
    sg.sgemm_test_switches(NO_SPLIT)
    try:
        C = host_product(sg, A, B, panels)
        assert np.array_equal(C, device_product(sg, A, B))
    finally:
        sg.sgemm_test_switches(0)


def test_several_panels_and_column_blocks(sg):
    # enough rows for several wave-rounded panels; N spans 8 column blocks of B
    # with a ragged last block
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 128 * sms * 2 + 77, 128 * 17 + 40, 160
    A, B = gen.operands(M, N, K, seed=123)
    C = host_product(sg, A, B, 3)
    rows = [0, 1, 127, 128, M // 2, M - 78, M - 77, M - 1] + list(np.random.default_rng(2).integers(0, M, 10))
    from helpers import check_rows
    check_rows(C, A, B, rows)
    sg.sgemm_test_switches(NO_SPLIT)
    try:
        assert np.array_equal(host_product(sg, A, B, 3), device_product(sg, A, B))
    finally:
        sg.sgemm_test_switches(0)


def test_strides_and_ragged(sg):
    A, B = gen.operands(333, 77, 129, seed=121)
    C = host_product(sg, A, B, 4, lda=131, ldb=81, ldc=83)
    check_full(C, A, B)


def test_more_panels_than_tiles_and_tiny(sg):
    A, B = gen.operands(6, 6, 9, seed=0)
    check_full(host_product(sg, A, B, 16), A, B)
    A, B = gen.operands(300, 40, 20, seed=122)
    check_full(host_product(sg, A, B, 50), A, B)


def test_k_zero_zeroes_host_rows(sg):
    C = host_product(sg, np.zeros((5, 0), np.float32), np.zeros((0, 7), np.float32), 2)
    assert np.array_equal(C, np.zeros((5, 7), np.float32))


def test_short_workspace_is_rejected(sg):
    import torch
    h = torch.zeros(64 * 64).pin_memory()
    ws = torch.empty(16, device="cuda")
    s = torch.cuda.current_stream()
    with pytest.raises(sg.SgemmError):
        sg.sgemm_f32_host(64, 64, 64, h, 64, h, 64, h, 64, 2, ws, 64, s, s, s)


def test_back_to_back_calls_share_a_workspace(sg):
    import torch
    M, N, K = 700, 300, 200
    pairs = [gen.operands(M, N, K, seed=130 + t) for t in range(3)]
    need = sg.sgemm_f32_host_workspace_size(M, N, K, 4)
    ws = torch.empty(need // 4, device="cuda")
    s0, s1, s2 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    hosts = []
    for A, B in pairs:
        hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
        hC = torch.full((M, N), float("nan")).pin_memory()
        sg.sgemm_f32_host(M, N, K, hA, K, hB, N, hC, N, 4, ws, need, s0, s1, s2)
        hosts.append((hA, hB, hC))
    s0.synchronize()
    for (A, B), (_, _, hC) in zip(pairs, hosts):
        check_full(hC.numpy(), A, B)

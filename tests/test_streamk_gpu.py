"""sgemm_f32_streamk: the product cut into (tile, 32-deep k-step) units dealt
evenly to every resident block (two per SM); the blocks that share a tile
each add up their own slice of its partial tiles, in an order fixed by the
shape (in k order, or in groups of consecutive partial tiles when a tile has
more sharers than its slices have chunks per thread).  Parity with the FP64
oracle on every element (the long-K shapes it is planned for, and other
shapes with stream-K forced by a test-only switch, at one and two blocks per
SM), exact small integers, the same bits on every run, the workspace
contract (canaries around it, garbage on entry, errors), the fall-back to
sgemm_f32's own launch, and the bounded-wait path."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, GUARD, WS_GUARD, _device_buffer, check_full

pytestmark = pytest.mark.gpu

FORCE_STREAMK = 4096
ONE_PER_SM = 1 << 13
TWO_PER_SM = 2 << 13


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)
    sg.sgemm_device_status()


def ld4(n):
    return (n + 3) // 4 * 4


def run_streamk(sg, A, B, lda=None, ldb=None, ldc=None, c_off=0, ws_fill=float("nan"), expect_ws=None):
    """C = A * B through sgemm_f32_streamk with canaries around C and the
    workspace (which starts filled with ``ws_fill``)."""
    import torch
    dev = torch.device("cuda", 0)
    M, K = A.shape
    N = B.shape[1]
    lda, ldb, ldc = lda or ld4(K), ldb or ld4(N), ldc or max(N, 1)
    a_buf, pa = _device_buffer(A, lda, 0, torch, dev)
    b_buf, pb = _device_buffer(B, ldb, 0, torch, dev)
    c_buf, pc = _device_buffer(np.zeros((M, 0), np.float32), ldc, c_off, torch, dev)
    need = sg.sgemm_f32_streamk_workspace_size(M, N, K)
    if expect_ws is not None:
        assert (need > 0) == expect_ws
    ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
    body = ws[WS_GUARD: WS_GUARD + need // 4]
    if ws_fill == "garbage":
        body.view(torch.int32).fill_(0x7fffffff)
    else:
        body.fill_(ws_fill)
    sg.sgemm_f32_streamk(M, N, K, pa, lda, pb, ldb, pc, ldc, ws.data_ptr() + 4 * WS_GUARD, need)
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


@pytest.mark.parametrize("M,N,K", [(256, 256, 65536), (128, 128, 131072), (384, 384, 16384), (130, 250, 20000),
                                   (1024, 1024, 8192), (520, 500, 16384)])
def test_planned_long_k_shapes(sg, M, N, K):
    A, B = gen.operands(M, N, K, seed=500 + M % 97)
    check_full(run_streamk(sg, A, B, expect_ws=True), A, B)


@pytest.mark.parametrize("M,N,K", [(256, 256, 65536), (1024, 1024, 8192), (1024, 1024, 1024), (128, 128, 96),
                                   (512, 512, 16384), (2048, 2048, 8192), (384, 384, 4096)])
def test_device_plan_matches_the_model(sg, M, N, K):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sg.sgemm_f32_streamk_workspace_size(M, N, K) == sg.sgemm_f32_streamk_plan_model(M, N, K, sms, 2)[1]


@pytest.fixture(params=["one-per-sm", "two-per-sm"])
def forced(request, sg):
    sg.sgemm_test_switches(FORCE_STREAMK | (TWO_PER_SM if request.param == "two-per-sm" else ONE_PER_SM))
    return request.param


def test_square_1024_every_element(sg, forced):
    A, B = gen.operands(1024, 1024, 1024, seed=1)
    check_full(run_streamk(sg, A, B, expect_ws=True), A, B)


@pytest.mark.parametrize("M,N,K", [(1000, 1000, 1000), (129, 131, 2047), (600, 500, 65), (1, 7, 4000),
                                   (257, 64, 96), (128, 128, 8192), (2048, 1024, 128), (2048, 2048, 512),
                                   (5, 3000, 700)])
def test_ragged_shapes(sg, forced, M, N, K):
    A, B = gen.operands(M, N, K, seed=500 + M % 97)
    check_full(run_streamk(sg, A, B, expect_ws=True), A, B)


def test_integers_exact(sg):
    A = gen.matrix(501, gen.STREAM_A_INT, 200, 30000, "int")
    B = gen.matrix(501, gen.STREAM_B_INT, 30000, 300, "int")
    check_full(run_streamk(sg, A, B, expect_ws=True), A, B, exact=True)


@pytest.mark.parametrize("M,N,K", [
    (256, 384, 20000),    # 6 tiles, about 51 sharers each: every slice summed in k order
    (128, 128, 65536),    # 1 tile, 304 sharers: slices of 13-14 chunks summed in 9 groups
])
def test_same_bits_every_run_and_garbage_workspace(sg, M, N, K):
    A, B = gen.operands(M, N, K, seed=502)
    c1 = run_streamk(sg, A, B, ws_fill=0.0)
    c2 = run_streamk(sg, A, B, ws_fill="garbage")   # counters start at 0x7fffffff: the call zeroes them
    c3 = run_streamk(sg, A, B)
    assert np.array_equal(c1, c2) and np.array_equal(c1, c3)
    check_full(c1, A, B)


def test_forced_on_a_grid_of_many_tiles(sg, forced):
    # more tiles than resident blocks: not planned, but the kernel is correct there too
    A, B = gen.operands(3000, 3100, 300, seed=503)
    check_full(run_streamk(sg, A, B, expect_ws=True), A, B)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 256), (1024, 1024, 1024), (3000, 3000, 64)])
def test_products_that_fill_the_sms_run_as_sgemm_f32(sg, M, N, K):
    import torch
    A, B = gen.operands(M, N, K, seed=504)
    C = run_streamk(sg, A, B, expect_ws=False)
    ref = sg.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()).cpu().numpy()
    assert np.array_equal(C, ref)


def test_unaligned_operands_run_as_sgemm_f32(sg):
    import torch
    A, B = gen.operands(200, 100, 20000, seed=505)
    C = run_streamk(sg, A, B, lda=20001, ldb=101)
    big = torch.zeros(200, 20001, device="cuda")
    big[:, :20000] = torch.from_numpy(A).cuda()
    bigb = torch.zeros(20000, 101, device="cuda")
    bigb[:, :100] = torch.from_numpy(B).cuda()
    ref = sg.matmul(big[:, :20000], bigb[:, :100]).cpu().numpy()
    assert np.array_equal(C, ref)
    check_full(C, A, B)


def test_unaligned_c_and_strides(sg):
    A, B = gen.operands(300, 250, 9000, seed=506)
    check_full(run_streamk(sg, A, B, ldc=653, c_off=1), A, B)


def test_workspace_errors(sg):
    import torch
    M, N, K = 256, 256, 16384
    dA = torch.zeros(M, K, device="cuda")
    dB = torch.zeros(K, N, device="cuda")
    dC = torch.zeros(M, N, device="cuda")
    need = sg.sgemm_f32_streamk_workspace_size(M, N, K)
    assert need > 0
    ws = torch.empty(need // 4 + 8, device="cuda")
    for ptr, nbytes in [(0, need), (ws.data_ptr(), need - 4), (ws.data_ptr() + 4, need)]:
        with pytest.raises(sg.SgemmError) as e:
            sg.sgemm_f32_streamk(M, N, K, dA, K, dB, N, dC, N, ptr, nbytes)
        assert e.value.status == sg.SGEMM_ERR_INVALID_ARG
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_f32_streamk(M, N, K, dA, K, dB, N, dC, N, dC, need)
    assert e.value.status == sg.SGEMM_ERR_ALIAS


def test_timeout_writes_nothing(sg):
    import torch
    M, N, K = 256, 512, 16384
    A, B = gen.operands(M, N, K, seed=507)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(np.full((M, N), CANARY_BITS, np.int32).view(np.float32)).cuda()
    need = sg.sgemm_f32_streamk_workspace_size(M, N, K)
    ws = torch.empty(need // 4, device="cuda")
    sg.sgemm_test_switches(1, 50_000_000)
    sg.sgemm_f32_streamk(M, N, K, dA, K, dB, N, dC, N, ws, need)
    assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    assert np.all(dC.cpu().numpy().view(np.int32) == CANARY_BITS)
    sg.sgemm_test_switches(0)
    sg.sgemm_f32_streamk(M, N, K, dA, K, dB, N, dC, N, ws, need)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    check_full(dC.cpu().numpy(), A, B)

"""Split-K (sgemm_f32_splitk): parity with the FP64 oracle for many split
counts and shapes, on both kernels; exactness on integers; determinism; the
under-filled 1024^3 workload with the suggested split count; workspace bounds."""

import numpy as np
import pytest

import gen
from helpers import check_full, run_sgemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    return sg


@pytest.fixture(params=["auto", "cp.async"])
def path(request, sg):
    sg.sgemm_test_switches(2 if request.param == "cp.async" else 0, 2_000_000_000)
    yield request.param
    sg.sgemm_test_switches(0, 2_000_000_000)


def test_square_1024_suggested_split(sg, path):
    A, B = gen.operands(1024, 1024, 1024, seed=1)
    s = sg.sgemm_f32_splitk_suggest(1024, 1024, 1024)
    assert 2 <= s <= 8
    check_full(run_sgemm(sg, A, B, splits=s), A, B)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 64])
def test_split_counts_ragged(sg, path, splits):
    A, B = gen.operands(300, 257, 1000, seed=40 + splits)
    check_full(run_sgemm(sg, A, B, splits=splits), A, B)


@pytest.mark.parametrize("M,N,K", [(1, 1, 100), (7, 5, 33), (129, 131, 64), (256, 128, 4096), (33, 1000, 17)])
def test_shapes(sg, path, M, N, K):
    A, B = gen.operands(M, N, K, seed=50)
    check_full(run_sgemm(sg, A, B, splits=4), A, B)


def test_strides_and_offsets(sg, path):
    A, B = gen.operands(150, 140, 333, seed=51)
    C = run_sgemm(sg, A, B, lda=333 + 3, ldb=140 + 1, ldc=140 + 7, a_off=1, c_off=2, splits=3)
    check_full(C, A, B)


def test_integer_exact(sg, path):
    A = gen.matrix(52, gen.STREAM_A_INT, 200, 3000, "int")
    B = gen.matrix(52, gen.STREAM_B_INT, 3000, 190, "int")
    check_full(run_sgemm(sg, A, B, splits=6), A, B, exact=True)


def test_deterministic(sg, path):
    A, B = gen.operands(400, 300, 2000, seed=53)
    assert np.array_equal(run_sgemm(sg, A, B, splits=5), run_sgemm(sg, A, B, splits=5))


def test_k_zero_and_small_k(sg):
    A = np.zeros((20, 0), np.float32)
    B = np.zeros((0, 30), np.float32)
    assert np.array_equal(run_sgemm(sg, A, B, splits=4), np.zeros((20, 30), np.float32))
    A, B = gen.operands(20, 30, 3, seed=54)      # one k-step: split count lowered to 1
    check_full(run_sgemm(sg, A, B, splits=8), A, B)


def test_matmul_splitk_wrapper(sg):
    import torch
    A, B = gen.operands(512, 384, 2048, seed=55)
    out = sg.matmul_splitk(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    check_full(out.cpu().numpy(), A, B)


def test_workspace_overlapping_c_is_rejected(sg):
    import torch
    buf = torch.zeros(1 << 20, device="cuda")
    A = torch.zeros(64, 64, device="cuda")
    B = torch.zeros(64, 64, device="cuda")
    need = sg.sgemm_f32_splitk_workspace_size(64, 64, 4)
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_f32_splitk(64, 64, 64, A, 64, B, 64, buf, 64, 4, buf.data_ptr() + 4 * 100, need)
    assert e.value.status == sg.SGEMM_ERR_ALIAS

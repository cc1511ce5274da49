"""The pages' kernel ladder on the GPU (naive, tiled 16 / 32 / 32 padded,
2-D register-tiled): parity with the FP64 oracle on the pages' sizes and on
ragged shapes, strides, offsets, K = 0 and small integers (exact)."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, GUARD, _device_buffer, check_full

pytestmark = pytest.mark.gpu

LEVELS = [0, 1, 2, 3, 4]


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    return sg


def run_ladder(sg, level, A, B, lda=None, ldb=None, ldc=None, a_off=0, c_off=0):
    import torch
    dev = torch.device("cuda", 0)
    M, K = A.shape
    N = B.shape[1]
    lda, ldb, ldc = lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1)
    a_buf, pa = _device_buffer(A, lda, a_off, torch, dev)
    b_buf, pb = _device_buffer(B, ldb, 0, torch, dev)
    c_buf, pc = _device_buffer(np.zeros((M, 0), np.float32), ldc, c_off, torch, dev)
    sg.sgemm_f32_ladder(level, M, N, K, pa, lda, pb, ldb, pc, ldc)
    torch.cuda.synchronize()
    host = c_buf.cpu().numpy().view(np.int32)
    start = GUARD + c_off
    C = np.empty((M, N), np.float32)
    touched = np.zeros(host.size, bool)
    for r in range(M):
        C[r] = host[start + r * ldc: start + r * ldc + N].view(np.float32)
        touched[start + r * ldc: start + r * ldc + N] = True
    assert np.all(host[~touched] == CANARY_BITS)
    return C


@pytest.mark.parametrize("level", LEVELS)
def test_pages_sizes(sg, level):
    for (M, N, K), seed in [((6, 6, 9), 0), ((4, 4, 8), 80), ((8, 8, 8), 81)]:
        A, B = gen.operands(M, N, K, seed=seed)
        check_full(run_ladder(sg, level, A, B), A, B)
    Ai, Bi = gen.operands(6, 6, 9, seed=0, integer_copy=True)
    check_full(run_ladder(sg, level, Ai, Bi), Ai, Bi, exact=True)


@pytest.mark.parametrize("level", LEVELS)
def test_square_1024(sg, level):
    A, B = gen.operands(1024, 1024, 1024, seed=1)
    check_full(run_ladder(sg, level, A, B), A, B)


@pytest.mark.parametrize("level", LEVELS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (33, 17, 65), (100, 129, 31), (257, 63, 130)])
def test_ragged(sg, level, M, N, K):
    A, B = gen.operands(M, N, K, seed=82)
    check_full(run_ladder(sg, level, A, B), A, B)


@pytest.mark.parametrize("level", LEVELS)
def test_strides_offsets_and_k0(sg, level):
    A, B = gen.operands(70, 90, 50, seed=83)
    check_full(run_ladder(sg, level, A, B, lda=53, ldb=97, ldc=91, a_off=1, c_off=3), A, B)
    Z = run_ladder(sg, level, np.zeros((5, 0), np.float32), np.zeros((0, 7), np.float32))
    assert np.array_equal(Z, np.zeros((5, 7), np.float32))


def test_integer_exact_multi_tile(sg):
    A = gen.matrix(84, gen.STREAM_A_INT, 130, 300, "int")
    B = gen.matrix(84, gen.STREAM_B_INT, 300, 70, "int")
    for level in LEVELS:
        check_full(run_ladder(sg, level, A, B), A, B, exact=True)


def test_bad_level(sg):
    import torch
    x = torch.zeros(16, device="cuda")
    with pytest.raises(sg.SgemmError):
        sg.sgemm_f32_ladder(9, 2, 2, 2, x, 2, x.data_ptr() + 16, 2, x.data_ptr() + 32, 2)


# ------------------------------------------------- the product kernels against the naive kernel
# Every product kernel of sgemm_f32 adds its k-terms to each output in order,
# k = 0, 1, ..., K - 1, one round-to-nearest FMA per term starting from zero --
# packed two to an instruction, but each half an ordinary FP32 FMA -- exactly as
# the pages' naive kernel does with one scalar fmaf per term.  So when no k-split
# divides the sum (a plain grid of 128 x 128 tiles, test-only cluster size 1),
# the results must agree bit for bit.

NO_SPLIT = 1 << 4
FORCE_CP = 2
FORCE_PHASED = 2048


@pytest.mark.parametrize("path,flags,pad", [("tma", NO_SPLIT, 4), ("small-k tma", 0, 4),
                                            ("phased", NO_SPLIT, 1), ("phased, aligned", NO_SPLIT | FORCE_PHASED, 4),
                                            ("cp.async", NO_SPLIT | FORCE_CP, 1)])
@pytest.mark.parametrize("M,N,K", [(300, 260, 777), (129, 520, 64), (640, 384, 1000)])
def test_product_kernels_equal_the_naive_kernel_bitwise(sg, path, flags, pad, M, N, K):
    if path == "small-k tma" and K > 64:
        pytest.skip("the small-K tile takes K <= 64")
    A, B = gen.operands(M, N, K, seed=90 + M % 13)
    lda = (K + 3) // 4 * 4 if pad == 4 else K + pad
    ldb = (N + 3) // 4 * 4 if pad == 4 else N + pad
    naive = run_ladder(sg, 0, A, B, lda=lda, ldb=ldb)
    from helpers import run_sgemm
    sg.sgemm_test_switches(flags)
    try:
        C = run_sgemm(sg, A, B, lda=lda, ldb=ldb)
    finally:
        sg.sgemm_test_switches(0)
    assert np.array_equal(C, naive), f"{path}: {np.count_nonzero(C != naive)} outputs differ from the naive kernel"

"""Parity of sgemm_f32 (the CUDA path, called through the C interface) with the
FP64 oracle, element by element, within |C - C64| <= 2 K u sum|a||b|, and
exactly for small-integer and identity inputs."""

import numpy as np
import pytest

import gen
from helpers import check_entries, check_full, check_full_blocked, check_rows, run_sgemm, workload_operands
from oracle import ref_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    return sg


@pytest.fixture(params=["auto", "no-cluster-split", "cp.async", "phased"])
def path(request, sg):
    """Run the test with the library's own kernel choice, again with the TMA
    path's cluster split switched off, again with every product routed to the
    cp.async kernel, and again with aligned operands read through the phase
    maps of the phased TMA kernel (test-only switches)."""
    flags = {"auto": 0, "no-cluster-split": 1 << 4, "cp.async": 2, "phased": 2048}[request.param]
    sg.sgemm_test_switches(flags, 2_000_000_000)
    yield request.param
    sg.sgemm_test_switches(0, 2_000_000_000)


# ------------------------------------------------------------------ the workloads

def test_tiny_6x6x9_uniform(sg, path):
    A, B = gen.operands(6, 6, 9, seed=0)
    check_full(run_sgemm(sg, A, B), A, B)


def test_tiny_6x6x9_integer_exact(sg, path):
    A, B = gen.operands(6, 6, 9, seed=0, integer_copy=True)
    check_full(run_sgemm(sg, A, B), A, B, exact=True)


def test_square_1024_full(sg, path):
    A, B = gen.operands(1024, 1024, 1024, seed=1)
    check_full(run_sgemm(sg, A, B), A, B)


def _device_product(sg, A, B):
    """The launch configuration the benchmark times: contiguous tensors, torch's stream."""
    import torch
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.full((A.shape[0], B.shape[1]), float("nan"), device="cuda")
    sg.matmul(dA, dB, out=dC)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def _sample(M, N, rng, n=400):
    return rng.integers(0, M, n), rng.integers(0, N, n)


def test_ragged_3001x4999x2047(sg):
    M, N, K, dist, seed = gen.WORKLOADS["ragged_3001x4999x2047"]
    A, B = workload_operands("ragged_3001x4999x2047")
    C = _device_product(sg, A, B)
    assert np.isfinite(C).all()
    # first/last rows of the first and the ragged last block row, plus random rows
    rng = np.random.default_rng(3)
    rows = [0, 1, 127, 128, 2943, 2944, 2999, 3000] + list(rng.integers(0, M, 24))
    check_rows(C, A, B, rows)
    # the ragged last block column, every row
    cols = np.arange(4992 - 64, N)
    rr = np.repeat(np.arange(0, M, 7), cols.size)
    cc = np.tile(cols, np.arange(0, M, 7).size)
    check_entries(C, A, B, rr, cc)
    # and every element (the oracle's 6.1e10 FP64 multiply-adds take a few seconds)
    check_full_blocked(C, A, B, key="ragged_3001x4999x2047")


def test_square_8192_full(sg):
    M, N, K, dist, seed = gen.WORKLOADS["square_8192"]
    A, B = workload_operands("square_8192")
    C = _device_product(sg, A, B)
    assert np.isfinite(C).all()
    # sampled rows and entries first (a quick first failure), then every element
    check_rows(C, A, B, [0, 1, 127, 128, 4095, 4096, 8190, 8191])
    check_entries(C, A, B, *_sample(M, N, np.random.default_rng(2), 2000))
    check_full_blocked(C, A, B, key="square_8192")


def test_skinny_16384x16384x32_full(sg):
    M, N, K, dist, seed = gen.WORKLOADS["skinny_16384x16384x32"]
    A, B = workload_operands("skinny_16384x16384x32")
    C = _device_product(sg, A, B)
    assert np.isfinite(C).all()
    check_rows(C, A, B, [0, 127, 128, 8191, 16383] + list(np.random.default_rng(4).integers(0, M, 27)))
    check_full_blocked(C, A, B, key="skinny_16384x16384x32")


def test_square_16384_sampled(sg):
    # the headline's product at twice the size (not one of the pages'
    # examples): every output finite, whole rows at tile edges and 2000 random
    # entries against the oracle.  Every one of its 2^28 outputs passed once
    # (max error/bound 2.3e-4), but the oracle takes five minutes on 16 cores
    M, N, K, dist, seed = gen.WORKLOADS["square_16384"]
    A, B = gen.operands(M, N, K, seed=seed, dist=dist)
    C = _device_product(sg, A, B)
    assert np.isfinite(C).all()
    check_rows(C, A, B, [0, 127, 128, 8191, 8192, 16383])
    check_entries(C, A, B, *_sample(M, N, np.random.default_rng(5), 2000))


def test_longk_256x256x65536_full(sg):
    # four output tiles over 65536 k-values: sgemm_f32's narrow tiles, each
    # split over a cluster of eight CTAs; and the same product through stream-K
    import torch
    M, N, K, dist, seed = gen.WORKLOADS["longk_256x256x65536"]
    A, B = workload_operands("longk_256x256x65536")
    C = _device_product(sg, A, B)
    check_full_blocked(C, A, B, key="longk_256x256x65536")
    Cs = sg.matmul_streamk(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()).cpu().numpy()
    assert sg.sgemm_f32_streamk_workspace_size(M, N, K) > 0
    check_full_blocked(Cs, A, B, key="longk_256x256x65536")


# ------------------------------------------------------------------ exactness

def test_integer_inputs_exact_multi_tile(sg, path):
    A = gen.matrix(21, gen.STREAM_A_INT, 300, 1000, "int")
    B = gen.matrix(21, gen.STREAM_B_INT, 1000, 257, "int")
    check_full(run_sgemm(sg, A, B), A, B, exact=True)


def test_identity_exact(sg, path):
    A, B = gen.operands(203, 190, 190, seed=22)
    I = np.eye(190, dtype=np.float32)
    assert np.array_equal(run_sgemm(sg, A, I), A)
    assert np.array_equal(run_sgemm(sg, I, B), B)


def test_k_zero_writes_zeros(sg, path):
    A = np.zeros((37, 0), np.float32)
    B = np.zeros((0, 45), np.float32)
    C = run_sgemm(sg, A, B)
    assert np.array_equal(C, np.zeros((37, 45), np.float32))


# ------------------------------------------------------------------ shapes, strides, offsets

SMALL = [1, 2, 3, 5, 7, 8, 13, 31, 32, 33, 64, 65, 127, 128, 129, 130, 255, 257]


@pytest.mark.parametrize("seed", range(12))
def test_small_ragged_sweep(sg, path, seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(6):
        M, N, K = (int(rng.choice(SMALL)) for _ in range(3))
        A, B = gen.operands(M, N, K, seed=1000 + seed)
        check_full(run_sgemm(sg, A, B), A, B)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 300, 17), (300, 1, 17), (17, 19, 1), (2, 3, 70),
                                   (129, 131, 133), (61, 67, 71)])
def test_prime_and_degenerate_shapes(sg, path, M, N, K):
    A, B = gen.operands(M, N, K, seed=7)
    check_full(run_sgemm(sg, A, B), A, B)


@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad", [(1, 0, 0), (0, 3, 0), (0, 0, 5), (1, 3, 5), (4, 4, 4),
                                                     (0, 1, 2)])
def test_leading_dimensions(sg, path, lda_pad, ldb_pad, ldc_pad):
    M, N, K = 150, 140, 100
    A, B = gen.operands(M, N, K, seed=8)
    C = run_sgemm(sg, A, B, lda=K + lda_pad, ldb=N + ldb_pad, ldc=N + ldc_pad)
    check_full(C, A, B)


@pytest.mark.parametrize("a_off,b_off,c_off", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1), (2, 2, 2)])
def test_unaligned_base_pointers(sg, path, a_off, b_off, c_off):
    M, N, K = 130, 136, 72
    A, B = gen.operands(M, N, K, seed=9)
    check_full(run_sgemm(sg, A, B, a_off=a_off, b_off=b_off, c_off=c_off), A, B)


def test_sixty_four_bit_offsets(sg):
    # (M - 1) * ldc exceeds 2^31 elements: the row offset must not wrap
    import torch
    M, N, K = 5, 4, 3
    ldc = (1 << 29) + 4
    A, B = gen.operands(M, N, K, seed=10)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    buf = torch.full(((M - 1) * ldc + N,), float("nan"), device="cuda")
    sg.sgemm_f32(M, N, K, dA, K, dB, N, buf, ldc)
    torch.cuda.synchronize()
    C = torch.stack([buf[r * ldc: r * ldc + N] for r in range(M)]).cpu().numpy()
    check_full(C, A, B)
    assert torch.isnan(buf[N: N + 1000]).all().item()
    del buf


# ------------------------------------------------------------------ behaviour

def test_deterministic(sg, path):
    A, B = gen.operands(777, 555, 333, seed=11)
    assert np.array_equal(run_sgemm(sg, A, B), run_sgemm(sg, A, B))


def test_side_stream(sg, path):
    import torch
    A, B = gen.operands(256, 320, 200, seed=12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = run_sgemm(sg, A, B, stream=s)
    check_full(C, A, B)


def test_alias_and_bad_args_raise(sg):
    import torch
    x = torch.zeros(64 * 64, device="cuda")
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_f32(8, 8, 8, x, 8, x.data_ptr() + 4 * 1024, 8, x.data_ptr() + 4 * 32, 8)
    assert e.value.status == sg.SGEMM_ERR_ALIAS
    with pytest.raises(sg.SgemmError):
        sg.sgemm_f32(8, 8, 8, x, 4, x, 8, x.data_ptr() + 4 * 2048, 8)


def test_matmul_wrapper_strided_views(sg):
    import torch
    A, B = gen.operands(100, 90, 80, seed=13)
    bigA = torch.zeros(100, 96, device="cuda")
    bigA[:, :80] = torch.from_numpy(A).cuda()
    out = sg.matmul(bigA[:, :80], torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    check_full(out.cpu().numpy(), A, B)


@pytest.mark.parametrize("case", ["a_rows_beyond_2gib", "a_vec_stride_demoted", "b_vec_stride_demoted"])
def test_strides_beyond_32_bits(sg, case):
    # the cp.async kernel keeps its copy strides in 32 bits: 16-byte copies of A
    # step 16 rows, of B 4 rows.  16 * lda >= 2^31 or 4 * ldb >= 2^31 must fall
    # back to 4-byte copies, and an unaligned A with 4 * lda >= 2^31 to the
    # 64-bit ladder kernel -- each still the exact product
    import torch
    M, N, K = 3, 5, 7
    if case == "a_rows_beyond_2gib":
        lda, ldb = (1 << 29) + 1, N              # unaligned A, 4 * lda > 2^31
    elif case == "a_vec_stride_demoted":
        lda, ldb = (1 << 27) + 4, N + 1          # aligned A with 16 * lda > 2^31; B unaligned
        M, K = 2, 64
    else:
        lda, ldb = K + 1, (1 << 29) + 4          # aligned B with 4 * ldb > 2^31; A unaligned
        K = 2
    A, B = gen.operands(M, N, K, seed=12, integer_copy=True)
    dA = torch.zeros((M - 1) * lda + K, device="cuda")
    dB = torch.zeros((K - 1) * ldb + N, device="cuda")
    for r in range(M):
        dA[r * lda: r * lda + K] = torch.from_numpy(A[r]).cuda()
    for r in range(K):
        dB[r * ldb: r * ldb + N] = torch.from_numpy(B[r]).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    sg.sgemm_f32(M, N, K, dA, lda, dB, ldb, C, N)
    torch.cuda.synchronize()
    C64, _ = ref_gemm.gemm_f64(A, B)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), C64)
    # one split where the cp.async kernel cannot run; the product is still exact
    need = sg.sgemm_f32_splitk_workspace_size(M, N, 2)
    ws = torch.empty(max(need // 4, 4), device="cuda")
    C2 = torch.full((M, N), float("nan"), device="cuda")
    sg.sgemm_f32_splitk(M, N, K, dA, lda, dB, ldb, C2, N, 2, ws, need)
    torch.cuda.synchronize()
    assert np.array_equal(C2.cpu().numpy().astype(np.float64), C64)
    del dA, dB

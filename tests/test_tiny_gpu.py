"""The one-thread-per-output kernel for tiny products (at most 16384 outputs,
1 <= K <= 128; "Shared Memory Tiling", 'The naive kernel'): against the FP64
oracle with odd strides, offsets and canary guard bands, exactly on small
integers, bit for bit against the tiled kernels and the pages' naive kernel,
with alpha/beta, and what sgemm_f32_plan reports for it.  The rest of the GPU
suite runs with this path off, so that its small shapes reach the tiled
kernels' edge handling."""

import numpy as np
import pytest

import gen
from helpers import check_full, run_sgemm

pytestmark = [pytest.mark.gpu, pytest.mark.tiny]


@pytest.fixture
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    return sg


SHAPES = [(1, 1, 1), (6, 6, 9), (5, 7, 128), (128, 128, 1), (1, 16384, 3), (16384, 1, 128), (100, 163, 77),
          (127, 129, 64)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_plan_reports_the_tiny_kernel(sg, M, N, K):
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K)
    assert (tn, cs) == (0, 1) and tiles == full == -(-M * N // 256)
    assert sg.sgemm_f32_plan(M, N, K, aligned=False)[3] == 0


def test_limits(sg):
    assert sg.sgemm_f32_plan(128, 128, 128)[3] == 0
    assert sg.sgemm_f32_plan(128, 128, 129)[3] != 0      # K > 128
    assert sg.sgemm_f32_plan(128, 129, 128)[3] != 0      # 16512 outputs
    assert sg.sgemm_f32_plan(16385, 1, 5)[3] != 0


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("pads", [(0, 0, 0, 0, 0, 0), (1, 3, 5, 1, 2, 3)], ids=["dense", "odd"])
def test_matches_oracle(sg, M, N, K, pads):
    lp, bp, cp, ao, bo, co = pads
    A, B = gen.operands(M, N, K, seed=600 + K)
    C = run_sgemm(sg, A, B, lda=K + lp, ldb=N + bp, ldc=N + cp, a_off=ao, b_off=bo, c_off=co)
    check_full(C, A, B)


@pytest.mark.parametrize("M,N,K", [(6, 6, 9), (100, 163, 77)])
def test_integers_exact(sg, M, N, K):
    A, B = gen.operands(M, N, K, seed=610, integer_copy=True)
    check_full(run_sgemm(sg, A, B), A, B, exact=True)


@pytest.mark.parametrize("M,N,K", [(6, 6, 9), (100, 163, 77), (127, 129, 64), (16384, 1, 128)])
def test_bitwise_equal_to_tiled_and_naive(sg, M, N, K):
    # the same per-element arithmetic (one round-to-nearest FMA per k, in order)
    # as the tiled kernels (no k-split at these K) and the pages' naive kernel
    import torch
    A, B = gen.operands(M, N, K, seed=611)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    tiny = sg.matmul(dA, dB)
    sg.sgemm_test_tiny_path(False)
    tiled = sg.matmul(dA, dB)
    sg.sgemm_test_tiny_path(True)
    naive = torch.empty_like(tiny)
    sg.sgemm_f32_ladder(0, M, N, K, dA, K, dB, N, naive, N)
    torch.cuda.synchronize()
    assert torch.equal(tiny, tiled) and torch.equal(tiny, naive)


def test_alpha_beta(sg):
    import torch
    from oracle import ref_gemm, tolerance
    M, N, K = 70, 90, 33
    A = gen.matrix(612, gen.STREAM_A, M, K)
    B = gen.matrix(612, gen.STREAM_B, K, N)
    C0 = gen.matrix(613, gen.STREAM_A, M, N)
    out = {}
    for tiny in (True, False):
        sg.sgemm_test_tiny_path(tiny)
        dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
        sg.sgemm_gemm(0, 0, 0, M, N, K, 1.75, dA, K, dB, N, -0.5, dC, N)
        assert sg.sgemm_device_status() == sg.SGEMM_OK
        out[tiny] = dC.cpu().numpy()
    sg.sgemm_test_tiny_path(True)
    C64, S, T = ref_gemm.gemm_general_f64(False, False, 1.75, A, B, -0.5, C0)
    assert tolerance.max_error_ratio_general(out[True], C64, S, T, K, 1.75) <= 1.0
    assert np.array_equal(out[True].view(np.int32), out[False].view(np.int32))


@pytest.mark.parametrize("M,N,K", [(6, 6, 9), (100, 163, 77)])
def test_other_entry_points_on_tiny_products(sg, M, N, K):
    # every entry point that runs sgemm_f32's launch takes the same kernel for
    # tiny products: one split of split-K, stream-K (which falls back to
    # sgemm_f32 when its plan fills the SMs), the allocation-free split-K and
    # the host-buffer pipeline; each result equals sgemm_f32's bit for bit
    import torch
    A, B = gen.operands(M, N, K, seed=614)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    want = sg.matmul(dA, dB)
    got = {}
    got["splitk"] = sg.matmul_splitk(dA, dB, splits=1)
    got["streamk"] = sg.matmul_streamk(dA, dB)
    c = torch.empty_like(want)
    sg.sgemm_f32_splitk_noalloc(M, N, K, dA, K, dB, N, c, N, 1)
    got["noalloc"] = c
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    ws_bytes = sg.sgemm_f32_host_workspace_size(M, N, K, 1)
    ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device="cuda")
    s0, s1, s2 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sg.sgemm_f32_host(M, N, K, hA, K, hB, N, hC, N, 1, ws, ws_bytes, s0, s1, s2)
    s0.synchronize()
    torch.cuda.synchronize()
    got["host"] = hC.cuda()
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    for name, c in got.items():
        assert torch.equal(c, want), name
    check_full(want.cpu().numpy(), A, B)

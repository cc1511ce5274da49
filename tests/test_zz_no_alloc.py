"""sgemm_f32_splitk_noalloc: the split-K product for callers that cannot
allocate device memory -- for example a plug-in that a host application hands
only its input and output buffers because the application owns the device
memory budget, or a latency-critical loop where an allocation (which may
synchronise the device) is not allowed.  Its partial products live in a fixed
array inside the library instead of a caller-provided workspace.

The test calls the entry point through the C interface twice in a row, on two
different problems, and checks each result against the workspace form
(sgemm_f32_splitk) with the tolerance the other parity tests use.  It also
checks that a request larger than the fixed array is refused without touching
C.  This file is collected last so that a run stopping at the first failure
has already run every other test; it also passes on its own in a fresh
process."""

import numpy as np
import pytest

import gen
from oracle import ref_gemm, tolerance

pytestmark = pytest.mark.gpu


def test_noalloc_matches_the_workspace_form_on_two_calls_in_a_row(cuda_device, lib):
    import torch

    import dense_fp32_matrix_04_gb300 as sg
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K, splits, seed in [(1024, 1024, 1024, 4, 60), (300, 257, 1000, 5, 61)]:
        A, B = gen.operands(M, N, K, seed=seed)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        c_noalloc = torch.full((M, N), float("nan"), device="cuda")
        c_ws = torch.full((M, N), float("nan"), device="cuda")

        st = lib.sgemm_f32_splitk_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, c_noalloc.data_ptr(), N,
                                          splits, stream)
        assert st == sg.SGEMM_OK, sg.status_string(st)

        need = lib.sgemm_f32_splitk_workspace_size(M, N, splits)
        ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
        st = lib.sgemm_f32_splitk(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, c_ws.data_ptr(), N, splits,
                                  ws.data_ptr(), need, stream)
        assert st == sg.SGEMM_OK, sg.status_string(st)
        torch.cuda.synchronize()

        got = c_noalloc.cpu().numpy()
        ref = c_ws.cpu().numpy()
        C64, S = ref_gemm.gemm_f64(A, B)
        assert np.isfinite(got).all()
        # against the existing entry point, within 2 K u sum|a||b|
        assert tolerance.max_error_ratio(got, ref.astype(np.float64), S, K) <= 1.0
        # and against the oracle, like every parity test
        assert tolerance.max_error_ratio(got, C64, S, K) <= 1.0


def test_noalloc_refuses_requests_beyond_its_fixed_array(cuda_device, lib):
    import torch

    import dense_fp32_matrix_04_gb300 as sg
    M = N = 1024
    K = 2048                       # 64 k-steps of 32: 64 splits stay 64
    dA = torch.zeros(M, K, device="cuda")
    dB = torch.zeros(K, N, device="cuda")
    dC = torch.full((M, N), 7.0, device="cuda")
    st = lib.sgemm_f32_splitk_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, 64,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == sg.SGEMM_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool((dC == 7.0).all())


def _noalloc_against_oracle(lib, M, N, K, splits, seed):
    import torch

    import dense_fp32_matrix_04_gb300 as sg
    A, B = gen.operands(M, N, K, seed=seed)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    st = lib.sgemm_f32_splitk_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, splits,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == sg.SGEMM_OK, sg.status_string(st)
    torch.cuda.synchronize()
    C64, S = ref_gemm.gemm_f64(A, B)
    assert tolerance.max_error_ratio(dC.cpu().numpy(), C64, S, K) <= 1.0


def test_noalloc_request_that_exactly_fills_the_array(cuda_device, lib):
    # 8 splits x 1024 rows x 1024 columns = 8,388,608 floats, the whole array
    _noalloc_against_oracle(lib, 1024, 1024, 256, 8, 62)


def test_noalloc_request_that_fits_only_after_the_split_count_is_lowered(cuda_device, lib):
    # K = 64 has two 32-deep k-steps, so 64 splits become 2: 2 x 2048 x 2048 floats
    # fill the array exactly, while 64 x 2048 x 2048 would not fit
    _noalloc_against_oracle(lib, 2048, 2048, 64, 64, 63)


def test_noalloc_timeout_leaves_no_stale_partials_in_c(cuda_device, lib):
    # a first call leaves valid partial sums in the shared array; a second call
    # whose copies never land (test-only switch) must not add them into C: the
    # blocks that give up fill their partial tiles with NaN
    import torch

    import dense_fp32_matrix_04_gb300 as sg
    M, N, K, splits = 512, 512, 512, 4
    _noalloc_against_oracle(lib, M, N, K, splits, 64)
    sg.sgemm_device_status()
    A, B = gen.operands(M, N, K, seed=65)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), device="cuda")
    sg.sgemm_test_switches(1, 50_000_000)
    try:
        st = lib.sgemm_f32_splitk_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, splits,
                                          torch.cuda.current_stream().cuda_stream)
        assert st == sg.SGEMM_OK
        assert sg.sgemm_device_status() == sg.SGEMM_ERR_TIMEOUT
    finally:
        sg.sgemm_test_switches(0, 2_000_000_000)
    assert bool(torch.isnan(dC).all())
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    # and the next call is correct again
    _noalloc_against_oracle(lib, M, N, K, splits, 66)

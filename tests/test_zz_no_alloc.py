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

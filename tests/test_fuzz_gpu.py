"""Seeded random cases across every product entry point: random shapes
(including 1 and values around the 128 / 64 / 32 tile edges), leading-dimension
padding, base offsets (which move operands off 16-byte alignment and onto the
phased TMA kernel, or the cp.async-fed one), forced launch shapes (no cluster split, clusters of 2 to
8, every tile split), split-K counts, the 3xTF32 path and the general form with
transposes and alpha/beta -- each compared with the FP64 oracle, element by
element, within the stated bound; C's guard bands and row gaps must stay
untouched."""

import numpy as np
import pytest

import gen
from helpers import CANARY_BITS, GUARD, WS_GUARD, _device_buffer
from oracle import ref_gemm, tolerance

pytestmark = pytest.mark.gpu

EDGES = [1, 2, 3, 31, 32, 33, 63, 64, 65, 95, 127, 128, 129, 191, 255, 256, 257, 300, 383, 511, 640]


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    sg.sgemm_device_status()
    yield sg
    sg.sgemm_test_switches(0, 2_000_000_000)


def _dim(rng, hi):
    return int(rng.choice(EDGES)) if rng.random() < 0.5 else int(rng.integers(1, hi))


def _read_c(c_buf, M, N, ldc, c_off):
    host = c_buf.cpu().numpy().view(np.int32)
    start = GUARD + c_off
    C = np.empty((M, N), np.float32)
    touched = np.zeros(host.size, bool)
    for r in range(M):
        C[r] = host[start + r * ldc: start + r * ldc + N].view(np.float32)
        touched[start + r * ldc: start + r * ldc + N] = True
    assert np.all(host[~touched] == CANARY_BITS), "wrote outside the M x N block of C"
    return C


def _case(sg, seed):
    import torch
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(5000 + seed)
    M, N, K = _dim(rng, 700), _dim(rng, 700), _dim(rng, 1500)
    entry = rng.choice(["f32", "f32", "splitk", "3xtf32", "gemm"])
    ta = tb = 0
    alpha, beta = 1.0, 0.0
    algo = 0
    if entry == "gemm":
        ta, tb = int(rng.integers(0, 2)), int(rng.integers(0, 2))
        alpha = float(rng.choice([1.0, -0.5, 2.25]))
        beta = float(rng.choice([0.0, 1.0, -0.75]))
        algo = int(rng.integers(0, 2))
    if entry == "3xtf32" or algo == 1:
        # the split's own error (up to about 12 u |ab| per product) is promised
        # within 2 (K + 2) u only once K is a few k-steps deep
        K = max(K, 16)
    # stored operand shapes
    a_rows, a_cols = (K, M) if ta else (M, K)
    b_rows, b_cols = (N, K) if tb else (K, N)
    A = gen.matrix(seed + 7000, gen.STREAM_A, a_rows, a_cols)
    B = gen.matrix(seed + 7000, gen.STREAM_B, b_rows, b_cols)
    C0 = gen.matrix(seed + 7001, gen.STREAM_A, M, N) if beta != 0.0 else np.zeros((M, N), np.float32)
    lda = a_cols + int(rng.choice([0, 0, 1, 3, 4]))
    ldb = b_cols + int(rng.choice([0, 0, 1, 2, 4]))
    ldc = N + int(rng.choice([0, 0, 3, 4]))
    a_off, b_off, c_off = (int(rng.choice([0, 0, 1, 2])) for _ in range(3))
    flags = int(rng.choice([0, 0, 1 << 4, (2 << 4) | 256, (3 << 4) | 256, (4 << 4), (8 << 4) | 256, 2, 2048]))
    sg.sgemm_test_switches(flags)
    try:
        a_buf, pa = _device_buffer(A, max(lda, 1), a_off, torch, dev)
        b_buf, pb = _device_buffer(B, max(ldb, 1), b_off, torch, dev)
        c_buf, pc = _device_buffer(C0, max(ldc, 1), c_off, torch, dev)
        lda, ldb, ldc = max(lda, 1), max(ldb, 1), max(ldc, 1)
        ws = None
        if entry == "f32":
            sg.sgemm_f32(M, N, K, pa, lda, pb, ldb, pc, ldc)
        elif entry == "splitk":
            splits = int(rng.integers(1, 9))
            need = sg.sgemm_f32_splitk_workspace_size(M, N, splits)
            ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
            sg.sgemm_f32_splitk(M, N, K, pa, lda, pb, ldb, pc, ldc, splits, ws.data_ptr() + 4 * WS_GUARD, need)
        elif entry == "3xtf32":
            need = sg.sgemm_f32_3xtf32_workspace_size(M, N, K)
            ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
            sg.sgemm_f32_3xtf32(M, N, K, pa, lda, pb, ldb, pc, ldc, ws.data_ptr() + 4 * WS_GUARD, need)
        else:
            need = sg.sgemm_gemm_workspace_size(algo, ta, tb, M, N, K)
            ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
            sg.sgemm_gemm(algo, ta, tb, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc,
                          ws.data_ptr() + 4 * WS_GUARD, need)
        assert sg.sgemm_device_status() == sg.SGEMM_OK
        if ws is not None:
            w = ws.cpu().numpy()
            assert np.isnan(w[:WS_GUARD]).all() and np.isnan(w[-WS_GUARD:]).all(), "wrote outside the workspace"
        C = _read_c(c_buf, M, N, ldc, c_off)
    finally:
        sg.sgemm_test_switches(0)
    C64, S, T = ref_gemm.gemm_general_f64(bool(ta), bool(tb), alpha, A, B, beta, C0)
    r = tolerance.max_error_ratio_general(C, C64, S, T, K, alpha)
    assert r <= 1.0, f"case {seed}: {entry} {M}x{N}x{K} ta={ta} tb={tb} flags={flags}: error/bound {r:.3g}"


@pytest.mark.parametrize("seed", range(60))
def test_random_case(sg, seed):
    _case(sg, seed)

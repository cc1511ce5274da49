"""Pins of the FP64 oracle's values against what mathematics fixes, independent of
the oracle's own code: exact integer sums, identities, closed forms, an
independent FP64 library product, and brute force at the visualizer's size
(6 x 6 x 9, "SGEMM: Shared Memory Tiling Visualizer", Problem Size).

The last group plants mistakes in the oracle (on the CPU) and checks that the
pins catch them."""

import math
from fractions import Fraction

import numpy as np
import pytest

import gen
from oracle import ref_gemm, tolerance


# ---------------------------------------------------------------- helpers

def brute_int(A, B):
    """Exact product of integer-valued matrices with Python integers."""
    M, K = A.shape
    N = B.shape[1]
    Ai = [[int(v) for v in row] for row in A]
    Bi = [[int(v) for v in row] for row in B]
    return np.array([[sum(Ai[i][k] * Bi[k][j] for k in range(K)) for j in range(N)]
                     for i in range(M)], dtype=np.float64).reshape(M, N)


def brute_exact(A, B):
    """Correctly rounded FP64 value of each element: exact rational sum of the
    exact products, rounded once (k-outer accumulation in Fractions)."""
    M, K = A.shape
    N = B.shape[1]
    acc = [[Fraction(0)] * N for _ in range(M)]
    for k in range(K):
        for i in range(M):
            a = Fraction(float(A[i, k]))
            for j in range(N):
                acc[i][j] += a * Fraction(float(B[k, j]))
    return np.array([[float(v) for v in row] for row in acc]).reshape(M, N)


def exact_pin(C, A, B):
    return np.array_equal(C, brute_int(A, B))


def close_pin(C, A, B, S):
    """Oracle error bound: sequential FP64 sum, |err| <= K * 2^-53 * S (1% slack)."""
    K = A.shape[1]
    ref = brute_exact(A, B)
    return bool(np.all(np.abs(C - ref) <= 1.01 * K * 2.0 ** -53 * S))


# ---------------------------------------------------------------- value pins

def test_integer_6x6x9_exact():
    A, B = gen.operands(6, 6, 9, seed=0, integer_copy=True)
    C, S = ref_gemm.gemm_f64(A, B)
    assert exact_pin(C, A, B)
    assert np.array_equal(S, brute_int(np.abs(A), np.abs(B)))


def test_uniform_6x6x9_brute_force():
    A, B = gen.operands(6, 6, 9, seed=0)
    C, S = ref_gemm.gemm_f64(A, B)
    assert close_pin(C, A, B, S)
    # and the fsum of exact products (another independent summation)
    for i in range(6):
        for j in range(6):
            f = math.fsum(float(A[i, k]) * float(B[k, j]) for k in range(9))
            assert abs(C[i, j] - f) <= 9 * 2.0 ** -53 * S[i, j]


def test_identity_products_exact():
    A, B = gen.operands(37, 29, 41, seed=5)
    I_k = np.eye(41, dtype=np.float32)
    C1, _ = ref_gemm.gemm_f64(A, I_k)
    assert np.array_equal(C1, A.astype(np.float64))
    C2, _ = ref_gemm.gemm_f64(I_k, B)
    assert np.array_equal(C2, B.astype(np.float64))


def test_closed_forms():
    M, N, K = 7, 5, 13
    ones = ref_gemm.gemm_f64(np.ones((M, K), np.float32), np.ones((K, N), np.float32))[0]
    assert np.all(ones == K)
    # A[i][k] = i + 1, B[k][j] = (k + 1) * (j + 1): C = (i+1)(j+1) K(K+1)/2
    A = np.fromfunction(lambda i, k: i + 1, (M, K)).astype(np.float32)
    B = np.fromfunction(lambda k, j: (k + 1) * (j + 1), (K, N)).astype(np.float32)
    C, _ = ref_gemm.gemm_f64(A, B)
    want = np.fromfunction(lambda i, j: (i + 1) * (j + 1) * K * (K + 1) / 2, (M, N))
    assert np.array_equal(C, want)
    # alternating signs cancel: A = 1, B[k][j] = (-1)^k with K even gives 0
    Bs = np.fromfunction(lambda k, j: (-1.0) ** k, (12, 3)).astype(np.float32)
    Z, S = ref_gemm.gemm_f64(np.ones((2, 12), np.float32), Bs)
    assert np.all(Z == 0) and np.all(S == 12)


def test_empty_and_degenerate_shapes():
    C, S = ref_gemm.gemm_f64(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert C.shape == (3, 4) and np.all(C == 0) and np.all(S == 0)
    C, _ = ref_gemm.gemm_f64(np.zeros((0, 5), np.float32), np.zeros((5, 4), np.float32))
    assert C.shape == (0, 4)
    a = np.array([[2.5]], np.float32)
    b = np.array([[-4.0]], np.float32)
    assert ref_gemm.gemm_f64(a, b)[0][0, 0] == -10.0


def test_against_independent_fp64_library_with_strides():
    A, B = gen.operands(257, 129, 300, seed=9)
    As = gen.strided(A, 307)[:, :300]      # lda = 307
    Bs = gen.strided(B, 131)[:, :129]      # ldb = 131
    C, S = ref_gemm.gemm_f64(As, Bs)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    assert np.all(np.abs(C - ref) <= 2 * 300 * 2.0 ** -53 * S)


def test_entries_agree_with_full_product():
    A, B = gen.operands(64, 48, 96, seed=11)
    C, S = ref_gemm.gemm_f64(A, B)
    rng = np.random.default_rng(0)
    r = rng.integers(0, 64, 50)
    c = rng.integers(0, 48, 50)
    ce, se = ref_gemm.gemm_entries(A, B, r, c)
    assert np.array_equal(ce, C[r, c]) and np.array_equal(se, S[r, c])


def test_abs_sum_is_product_of_abs():
    A, B = gen.operands(20, 30, 40, seed=12)
    _, S = ref_gemm.gemm_f64(A, B)
    ref = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64)
    assert np.allclose(S, ref, rtol=1e-13, atol=0)


# ---------------------------------------------------------------- tolerance pins

def fp32_sequential(A, B):
    """A plain FP32 dot product in increasing k, as a GPU thread would do it."""
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N), np.float32)
    for k in range(K):
        C = (C + np.float32(1) * (A[:, k:k + 1] * B[k:k + 1, :])).astype(np.float32)
    return C


def test_tolerance_accepts_fp32_rounding_and_rejects_a_dropped_term():
    A, B = gen.operands(6, 6, 9, seed=0)
    C64, S = ref_gemm.gemm_f64(A, B)
    C32 = fp32_sequential(A, B)
    assert tolerance.within(C32, C64, S, 9)
    dropped = fp32_sequential(A[:, 1:], B[1:, :])
    assert not tolerance.within(dropped, C64, S, 9)
    assert tolerance.max_error_ratio(np.full((6, 6), np.nan, np.float32), C64, S, 9) == np.inf


def test_tolerance_zero_bound_needs_exact_zero():
    C64 = np.zeros((2, 2))
    S = np.zeros((2, 2))
    assert tolerance.within(np.zeros((2, 2), np.float32), C64, S, 0)
    assert not tolerance.within(np.full((2, 2), 1e-30, np.float32), C64, S, 0)


# ---------------------------------------------------------------- planted mistakes

@pytest.mark.parametrize("mistake", ["transposed_B", "dropped_term", "sign", "swapped_rows", "lda_off_by_one"])
def test_pins_catch_planted_mistakes(mistake):
    """Each plausible oracle bug, planted on the CPU, fails the integer pin."""
    A, B = gen.operands(6, 6, 9, seed=0, integer_copy=True)
    if mistake == "transposed_B":
        Bsq = gen.matrix(0, gen.STREAM_B_INT, 9, 9, "int")
        Asq = gen.matrix(0, gen.STREAM_A_INT, 6, 9, "int")
        bad, _ = ref_gemm.gemm_f64(Asq, np.ascontiguousarray(Bsq.T))
        assert not exact_pin(bad, Asq, Bsq)
        return
    if mistake == "dropped_term":
        bad, _ = ref_gemm.gemm_f64(A[:, :-1], B[:-1, :])
    elif mistake == "sign":
        bad, _ = ref_gemm.gemm_f64(-A, B)
    elif mistake == "swapped_rows":
        bad, _ = ref_gemm.gemm_f64(A[::-1].copy(), B)
    else:
        buf = gen.strided(A, 10, fill=1.0)
        flat = buf.reshape(-1)
        bad, _ = ref_gemm.gemm_f64(np.lib.stride_tricks.as_strided(flat, (6, 9), (9 * 4, 4)), B)
    assert not exact_pin(bad, A, B)


# ---------------------------------------------------------------- the general form alpha op(A) op(B) + beta C

def test_general_form_pins():
    """alpha/beta and transposes: exact small-integer cases checked against
    brute force written independently of the oracle."""
    A = gen.matrix(90, gen.STREAM_A_INT, 9, 6, "int")      # stored K x M: op(A) = A^T is 6 x 9
    B = gen.matrix(90, gen.STREAM_B_INT, 7, 9, "int")      # stored N x K: op(B) = B^T is 9 x 7
    C0 = gen.matrix(91, gen.STREAM_A_INT, 6, 7, "int")
    C64, S, T = ref_gemm.gemm_general_f64(True, True, 2.0, A, B, -3.0, C0)
    want = np.array([[2 * sum(int(A[k, i]) * int(B[j, k]) for k in range(9)) - 3 * int(C0[i, j])
                      for j in range(7)] for i in range(6)], dtype=np.float64)
    assert np.array_equal(C64, want)
    assert np.array_equal(T, 3.0 * np.abs(C0))
    # beta = 0 never reads C0 (NaN in C0 must not appear)
    nan_c = np.full((6, 7), np.nan, np.float32)
    C64b, _, Tb = ref_gemm.gemm_general_f64(True, True, 1.0, A, B, 0.0, nan_c)
    assert np.isfinite(C64b).all() and np.all(Tb == 0)
    # no transposes, alpha = 1, beta = 0 is the plain product
    A2, B2 = gen.operands(5, 4, 3, seed=92, integer_copy=True)
    assert np.array_equal(ref_gemm.gemm_general_f64(False, False, 1.0, A2, B2, 0.0, None)[0],
                          ref_gemm.gemm_f64(A2, B2)[0])


def test_general_tolerance_accepts_fp32_and_rejects_a_wrong_beta():
    A, B = gen.operands(6, 6, 9, seed=0)
    C0 = gen.matrix(93, gen.STREAM_A, 6, 6)
    C64, S, T = ref_gemm.gemm_general_f64(False, False, 0.5, A, B, 2.0, C0)
    C32 = (np.float32(0.5) * fp32_sequential(A, B) + np.float32(2.0) * C0).astype(np.float32)
    assert tolerance.max_error_ratio_general(C32, C64, S, T, 9, 0.5) <= 1.0
    wrong = (np.float32(0.5) * fp32_sequential(A, B) + np.float32(1.0) * C0).astype(np.float32)
    assert tolerance.max_error_ratio_general(wrong, C64, S, T, 9, 0.5) > 1.0

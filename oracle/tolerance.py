"""Elementwise acceptance test of an FP32 product against the FP64 oracle
(test infrastructure only).

Bound: ``|C - C64| <= 2 * K * u * S`` with ``u = 2**-24`` (FP32 unit roundoff)
and ``S[i][j] = sum_k |A[i][k]| |B[k][j]|``.  ``K * u * S`` is the classical
worst-case error of a length-K FP32 dot product summed in any order with
round-to-nearest (recursive, blocked or split summation, with or without fused
multiply-add); the factor 2 leaves room for the final rounding of the FP64
value and for split-precision schemes.  When every input is a small integer the
FP32 result is exact in any order, so the test there is equality.
"""

from __future__ import annotations

import numpy as np

U32 = 2.0 ** -24


def bound(S: np.ndarray, K: int) -> np.ndarray:
    return 2.0 * K * U32 * np.asarray(S, dtype=np.float64)


def error_ratio(C: np.ndarray, C64: np.ndarray, S: np.ndarray, K: int) -> np.ndarray:
    """|C - C64| / bound, elementwise; 0 where both the error and the bound are 0,
    and +inf where the error is positive and the bound is 0 (or C is not finite)."""
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - np.asarray(C64, dtype=np.float64))
    b = bound(S, K)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(b > 0, err / np.where(b > 0, b, 1.0), np.where(err > 0, np.inf, 0.0))
    r = np.where(np.isfinite(C), r, np.inf)
    return r


def max_error_ratio(C, C64, S, K) -> float:
    r = error_ratio(C, C64, S, K)
    return float(r.max()) if r.size else 0.0


def within(C, C64, S, K) -> bool:
    return max_error_ratio(C, C64, S, K) <= 1.0


def bound_general(S, T, K, alpha):
    """Bound for C = alpha * op(A) op(B) + beta * C0 computed in FP32:
    the product's 2 K u |alpha| S, plus two more roundings (the scaling by
    alpha and the final addition) of each term: 2 (K + 2) u (|alpha| S + T)."""
    return 2.0 * (K + 2) * U32 * (abs(float(alpha)) * np.asarray(S, np.float64) + np.asarray(T, np.float64))


def max_error_ratio_general(C, C64, S, T, K, alpha) -> float:
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - np.asarray(C64, dtype=np.float64))
    b = bound_general(S, T, K, alpha)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(b > 0, err / np.where(b > 0, b, 1.0), np.where(err > 0, np.inf, 0.0))
    r = np.where(np.isfinite(C), r, np.inf)
    return float(r.max()) if r.size else 0.0

"""ctypes front end of the C oracle in ``ref_gemm.c`` (test infrastructure only).

``gemm_f64(A, B)`` returns the FP64 product and the absolute-value sum
``S[i][j] = sum_k |A[i][k]| |B[k][j]|``; ``gemm_entries`` does the same for a
list of single elements.  Both follow the definition of the output element as
the dot product of row i of A and column j of B ("SGEMM: Shared Memory Tiling
Visualizer", tiled kernel; "Shared Memory Tiling", naive kernel).

The shared object is compiled with the system C compiler (``build()``), never
with the GPU toolchain, and is loaded on first use.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_gemm.c")
_LIB_PATH = os.path.join(_HERE, "libref_gemm.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``ref_gemm.c`` into ``libref_gemm.so`` beside it; return its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_gemm_f64.argtypes = [_i64, _i64, _i64, _fp, _i64, _fp, _i64, _dp, _dp, _i64]
            lib.oracle_gemm_f64.restype = None
            lib.oracle_gemm_entries.argtypes = [_i64, _fp, _i64, _fp, _i64, _i64, _lp, _lp, _dp, _dp]
            lib.oracle_gemm_entries.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = None
            _lib = lib
    return _lib


def _as_f32_rows(x: np.ndarray, name: str):
    """Check a 2-D float32 array with unit column stride; return it and its row stride."""
    x = np.asarray(x)
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if x.shape[1] > 1 and x.strides[1] != 4:
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)
    return x, ld


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def gemm_f64(A: np.ndarray, B: np.ndarray, with_abs: bool = True):
    """Return ``(C64, S)``: the FP64 product of A (M x K) and B (K x N) and, if
    ``with_abs``, the FP64 sum of absolute products (else ``None``)."""
    A, lda = _as_f32_rows(A, "A")
    B, ldb = _as_f32_rows(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    if M and N:
        _load().oracle_gemm_f64(
            M, N, K,
            A.ctypes.data_as(_fp), lda, B.ctypes.data_as(_fp), ldb,
            C.ctypes.data_as(_dp), S.ctypes.data_as(_dp) if with_abs else None, N)
    return C, S


def gemm_entries(A: np.ndarray, B: np.ndarray, rows, cols):
    """FP64 values and absolute sums of the single elements ``(rows[t], cols[t])``."""
    A, lda = _as_f32_rows(A, "A")
    B, ldb = _as_f32_rows(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("element index outside the product")
    out_c = np.empty(r.size, dtype=np.float64)
    out_s = np.empty(r.size, dtype=np.float64)
    if r.size:
        _load().oracle_gemm_entries(
            K, A.ctypes.data_as(_fp), lda, B.ctypes.data_as(_fp), ldb,
            r.size, r.ctypes.data_as(_lp), c.ctypes.data_as(_lp),
            out_c.ctypes.data_as(_dp), out_s.ctypes.data_as(_dp))
    return out_c, out_s


def op(X: np.ndarray, trans: bool) -> np.ndarray:
    """op(X) = X or its transpose (a view, no copy)."""
    return X.T if trans else X


def gemm_general_f64(transa: bool, transb: bool, alpha: float, A: np.ndarray, B: np.ndarray, beta: float,
                     C0: np.ndarray):
    """``alpha * op(A) op(B) + beta * C0`` in FP64 and its error scale.

    The product term is the oracle's FP64 dot product of rows of op(A) with
    columns of op(B) (the same definition as ``gemm_f64``, on transposed
    operands where asked); alpha and beta are applied once per element in
    FP64.  When beta == 0, C0 is not read (its NaNs do not propagate).
    Returns ``(C64, S, T)`` with S = sum |a||b| of the product and
    T = |beta| |C0| (0 where beta == 0).
    """
    opA = np.ascontiguousarray(op(np.asarray(A, np.float32), transa))
    opB = np.ascontiguousarray(op(np.asarray(B, np.float32), transb))
    P, S = gemm_f64(opA, opB)
    C64 = float(alpha) * P
    T = np.zeros_like(C64)
    if beta != 0.0:
        C0d = np.asarray(C0, dtype=np.float64)
        C64 = C64 + float(beta) * C0d
        T = abs(float(beta)) * np.abs(C0d)
    return C64, S, T

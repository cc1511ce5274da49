"""Python binding of libsgemm: FP32 C = A * B on a GB300, through the C interface
declared in include/sgemm.h.

The binding only marshals arguments: every step of the product runs in the
library's CUDA kernels.  There is no CPU or library fallback; if the shared
library is missing or fails to load, ``load()`` raises.

* ``sgemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream=None)`` -- the C entry
  point, with pointers given as integers or CUDA tensors (their ``data_ptr()``)
  and the stream as a ``torch.cuda.Stream``, a raw handle or ``None`` (torch's
  current stream on the current device).  Raises ``SgemmError`` on a non-OK
  status.
* ``matmul(A, B, out=None)`` -- convenience wrapper for 2-D float32 CUDA tensors
  with unit column stride (row-major, possibly with a padded row stride).
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsgemm.so")

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = 1
SGEMM_ERR_ALIAS = 2
SGEMM_ERR_LAUNCH = 3
SGEMM_ERR_DEVICE = 4
SGEMM_ERR_TIMEOUT = 5
SGEMM_ERR_SCRATCH_LIMIT = 6

OP_N = 0
OP_T = 1
ALGO_FFMA = 0
ALGO_3XTF32 = 1

LADDER_NAIVE = 0
LADDER_TILED_16 = 1
LADDER_TILED_32 = 2
LADDER_TILED_32_PADDED = 3
LADDER_REGISTER_2D = 4

#: Every entry point include/sgemm.h declares, with its ctypes signature.
_SIGNATURES = {
    "sgemm_f32": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "sgemm_f32_plan": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong),
                                      ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "sgemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sgemm_version": (ctypes.c_int, []),
    "sgemm_f32_splitk": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p]),
    "sgemm_f32_splitk_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "sgemm_f32_splitk_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "sgemm_f32_3xtf32": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]),
    "sgemm_f32_3xtf32_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "sgemm_f32_streamk": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p]),
    "sgemm_f32_streamk_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "sgemm_f32_splitk_suggest": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_int)]),
    "sgemm_f32_ladder": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "sgemm_gemm": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                  ctypes.c_void_p]),
    "sgemm_gemm_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int]),
    "sgemm_f32_host": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "sgemm_f32_host_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "sgemm_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    # test-only interface (include/sgemm_testing.h)
    "sgemm_test_switches": (ctypes.c_int, [ctypes.c_int, ctypes.c_ulonglong]),
    "sgemm_test_tiny_path": (ctypes.c_int, [ctypes.c_int]),
    "sgemm_f32_plan_model": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong),
                                            ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "sgemm_f32_3xtf32_plan_model": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "sgemm_f32_streamk_plan_model": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.POINTER(ctypes.c_longlong),
                                                    ctypes.POINTER(ctypes.c_size_t)]),
}

_lock = threading.Lock()
_lib = None


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load(path: str | None = None):
    """Load libsgemm.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libsgemm.so not built at {p}: run dense_fp32_matrix_04_gb300.build.build()")
            lib = ctypes.CDLL(p)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().sgemm_status_string(int(status)).decode()


sgemm_status_string = status_string


def sgemm_version() -> int:
    return int(load().sgemm_version())


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != SGEMM_OK:
        raise SgemmError(status, where)


def sgemm_f32(M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int, stream=None) -> None:
    """C = A * B on the GPU (see include/sgemm.h for the full contract)."""
    lib = load()
    st = lib.sgemm_f32(int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C), int(ldc),
                       _stream(stream))
    _check(st, "sgemm_f32")


def sgemm_f32_splitk(M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int, splits: int,
                     workspace, workspace_bytes: int, stream=None) -> None:
    """Split-K C = A * B with a caller-owned device workspace (include/sgemm.h)."""
    lib = load()
    st = lib.sgemm_f32_splitk(int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C), int(ldc),
                              int(splits), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "sgemm_f32_splitk")


def sgemm_f32_splitk_noalloc(M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int, splits: int,
                             stream=None) -> None:
    """Split-K product whose partials live in the library's fixed device
    array, for callers that cannot allocate device memory (include/sgemm.h).
    Calls that overlap on the GPU race on that array."""
    lib = load()
    st = lib.sgemm_f32_splitk_noalloc(int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C),
                                      int(ldc), int(splits), _stream(stream))
    _check(st, "sgemm_f32_splitk_noalloc")


def sgemm_f32_3xtf32(M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int, workspace,
                     workspace_bytes: int, stream=None) -> None:
    """3xTF32 tensor-core product with a caller-owned workspace (include/sgemm.h)."""
    lib = load()
    st = lib.sgemm_f32_3xtf32(int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C), int(ldc),
                              _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "sgemm_f32_3xtf32")


def sgemm_f32_streamk(M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int, workspace,
                      workspace_bytes: int, stream=None) -> None:
    """Stream-K C = A * B with a caller-owned device workspace (include/sgemm.h)."""
    lib = load()
    st = lib.sgemm_f32_streamk(int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C), int(ldc),
                               _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "sgemm_f32_streamk")


def sgemm_f32_streamk_workspace_size(M: int, N: int, K: int) -> int:
    return int(load().sgemm_f32_streamk_workspace_size(int(M), int(N), int(K)))


def matmul_streamk(A, B, out=None, workspace=None, stream=None):
    """Stream-K product of CUDA tensors; allocates the workspace with torch if none is given."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    need = sgemm_f32_streamk_workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need // 4, 4), dtype=torch.float32, device=A.device)
    lda, ldb, ldc = _rows(A, "A"), _rows(B, "B"), _rows(out, "out")
    sgemm_f32_streamk(M, N, K, A, lda, B, ldb, out, ldc, workspace, workspace.numel() * 4, stream)
    return out


def sgemm_f32_3xtf32_workspace_size(M: int, N: int, K: int) -> int:
    return int(load().sgemm_f32_3xtf32_workspace_size(int(M), int(N), int(K)))


def matmul_3xtf32(A, B, out=None, workspace=None, stream=None):
    """3xTF32 product of CUDA tensors; allocates the workspace with torch if none is given."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    need = sgemm_f32_3xtf32_workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need // 4, 4), dtype=torch.float32, device=A.device)
    lda, ldb, ldc = _rows(A, "A"), _rows(B, "B"), _rows(out, "out")
    sgemm_f32_3xtf32(M, N, K, A, lda, B, ldb, out, ldc, workspace, workspace.numel() * 4, stream)
    return out


def sgemm_f32_splitk_workspace_size(M: int, N: int, splits: int) -> int:
    return int(load().sgemm_f32_splitk_workspace_size(int(M), int(N), int(splits)))


def sgemm_f32_plan(M: int, N: int, K: int, aligned: bool = True):
    """(tiles, full_tiles, cluster_size, tile_n): how sgemm_f32 launches an
    M x N x K product on the current device, for operands the TMA can address
    (aligned) or not.  Tiles are 128 x tile_n; tiles past full_tiles are split
    over thread-block clusters of cluster_size blocks (1: no split)."""
    t, f, c, n = ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().sgemm_f32_plan(int(M), int(N), int(K), 1 if aligned else 0, ctypes.byref(t), ctypes.byref(f),
                                 ctypes.byref(c), ctypes.byref(n)), "sgemm_f32_plan")
    return int(t.value), int(f.value), int(c.value), int(n.value)


def sgemm_f32_splitk_suggest(M: int, N: int, K: int) -> int:
    out = ctypes.c_int(0)
    _check(load().sgemm_f32_splitk_suggest(int(M), int(N), int(K), ctypes.byref(out)), "sgemm_f32_splitk_suggest")
    return int(out.value)


def matmul_splitk(A, B, out=None, splits=None, workspace=None, stream=None):
    """Split-K product of CUDA tensors; allocates the workspace with torch if none is given."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if splits is None:
        splits = sgemm_f32_splitk_suggest(M, N, K)
    need = sgemm_f32_splitk_workspace_size(M, N, splits)
    if workspace is None:
        workspace = torch.empty(max(need // 4, 4), dtype=torch.float32, device=A.device)
    lda, ldb, ldc = _rows(A, "A"), _rows(B, "B"), _rows(out, "out")
    sgemm_f32_splitk(M, N, K, A, lda, B, ldb, out, ldc, splits, workspace, workspace.numel() * 4, stream)
    return out


def sgemm_f32_ladder(level: int, M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int,
                     stream=None) -> None:
    """One of the pages' ladder kernels (naive, tiled, register-tiled); see include/sgemm.h."""
    lib = load()
    st = lib.sgemm_f32_ladder(int(level), int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C),
                              int(ldc), _stream(stream))
    _check(st, "sgemm_f32_ladder")


def sgemm_gemm(algo: int, transa: int, transb: int, M: int, N: int, K: int, alpha: float, A, lda: int, B,
               ldb: int, beta: float, C, ldc: int, workspace=None, workspace_bytes: int = 0, stream=None) -> None:
    """C = alpha op(A) op(B) + beta C (row-major, BLAS-style); see include/sgemm.h."""
    lib = load()
    st = lib.sgemm_gemm(int(algo), int(transa), int(transb), int(M), int(N), int(K), float(alpha), _ptr(A), int(lda),
                        _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc), _ptr(workspace), int(workspace_bytes),
                        _stream(stream))
    _check(st, "sgemm_gemm")


def sgemm_gemm_workspace_size(algo: int, transa: int, transb: int, M: int, N: int, K: int) -> int:
    return int(load().sgemm_gemm_workspace_size(int(algo), int(transa), int(transb), int(M), int(N), int(K)))


def sgemm_f32_host(M: int, N: int, K: int, A, lda: int, B, ldb: int, C, ldc: int, panels: int, workspace,
                   workspace_bytes: int, stream, h2d_stream, d2h_stream) -> None:
    """C = A * B with host-memory A, B, C, copies overlapped with the product
    (include/sgemm.h).  Pointers are ints or tensors (pinned CPU tensors for overlap)."""
    lib = load()
    st = lib.sgemm_f32_host(int(M), int(N), int(K), _ptr(A), int(lda), _ptr(B), int(ldb), _ptr(C), int(ldc),
                            int(panels), _ptr(workspace), int(workspace_bytes), _stream(stream), _stream(h2d_stream),
                            _stream(d2h_stream))
    _check(st, "sgemm_f32_host")


def sgemm_f32_host_workspace_size(M: int, N: int, K: int, panels: int) -> int:
    return int(load().sgemm_f32_host_workspace_size(int(M), int(N), int(K), int(panels)))


def sgemm_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().sgemm_device_status(_stream(stream)))


def sgemm_test_switches(flags: int, wait_limit_ns: int = 2_000_000_000) -> None:
    """Test-only switches of the library (include/sgemm_testing.h); they take
    effect only in a process whose environment has SGEMM_TEST_SWITCHES=1."""
    _check(load().sgemm_test_switches(int(flags), int(wait_limit_ns)), "sgemm_test_switches")


PLAN_PATHS = {"tma": 0, "phased": 1, "cp": 2}


def sgemm_test_tiny_path(enable: bool) -> None:
    """Test-only: tiny products take the one-thread-per-output kernel (True,
    the default) or the tiled kernels (False); needs SGEMM_TEST_SWITCHES=1."""
    _check(load().sgemm_test_tiny_path(1 if enable else 0), "sgemm_test_tiny_path")


def sgemm_f32_plan_model(M: int, N: int, K: int, sms: int, path: str = "tma"):
    """Test-only: the plan sgemm_f32_plan reports for kernel path ``path``
    ("tma", "phased" or "cp") on a GPU with ``sms`` SMs (every cluster size
    assumed resident, no test switch), computed without a device."""
    t, f, c, n = ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().sgemm_f32_plan_model(int(M), int(N), int(K), PLAN_PATHS[path], int(sms), ctypes.byref(t),
                                       ctypes.byref(f), ctypes.byref(c), ctypes.byref(n)), "sgemm_f32_plan_model")
    return int(t.value), int(f.value), int(c.value), int(n.value)


def sgemm_f32_3xtf32_plan_model(M: int, N: int, K: int, sms: int):
    """Test-only: (tile width, k-splits) of sgemm_f32_3xtf32 for an M x N x K
    product on a GPU with ``sms`` SMs, computed without a device."""
    w, s = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().sgemm_f32_3xtf32_plan_model(int(M), int(N), int(K), int(sms), ctypes.byref(w), ctypes.byref(s)),
           "sgemm_f32_3xtf32_plan_model")
    return int(w.value), int(s.value)


def sgemm_f32_streamk_plan_model(M: int, N: int, K: int, sms: int, blocks_per_sm: int = 2):
    """Test-only: (stream-K blocks, workspace bytes) of sgemm_f32_streamk for
    an M x N x K product of aligned operands on a GPU with ``sms`` SMs and
    ``blocks_per_sm`` resident blocks per SM; (0, 0) when it runs as
    sgemm_f32.  Computed without a device."""
    b, w = ctypes.c_longlong(0), ctypes.c_size_t(0)
    _check(load().sgemm_f32_streamk_plan_model(int(M), int(N), int(K), int(sms), int(blocks_per_sm), ctypes.byref(b),
                                               ctypes.byref(w)), "sgemm_f32_streamk_plan_model")
    return int(b.value), int(w.value)


def _rows(t, name):
    """Leading dimension of a row-major 2-D float32 CUDA tensor."""
    import torch
    if t.dim() != 2 or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a 2-D float32 CUDA tensor")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def matmul(A, B, out=None, stream=None):
    """Row-major FP32 product of two CUDA tensors via ``sgemm_f32``; returns ``out``."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    lda, ldb, ldc = _rows(A, "A"), _rows(B, "B"), _rows(out, "out")
    if tuple(out.shape) != (M, N):
        raise ValueError("out has the wrong shape")
    sgemm_f32(M, N, K, A, lda, B, ldb, out, ldc, stream)
    return out

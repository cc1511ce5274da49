"""GPU-side test helpers: run the library's sgemm_f32 on device buffers laid out
with arbitrary leading dimensions and base offsets, surrounded by canary
guard bands, and compare with the oracle."""

from __future__ import annotations

import numpy as np

from oracle import ref_gemm, tolerance

CANARY_BITS = np.int32(0x7FC0_1234)   # a quiet NaN with a payload no kernel produces
GUARD = 64                            # guard words before and after each buffer (offset 0 stays 16-byte aligned)
WS_GUARD = 64                         # guard words around a split-K workspace (keeps 16-byte alignment)


def _device_buffer(mat, ld, offset, torch, dev):
    """Place a rows x cols matrix into a flat device buffer: GUARD canaries,
    ``offset`` words, rows of ``ld`` words (gaps hold canaries), GUARD canaries.
    Returns (buffer, element pointer)."""
    rows, cols = mat.shape
    body = max(rows * ld, 1)
    host = np.full(GUARD + offset + body + GUARD, 0, np.int32)
    host[:] = CANARY_BITS
    f = host.view(np.float32)
    start = GUARD + offset
    for r in range(rows):
        f[start + r * ld: start + r * ld + cols] = mat[r]
    buf = torch.from_numpy(host.view(np.float32)).to(dev)
    return buf, buf.data_ptr() + 4 * start


def run_sgemm(sg, A, B, lda=None, ldb=None, ldc=None, a_off=0, b_off=0, c_off=0, stream=None, splits=None):
    """C = A * B through sgemm_f32 (or sgemm_f32_splitk when ``splits`` is given,
    with a canary-guarded workspace); checks that nothing outside the M x N
    block of C (guards and the row gaps between N and ldc) was written."""
    import torch
    dev = torch.device("cuda", 0)
    M, K = A.shape
    N = B.shape[1]
    lda = lda or max(K, 1)
    ldb = ldb or max(N, 1)
    ldc = ldc or max(N, 1)
    a_buf, pa = _device_buffer(A, lda, a_off, torch, dev)
    b_buf, pb = _device_buffer(B, ldb, b_off, torch, dev)
    c_init = np.zeros((M, 0), np.float32)
    c_buf, pc = _device_buffer(c_init, ldc, c_off, torch, dev)
    ws = None
    if splits is None:
        sg.sgemm_f32(M, N, K, pa, lda, pb, ldb, pc, ldc, stream=stream)
    else:
        need = sg.sgemm_f32_splitk_workspace_size(M, N, splits)
        ws = torch.full((need // 4 + 2 * WS_GUARD,), float("nan"), device=dev)
        sg.sgemm_f32_splitk(M, N, K, pa, lda, pb, ldb, pc, ldc, splits, ws.data_ptr() + 4 * WS_GUARD, need, stream)
    torch.cuda.synchronize()
    if ws is not None:
        w = ws.cpu().numpy()
        assert np.isnan(w[:WS_GUARD]).all() and np.isnan(w[-WS_GUARD:]).all(), "split-K wrote outside its workspace"
    host = c_buf.cpu().numpy().view(np.int32)
    start = GUARD + c_off
    C = np.empty((M, N), np.float32)
    touched = np.zeros(host.size, bool)
    for r in range(M):
        seg = host[start + r * ldc: start + r * ldc + N]
        C[r] = seg.view(np.float32)
        touched[start + r * ldc: start + r * ldc + N] = True
    outside = host[~touched]
    assert np.all(outside == CANARY_BITS), "sgemm_f32 wrote outside the M x N block of C"
    del a_buf, b_buf
    return C


def check_full(C, A, B, exact=False):
    """Compare a whole product with the oracle; return the max error/bound ratio."""
    C64, S = ref_gemm.gemm_f64(A, B)
    K = A.shape[1]
    if exact:
        assert np.array_equal(C.astype(np.float64), C64), "integer product is not exact"
        return 0.0
    r = tolerance.max_error_ratio(C, C64, S, K)
    assert r <= 1.0, f"error exceeds 2*K*u*sum|a||b| by a factor {r:.3g}"
    return r


def check_rows(C, A, B, rows):
    """Compare whole rows of a large product with the oracle."""
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    C64, S = ref_gemm.gemm_f64(np.ascontiguousarray(A[rows]), B)
    r = tolerance.max_error_ratio(C[rows], C64, S, A.shape[1])
    assert r <= 1.0, f"sampled rows: error/bound {r:.3g}"
    return r


def check_entries(C, A, B, rows, cols):
    c64, s = ref_gemm.gemm_entries(A, B, rows, cols)
    r = tolerance.max_error_ratio(C[rows, cols], c64, s, A.shape[1])
    assert r <= 1.0, f"sampled entries: error/bound {r:.3g}"
    return r


# Operands and oracle results of the large workloads, kept for the session so
# that the FFMA and 3xTF32 tests of one workload draw and check them once.
_OPERANDS = {}
_ORACLE = {}
CACHE_ORACLE_BELOW = 2 ** 26 + 1   # outputs up to 8192 x 8192 (1 GB of FP64 results) are kept


def workload_operands(name):
    """(A, B) of a named workload, generated once per session."""
    import gen
    if name not in _OPERANDS:
        M, N, K, dist, seed = gen.WORKLOADS[name]
        _OPERANDS[name] = gen.operands(M, N, K, seed=seed, dist=dist)
    return _OPERANDS[name]


def check_full_blocked(C, A, B, key=None, block_rows=512):
    """Compare every element of a large product with the oracle, computed in
    blocks of rows (bounded host memory); return the max error/bound ratio over
    all M x N outputs.  With ``key`` (and an output of at most 2^26 elements)
    the oracle's blocks are kept for the next product of the same inputs."""
    M, K = A.shape
    cache = key is not None and M * B.shape[1] < CACHE_ORACLE_BELOW
    blocks = _ORACLE.get(key) if cache else None
    if blocks is None:
        blocks = (( r0, *ref_gemm.gemm_f64(np.ascontiguousarray(A[r0:r0 + block_rows]), B))
                  for r0 in range(0, M, block_rows))
        if cache:
            blocks = list(blocks)
            _ORACLE[key] = blocks
    worst = 0.0
    for r0, C64, S in blocks:
        r = tolerance.max_error_ratio(C[r0:r0 + C64.shape[0]], C64, S, K)
        assert r <= 1.0, f"rows {r0}..{r0 + C64.shape[0] - 1}: error exceeds 2*K*u*sum|a||b| by {r:.3g}"
        worst = max(worst, r)
    print(f"every one of {M} x {B.shape[1]} outputs checked: max error/bound {worst:.3g}")
    return worst

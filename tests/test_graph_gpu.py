"""The device entry points inside a captured CUDA graph: after one eager call
(which does the per-device set-up: shared-memory limits, the cluster
occupancy query), sgemm_f32 -- on the plain grid, the cluster split alone,
the plain grid followed by a programmatically overlapped cluster split, the
phased TMA kernel (rows only 4-byte aligned), the cp.async-fed kernel (fewer
than four rows of A) and the small-K tile -- sgemm_f32_splitk, sgemm_f32_3xtf32
and sgemm_gemm (both algorithms, A transposed) are captured with
torch.cuda.graph, replayed on new inputs written into the same buffers, and
must equal the eager results bit for bit."""

import numpy as np
import pytest

import gen
from helpers import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg(cuda_device, lib):
    import dense_fp32_matrix_04_gb300 as sg
    return sg


def _pad(n):
    return (n + 3) // 4 * 4


def _buffers(torch, M, N, K, aligned):
    lda, ldb = (_pad(K), _pad(N)) if aligned else (K, N)
    A = torch.zeros(M, lda, device="cuda")[:, :K]
    B = torch.zeros(K, ldb, device="cuda")[:, :N]
    C = torch.full((M, N), float("nan"), device="cuda")
    return A, B, C


@pytest.mark.parametrize("M,N,K,aligned,expect", [
    (8192, 2048, 512, True, "plain"),            # 1024 tiles: no split
    (768, 1024, 2048, True, "split"),            # every tile in clusters
    (1024, 1024, 1024, True, "ksplit"),          # one round of tiles, two warp groups per tile
    (2048, 2048, 2048, True, "plain+split"),     # primary grid + overlapped clusters
    (3001, 4999, 2047, False, "phased"),         # unaligned: phase maps, with a cluster tail
    (3, 2000, 1001, False, "cp.async"),          # unaligned, three rows of A: cp.async-fed
    (4096, 4096, 32, True, "small-k"),
])
def test_sgemm_f32_replays_bitwise(sg, M, N, K, aligned, expect):
    import torch
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K, aligned)
    if expect == "split":
        assert cs > 1 and full == 0
    if expect == "plain+split":
        assert cs > 1 and 0 < full < tiles
    if expect == "ksplit":
        assert (full, cs, tn) == (tiles, 1, 64)
    A, B, C = _buffers(torch, M, N, K, aligned)
    a0, b0 = gen.operands(M, N, K, seed=400)
    A.copy_(torch.from_numpy(a0))
    B.copy_(torch.from_numpy(b0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sg.matmul(A, B, out=C)                     # eager warm-up: per-device set-up happens here
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sg.matmul(A, B, out=C)
    for seed in (401, 402):
        a, b = gen.operands(M, N, K, seed=seed)
        A.copy_(torch.from_numpy(a))
        B.copy_(torch.from_numpy(b))
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = C.clone()
        C.fill_(float("nan"))
        sg.matmul(A, B, out=C)
        torch.cuda.synchronize()
        assert torch.equal(got, C)
    assert sg.sgemm_device_status() == sg.SGEMM_OK


def test_splitk_3xtf32_and_gemm_replay_bitwise(sg):
    import torch
    M, N, K = 768, 640, 3000
    A, B, C = _buffers(torch, M, N, K, True)
    splits = sg.sgemm_f32_splitk_suggest(M, N, K)
    wk = torch.empty(sg.sgemm_f32_splitk_workspace_size(M, N, splits) // 4 + 4, device="cuda")
    w3 = torch.empty(sg.sgemm_f32_3xtf32_workspace_size(M, N, K) // 4 + 4, device="cuda")
    C3 = torch.empty_like(C)

    # sgemm_gemm on both algorithms with A stored transposed (K x M) into its own workspace
    At = torch.zeros(K, M, device="cuda")
    Cg = [torch.zeros(M, N, device="cuda") for _ in range(2)]
    wg = [torch.empty(max(sg.sgemm_gemm_workspace_size(algo, 1, 0, M, N, K) // 4, 4) + 4, device="cuda")
          for algo in (0, 1)]

    def step():
        sg.matmul_splitk(A, B, out=C, splits=splits, workspace=wk)
        sg.matmul_3xtf32(A, B, out=C3, workspace=w3)
        At.copy_(A.t())
        for algo in (0, 1):
            sg.sgemm_gemm(algo, 1, 0, M, N, K, 0.5, At, M, B, B.stride(0), 0.25, Cg[algo], N, wg[algo],
                          wg[algo].numel() * 4)
    a0, b0 = gen.operands(M, N, K, seed=403)
    A.copy_(torch.from_numpy(a0))
    B.copy_(torch.from_numpy(b0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    a, b = gen.operands(M, N, K, seed=404)
    A.copy_(torch.from_numpy(a))
    B.copy_(torch.from_numpy(b))
    prev = Cg[0].clone()                 # C = 0.5 op(A) B + 0.25 C reads C: replay and eager start alike
    Cg[1].copy_(prev)
    g.replay()
    torch.cuda.synchronize()
    got, got3 = C.clone(), C3.clone()
    got_g = [c.clone() for c in Cg]
    for c in Cg:
        c.copy_(prev)
    step()
    torch.cuda.synchronize()
    assert torch.equal(got, C) and torch.equal(got3, C3)
    for algo in (0, 1):
        assert torch.equal(got_g[algo], Cg[algo])
    assert sg.sgemm_device_status() == sg.SGEMM_OK


def test_streamk_replays_bitwise(sg):
    # the stream-K kernel is a cooperative launch after a memset of its tile
    # counters: both are captured, and a replay gives the eager call's bits
    import torch
    M, N, K = 256, 256, 16384
    A, B, C = _buffers(torch, M, N, K, True)
    need = sg.sgemm_f32_streamk_workspace_size(M, N, K)
    assert need > 0
    ws = torch.empty(need // 4, device="cuda")
    a0, b0 = gen.operands(M, N, K, seed=405)
    A.copy_(torch.from_numpy(a0))
    B.copy_(torch.from_numpy(b0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sg.matmul_streamk(A, B, out=C, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sg.matmul_streamk(A, B, out=C, workspace=ws)
    for seed in (406, 407):
        a, b = gen.operands(M, N, K, seed=seed)
        A.copy_(torch.from_numpy(a))
        B.copy_(torch.from_numpy(b))
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = C.clone()
        C.fill_(float("nan"))
        sg.matmul_streamk(A, B, out=C, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got, C)
        check_full(got.cpu().numpy(), a, b)
    assert sg.sgemm_device_status() == sg.SGEMM_OK

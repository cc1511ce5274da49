#!/usr/bin/env python3
"""Benchmark of the FP32 SGEMM path on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload square_8192]

A step is one C = A * B over the whole workload (one sgemm_f32 call, one kernel
launch).  The default workload is the compute-bound square problem
M = N = K = 8192 with A, B ~ N(0, 1) from seed 2.  Inputs are generated on the
host, copied to HBM once, and are larger than L2 (805 MB vs 129 MB), so no L2
flush is needed between steps.

* ``value``: TFLOP/s = 2MNK * steps * ranks / (max over ranks of the device
  time of the K timed steps), inputs resident in HBM.
* ``e2e``: the same metric through the public call with host buffers: each
  step copies A and B from pinned host memory, runs sgemm_f32 and copies C back
  (sgemm_f32_host, copies overlapped with the product); the median of three
  rounds of --e2e-steps calls, every round listed.
* ``roofline``: the kernel is bound by the FP32 FFMA pipes.  Peak =
  SMs x 128 FP32 lanes x 2 FLOP x clock, at the maximum SM clock (2070 MHz)
  and, beside it, at the median clock sampled during the timed region.
* ``cpu_baseline``: the CPU oracle (FP64 triple loop) on a bounded sample of the
  rows of the same product, on this host's cores.
* ``variants``: the same product through sgemm_f32_3xtf32 (tensor cores).
* ``configs``: every other workload (6x6x9, 1024^3, 3001x4999x2047,
  16384^2x32, 16384^3, 256x256x65536), each through sgemm_f32 over about two
  seconds of steps with its own clock samples, roofline, DRAM bytes from its
  committed ncu summary, sampled oracle check and end-to-end figure; with the
  3xTF32 and stream-K entry points beside it where they apply.

Under torchrun (N > 1) each rank runs its own full replica of the product
(one process per GPU, no collective on the data path); ``--impl reference``
runs on rank 0 only.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "SGEMM TFLOP/s (2MNK/t) and % of FP32 roofline at M=N=K=8192"
DEFAULT_WORKLOAD = "square_8192"
# the other workloads, each measured in the line's "configs" block
CONFIG_WORKLOADS = ["tiny_6x6x9", "square_1024", "ragged_3001x4999x2047", "skinny_16384x16384x32", "square_16384",
                    "longk_256x256x65536"]
# configs also timed through sgemm_f32_3xtf32 (the headline's variant is timed beside the headline)
X3_CONFIG_WORKLOADS = ["square_1024", "ragged_3001x4999x2047", "skinny_16384x16384x32"]
FLUSH_BYTES = 256 * 2 ** 20   # twice L2: written between steps of workloads that fit in L2
E2E_ROUNDS = 3                # rounds of the headline's end-to-end timing
L2_BYTES = 129e6
FALLBACK_HBM_GBS = 6800.0
FP32_LANES_PER_SM = 128
MAX_SM_MHZ = 2070.0
KERNEL_SOURCES = ["dense_fp32_matrix_04_gb300/csrc/ffma_tma_sgemm.cuh", "dense_fp32_matrix_04_gb300/csrc/ptx.cuh",
                  "dense_fp32_matrix_04_gb300/csrc/tile_map.cuh"]
TILES = "dense_fp32_matrix_04_gb300/csrc/tiles.cuh"
# workload -> (committed ncu summary with its DRAM bytes, kernel sources the
# capture covers, the tile configuration in TILES it ran)
TRAFFIC_PROFILES = {
    "square_8192": ("ffma_tma_square_8192.md", KERNEL_SOURCES, "TmaMainTile"),
    "ragged_3001x4999x2047": ("ffma_phased_ragged_3001x4999x2047.md",
                              ["dense_fp32_matrix_04_gb300/csrc/ffma_tma_phased.cuh"] + KERNEL_SOURCES, "TmaMainTile"),
    "skinny_16384x16384x32": ("ffma_tma_skinny_16384x16384x32.md",
                              ["dense_fp32_matrix_04_gb300/csrc/ffma_tma_smallk.cuh"] + KERNEL_SOURCES,
                              "TmaSmallKStoreTile"),
    "square_1024": ("ffma_ksplit_square_1024.md", ["dense_fp32_matrix_04_gb300/csrc/ffma_tma_ksplit.cuh"] + KERNEL_SOURCES,
                    "TmaKSplitTile"),
    "square_16384": ("ffma_tma_square_16384.md", KERNEL_SOURCES, "TmaMainTile"),
    "tiny_6x6x9": ("ffma_tiny_6x6x9.md", ["dense_fp32_matrix_04_gb300/csrc/ffma_tiny.cuh",
                                          "dense_fp32_matrix_04_gb300/csrc/epilogue.cuh"], None),
    "longk_256x256x65536": ("ffma_narrow_longk_256x256x65536.md", KERNEL_SOURCES, "TmaNarrowTile"),
}
# the same for sgemm_f32_streamk's kernel, on the workloads that take it
STREAMK_PROFILES = {
    "longk_256x256x65536": ("ffma_tma_streamk_longk_256x256x65536.md",
                            ["dense_fp32_matrix_04_gb300/csrc/ffma_tma_streamk.cuh"] + KERNEL_SOURCES, "TmaMainTile"),
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=150)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gen.WORKLOADS))
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--path", choices=["ffma", "splitk", "streamk", "3xtf32", "gemm"] + sorted(LADDER),
                   default="ffma",
                   help="ffma: sgemm_f32 (the headline); splitk: sgemm_f32_splitk with the suggested split "
                        "count; streamk: sgemm_f32_streamk; 3xtf32: sgemm_f32_3xtf32 (tensor cores). "
                        "Workspaces are allocated untimed.")
    p.add_argument("--no-context", action="store_true",
                   help="skip the torch.matmul (cuBLAS SGEMM) context timing")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the extra 3xTF32 measurement reported beside the headline")
    p.add_argument("--configs", default=",".join(CONFIG_WORKLOADS),
                   help="comma-separated workloads measured beside the headline in the 'configs' block "
                        "('' for none)")
    p.add_argument("--min-seconds", type=float, default=2.0,
                   help="wall time of each config's timed region, and of the sustained load under which the "
                        "headline's clocks are sampled")
    return p.parse_args()


def workload_config(name):
    M, N, K, dist, seed = gen.WORKLOADS[name]
    alg_bytes = 4 * (M * K + K * N + M * N)
    return M, N, K, dist, seed, {
        "workload": f"{name}: C = A*B, M={M} N={N} K={K}, FP32 row-major, A,B ~ "
                    f"{'N(0,1)' if dist == 'normal' else 'uniform[-1,1]'} from seed {seed}",
        "M": M, "N": N, "K": K,
        "l2": (f"inputs larger than L2 ({alg_bytes / 1e6:.0f} MB of A+B+C vs 129 MB); no flush"
               if alg_bytes > 2 * L2_BYTES else
               f"working set {alg_bytes / 1e6:.0f} MB is within 2x L2: a 512 MB buffer is written between "
               "timed steps (outside the per-step events)"),
    }


def metric_name(workload):
    if workload == DEFAULT_WORKLOAD:
        return METRIC
    M, N, K = gen.WORKLOADS[workload][:3]
    return f"SGEMM TFLOP/s (2MNK/t) and % of roofline at M={M} N={N} K={K}"


def measured_hbm_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------- oracle legs

def oracle_rows_sample(A, B, target_s):
    """Time the CPU oracle on the first R rows of the product, R sized to ~target_s."""
    from oracle import ref_gemm
    M, K = A.shape
    N = B.shape[1]
    r = min(M, max(4, 2 * ref_gemm.num_threads()))
    t0 = time.perf_counter()
    ref_gemm.gemm_f64(A[:r], B, with_abs=False)
    dt = max(time.perf_counter() - t0, 1e-4)
    R = int(max(1, min(M, round(r * target_s / dt))))
    t0 = time.perf_counter()
    ref_gemm.gemm_f64(A[:R], B, with_abs=False)
    dt = time.perf_counter() - t0
    return R, dt, ref_gemm.num_threads()


def cpu_baseline(A, B, target_s):
    M, K = A.shape
    N = B.shape[1]
    R, dt, cores = oracle_rows_sample(A, B, target_s)
    tflops = 2.0 * R * N * K / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{R - 1} of C ({R}x{N}x{K}, FP64 accumulation, product only), "
                      f"{dt:.2f} s on {cores} host threads"}


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = (uuid or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 5 and os.path.getsize(self.path) == 0:
                time.sleep(0.05)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1].lower():
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[6:10]):
                if v.lower() == "active":
                    reasons.add(name)
        power = [num(r[4]) for r in rows if num(r[4]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][3]), "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------- ncu traffic

def code_only(text):
    """C++ source without its comments and with runs of whitespace collapsed,
    so that a digest follows the code a capture ran and not its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest(sources=None, tile=None):
    """Digest of the kernel sources' code and, if named, the one line of TILES
    that defines the tile configuration (so other configurations may change)."""
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            h.update(code_only(f.read()).encode())
    if tile:
        with open(os.path.join(ROOT, TILES)) as f:
            lines = [l.strip() for l in f if l.strip().startswith(f"using {tile} =")]
        if len(lines) != 1:
            raise ValueError(f"{tile}: expected one definition in {TILES}")
        h.update(lines[0].encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload=DEFAULT_WORKLOAD, profiles=None):
    """DRAM bytes of one product of the workload from its committed ncu summary
    (sgemm_f32's kernel, or the kernel of the table ``profiles``), if the
    capture was taken on the kernel sources as they are now; else None."""
    profiles = TRAFFIC_PROFILES if profiles is None else profiles
    if workload not in profiles:
        return None
    name, sources, tile = profiles[workload]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    d = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_source_digest(sources, tile):
        return None
    return int(m.group(1))


# ---------------------------------------------------------------------- arms

LADDER = {"ladder-naive": 0, "ladder-tiled16": 1, "ladder-tiled32": 2, "ladder-tiled32p": 3, "ladder-register": 4}


def make_step(sg, path, M, N, K, dA, dB, dC, handle, cfg, dev):
    """One step of the chosen path through the C interface; workspaces are allocated here, untimed."""
    import torch
    if path == "splitk":
        splits = sg.sgemm_f32_splitk_suggest(M, N, K)
        ws_bytes = sg.sgemm_f32_splitk_workspace_size(M, N, splits)
        ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
        cfg["splitk"] = splits

        def step():
            sg.sgemm_f32_splitk(M, N, K, dA, K, dB, N, dC, N, splits, ws, ws_bytes, handle)
        return step, (2 if splits > 1 else f32_launches(sg, M, N, K))
    if path == "gemm":
        # sgemm_gemm, FFMA form, alpha = 1, beta = 0, no transposes: unaligned
        # operands are read in place (phase maps) unless M or K is below 4
        ws_bytes = sg.sgemm_gemm_workspace_size(0, 0, 0, M, N, K)
        ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
        cfg["path"] = "sgemm_gemm (FFMA, alpha = 1, beta = 0, no transposes)"

        def step():
            sg.sgemm_gemm(0, 0, 0, M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, ws, ws_bytes, handle)
        # the same launches as sgemm_f32 (a repacking copy, below four rows, is
        # not a kernel of ours)
        return step, f32_launches(sg, M, N, K)
    if path == "streamk":
        ws_bytes = sg.sgemm_f32_streamk_workspace_size(M, N, K)
        ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
        cfg["path"] = "sgemm_f32_streamk" + ("" if ws_bytes else " (runs as sgemm_f32: its plan fills the SMs)")

        def step():
            sg.sgemm_f32_streamk(M, N, K, dA, K, dB, N, dC, N, ws, ws_bytes, handle)
        # one kernel (and a memset of the tile counters) when stream-K is taken
        return step, (1 if ws_bytes else f32_launches(sg, M, N, K))
    if path in LADDER:
        cfg["path"] = path

        def step():
            sg.sgemm_f32_ladder(LADDER[path], M, N, K, dA, K, dB, N, dC, N, handle)
        return step, 1
    if path == "3xtf32":
        ws_bytes = sg.sgemm_f32_3xtf32_workspace_size(M, N, K)
        ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
        cfg["path"] = "3xtf32"

        def step():
            sg.sgemm_f32_3xtf32(M, N, K, dA, K, dB, N, dC, N, ws, ws_bytes, handle)
        return step, x3_launches(sg, M, N, K)

    def step():
        sg.sgemm_f32(M, N, K, dA, K, dB, N, dC, N, handle)
    return step, f32_launches(sg, M, N, K)


def x3_launches(sg, M, N, K):
    """Kernels one sgemm_f32_3xtf32 call launches: the two split passes and the
    tensor-core product, plus the reduction when the product is divided (its
    workspace then holds partial tiles beyond the split operands)."""
    operands = (4 * ((K + 3) // 4 * 4) * (2 * M + 2 * N) + 255) // 256 * 256
    return 4 if sg.sgemm_f32_3xtf32_workspace_size(M, N, K) > operands else 3


def f32_launches(sg, M, N, K):
    """Kernels one sgemm_f32 call launches: one, or two when a cluster-split
    grid follows whole rounds of plain tiles (sgemm_f32_plan)."""
    if K > 0 and M * N > 0:
        tiles, full, cs, _ = sg.sgemm_f32_plan(M, N, K)
        return 2 if cs > 1 and 0 < full < tiles else 1
    return 1


TF32_PEAK_NOTE = ("DERIVED, not measured: dense TF32 tensor peak = {tsrc}; the tensor-core kernel alone "
                  "reads at or above it, so this peak is low and frac overstates the kernel's use of the "
                  "tensor pipe")
TF32_PROFILES = {"square_8192": "tf32x3_tcgen05_square_8192.md",
                 "ragged_3001x4999x2047": "tf32x3_tcgen05_ragged_3001x4999x2047.md"}
TF32_SOURCES = ["dense_fp32_matrix_04_gb300/csrc/tf32x3_tcgen05.cuh", "dense_fp32_matrix_04_gb300/csrc/tcgen05.cuh",
                "dense_fp32_matrix_04_gb300/csrc/ptx.cuh", "dense_fp32_matrix_04_gb300/csrc/tile_map.cuh",
                "dense_fp32_matrix_04_gb300/csrc/epilogue.cuh"]


def recorded_tensor_pipe(workload):
    """The tensor-pipe busy fraction ncu measured for the 3xTF32 kernel on this
    workload (from its committed summary), or None."""
    try:
        text = open(os.path.join(ROOT, "profiles", TF32_PROFILES[workload])).read()
    except (KeyError, OSError):
        return None
    m = re.search(r"tensor_pipe_active_pct:\s*([0-9.]+)", text)
    d = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_source_digest(TF32_SOURCES):
        return None
    return float(m.group(1)) / 100


def tf32_peak_tflops():
    """Dense TF32 tensor peak: the measured bf16 burst peak x the nominal TF32/bf16 ratio (1.1/2.25)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]) * 1.1 / 2.25, "measured bf16 x nominal 1.1/2.25"
    except (OSError, KeyError, ValueError):
        return 1900.0 * 1.1 / 2.25, "fallback bf16 1.9 PFLOP/s x nominal 1.1/2.25"


def time_steps(step, steps, stream, dev):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1)


STREAMK_KERNEL = ("sgemm_ffma_tma_streamk_kernel (128x128x32 TMA-fed tile, 3 stages, 8x16 per thread as "
                  "fma.rn.f32x2 column pairs; a cooperative grid of two blocks per SM, each an equal run of (tile, "
                  "k-step) units across tile boundaries; partial tiles meet in the caller's workspace and every "
                  "block that shares a tile adds up its own slice of them in a fixed order)")


def kernel_name(sg, M, N, K):
    """The kernel sgemm_f32 launches for a contiguous M x K by K x N product."""
    if K > 0 and sg.sgemm_f32_plan(M, N, K)[3] == 0:
        return ("sgemm_ffma_tiny_kernel (one thread per output, the K-long dot product read straight from "
                "memory; products of at most 16384 outputs with K <= 128)")
    if K > 0 and K % 4 == 0 and N % 4 == 0:
        if K <= 32:
            # the bench's products have beta == 0 and a 16-byte aligned C
            return ("sgemm_ffma_tma_smallk_store_kernel (128x64x32 TMA-fed tile of two warps, 1 stage, 8x16 per "
                    "thread as fma.rn.f32x2 column pairs with the rows walked down and up in turn; the C tile "
                    "staged in shared memory and written by TMA bulk tensor stores)")
        if K <= 64:
            return ("sgemm_ffma_tma_kernel (128x64x32 TMA-fed small-K tile, 1 stage, 8x8 per thread as "
                    "fma.rn.f32x2 column pairs, k-groups unrolled by 8, 4 CTAs/SM)")
        tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K)
        if tn == 64 and cs == 1:
            return (f"sgemm_ffma_tma_ksplit_kernel (one round of {tiles} 128x64x32 TMA-fed tiles, one CTA each of two "
                    "groups of two warps on alternate k-steps, a 4-stage ring, 8x16 per thread as fma.rn.f32x2 "
                    "column pairs; the groups' sums added through shared memory)")
        if tn == 64:
            return ("sgemm_ffma_tma_kernel (128x64x32 TMA-fed narrow tile, 2 stages, 8x8 per thread as "
                    f"fma.rn.f32x2 column pairs, 4 CTAs/SM); all {tiles} tiles split over {cs}-CTA clusters "
                    "(k-steps divided, partial sums added through distributed shared memory)")
        name = ("sgemm_ffma_tma_kernel (128x128x32 TMA-fed tile, 3 stages, 8x16 per thread as fma.rn.f32x2 "
                "column pairs with the rows walked down and up in turn, 2 CTAs/SM)")
        if cs > 1:
            name += (f"; tiles {full}..{tiles - 1} split over {cs}-CTA clusters (k-steps divided, partial sums "
                     "added through distributed shared memory)")
        return name
    tiles, full, cs, tn = sg.sgemm_f32_plan(M, N, K, aligned=False) if K > 0 else (0, 0, 1, 128)
    if M >= 4 and K >= 4:
        # rows only 4-byte aligned: each operand read by TMA through four phase maps
        if tn == 64:
            return ("sgemm_ffma_tma_phased_kernel (128x64x32 narrow tile, A and B each read by TMA through four "
                    "phase maps and realigned in shared memory, 2 stages, 8x8 per thread as fma.rn.f32x2 column "
                    f"pairs, 4 CTAs/SM); all {tiles} tiles split over {cs}-CTA clusters (k-steps divided, partial "
                    "sums added through distributed shared memory)")
        name = ("sgemm_ffma_tma_phased_kernel (128x128x32 tile, A and B each read by TMA through four phase maps "
                "and realigned in shared memory, 3 stages, 8x16 per thread as fma.rn.f32x2 column pairs with the "
                "rows walked down and up in turn, 2 CTAs/SM)")
    elif tn == 64:
        return ("sgemm_ffma_cp_kernel (128x64x32 narrow tile fed by cp.async, 3 stages, 8x8 per thread as "
                f"fma.rn.f32x2 column pairs, 3 CTAs/SM); all {tiles} tiles split over {cs}-CTA clusters (k-steps "
                "divided, partial sums added through distributed shared memory)")
    else:
        name = ("sgemm_ffma_cp_kernel (128x128x32 tile fed by cp.async, 3 stages, 8x16 per thread as fma.rn.f32x2 "
                "column pairs with the rows walked down and up in turn, 2 CTAs/SM)")
    if cs > 1:
        name += (f"; tiles {full}..{tiles - 1} split over {cs}-CTA clusters (k-steps divided, partial sums "
                 "added through distributed shared memory)")
    return name


def alu_peak_tflops(sms, mhz=MAX_SM_MHZ):
    return sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def config_roofline(M, N, K, ms, sms, hbm_gbs, hbm_src, clocks):
    """Roofline of one product: achieved 2MNK/t against min(FP32 ALU peak,
    intensity x HBM bandwidth), the intensity over the algorithmic bytes
    4(MK + KN + MN)."""
    flop = 2.0 * M * N * K
    alg_bytes = 4 * (M * K + K * N + M * N)
    p_alu = alu_peak_tflops(sms)
    p_hbm = flop / alg_bytes * hbm_gbs * 1e9 / 1e12
    achieved = flop / (ms / 1e3) / 1e12
    r = {"bound": "alu" if p_alu <= p_hbm else "hbm", "achieved": achieved, "unit": "TFLOP/s",
         "peak": min(p_alu, p_hbm), "frac": achieved / min(p_alu, p_hbm),
         "peak_basis": (f"min({sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x {MAX_SM_MHZ:.0f} MHz = "
                        f"{p_alu:.2f}, {flop / alg_bytes:.1f} FLOP/B x {hbm_gbs:.0f} GB/s ({hbm_src}) = "
                        f"{p_hbm:.2f}) TFLOP/s"),
         "algorithmic_bytes": alg_bytes, "alu_floor_ms": flop / (p_alu * 1e12) * 1e3,
         "hbm_floor_ms": alg_bytes / (hbm_gbs * 1e9) * 1e3}
    if clocks.get("sm_mhz") and r["bound"] == "alu":
        r["frac_at_sampled_clock"] = achieved / alu_peak_tflops(sms, clocks["sm_mhz"])
    return r


def timed_steps(step, stream, dev, flush_buf, min_s, max_steps=200000):
    """Run ``step`` for about ``min_s`` seconds of wall time; return (steps, device ms per step).
    With ``flush_buf`` every step is timed between its own events, after a
    write of the buffer (twice L2) outside them; otherwise the steps run back
    to back between two events."""
    import torch

    # probe the wall cost of one step (with its flush) to size the region: the
    # second of two rounds, after one-time costs have settled
    def probe(k):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(k):
            if flush_buf is not None:
                flush_buf.fill_(1)
            step()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / k
    per = probe(5)
    per = probe(int(min(200, max(5, 0.1 / max(per, 1e-6)))))
    n = int(min(max_steps, max(5, -(-min_s // max(per, 1e-6)))))
    if flush_buf is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return n, e0.elapsed_time(e1) / n
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        flush_buf.fill_(1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return n, sum(a.elapsed_time(b) for a, b in evs) / n


def measure_config(sg, name, dev, stream, sms, props, min_s, flush_buf):
    """One entry of the "configs" block: the workload through sgemm_f32 with
    its inputs resident in HBM (device time over a timed region of about
    ``min_s`` seconds, clocks sampled during it), its roofline, a check of
    sampled rows against the oracle, and the same product end to end through
    sgemm_f32_host with host buffers."""
    import numpy as np
    import torch

    from oracle import ref_gemm, tolerance
    M, N, K, dist_name, seed, cfg = workload_config(name)
    A, B = gen.operands(M, N, K, seed=seed, dist=dist_name)
    dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    handle = stream.cuda_stream
    step, launches = make_step(sg, "ffma", M, N, K, dA, dB, dC, handle, cfg, dev)
    alg_bytes = 4 * (M * K + K * N + M * N)
    flush = flush_buf if alg_bytes <= 2 * L2_BYTES and name != "tiny_6x6x9" else None
    for _ in range(3):
        step()
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    steps, ms = timed_steps(step, stream, dev, flush, min_s)
    clocks = sampler.stop()
    hbm_gbs, hbm_src = measured_hbm_gbs()
    entry = {"workload": cfg["workload"], "M": M, "N": N, "K": K, "path": "sgemm_f32",
             "kernel": kernel_name(sg, M, N, K), "steps": steps, "ms_per_step": ms,
             "value": 2.0 * M * N * K / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
             "l2": ("each step between its own events after a 256 MB buffer write (outside them)" if flush is not None
                    else "back-to-back calls (launch-latency bound; 576 bytes of operands)" if name == "tiny_6x6x9"
                    else "inputs larger than L2; no flush"),
             "roofline": config_roofline(M, N, K, ms, sms, hbm_gbs, hbm_src, clocks),
             "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
             "gpu_launches": steps * launches}
    entry["roofline"]["traffic"] = recorded_traffic(name)
    # products with fewer tiles than resident blocks: the stream-K entry point too
    sk_bytes = sg.sgemm_f32_streamk_workspace_size(M, N, K)
    if sk_bytes > 0:
        sk_ws = torch.empty(sk_bytes // 4, dtype=torch.float32, device=dev)

        def sk_step():
            sg.sgemm_f32_streamk(M, N, K, dA, K, dB, N, dC, N, sk_ws, sk_bytes, handle)
        for _ in range(3):
            sk_step()
        sampler = ClockSampler(str(getattr(props, "uuid", "")))
        sampler.start()
        sk_n, sk_ms = timed_steps(sk_step, stream, dev, flush, min_s)
        sk_clocks = sampler.stop()
        sk_roof = config_roofline(M, N, K, sk_ms, sms, hbm_gbs, hbm_src, sk_clocks)
        sk_roof["traffic"] = recorded_traffic(name, STREAMK_PROFILES)
        entry["variants"] = [{
            "path": "sgemm_f32_streamk (equal runs of (tile, k-step) units per resident block; caller workspace "
                    f"of {sk_bytes / 2 ** 20:.1f} MiB, allocated untimed)",
            "kernel": STREAMK_KERNEL,
            "steps": sk_n, "ms_per_step": sk_ms, "value": 2.0 * M * N * K / (sk_ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "roofline": sk_roof,
            "clocks": {k: sk_clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
            "gpu_launches": sk_n, "memsets": sk_n}]
    if name in X3_CONFIG_WORKLOADS:
        # the same product on the tensor cores (sgemm_f32_3xtf32, caller workspace allocated untimed)
        x3_bytes = sg.sgemm_f32_3xtf32_workspace_size(M, N, K)
        x3_ws = torch.empty(max(x3_bytes // 4, 4), dtype=torch.float32, device=dev)

        def x3_step():
            sg.sgemm_f32_3xtf32(M, N, K, dA, K, dB, N, dC, N, x3_ws, x3_bytes, handle)
        for _ in range(3):
            x3_step()
        sampler = ClockSampler(str(getattr(props, "uuid", "")))
        sampler.start()
        x3_n, x3_ms = timed_steps(x3_step, stream, dev, flush, min_s)
        x3_clocks = sampler.stop()
        tpk, tsrc = tf32_peak_tflops()
        x3_tf = 2.0 * M * N * K / (x3_ms / 1e3) / 1e12
        width, parts = sg.sgemm_f32_3xtf32_plan_model(M, N, K, sms)
        entry.setdefault("variants", []).append({
            "path": f"sgemm_f32_3xtf32 (tensor cores, 3xTF32 split precision; 128x{width} tiles"
                    + (f", {parts} k-parts" if parts > 1 else "") + ")",
            "steps": x3_n, "ms_per_step": x3_ms, "value": x3_tf, "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": 3 * x3_tf, "peak": tpk, "unit": "TFLOP/s",
                         "frac": 3 * x3_tf / tpk, "peak_basis": TF32_PEAK_NOTE.format(tsrc=tsrc),
                         "tensor_pipe_active_ncu": recorded_tensor_pipe(name),
                         "note": "3 TF32 products per FP32 product over the whole step (operand splitting "
                                 "included); tensor_pipe_active_ncu is the hardware counter's fraction"},
            "clocks": {k: x3_clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
            "gpu_launches": 2 * x3_n + (x3_n if parts > 1 else 0)})
        step()  # the oracle check below reads sgemm_f32's output
        torch.cuda.synchronize(dev)
        del x3_ws
    if name == "square_16384":
        # context, not this library: cuBLAS SGEMM (torch.matmul, TF32 off) on the same inputs
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False

        def cublas_step():
            torch.matmul(dA, dB, out=dC)
        for _ in range(2):
            cublas_step()
        c_steps, c_ms = timed_steps(cublas_step, stream, dev, None, min(min_s, 1.0))
        torch.backends.cuda.matmul.allow_tf32 = prev
        entry["context"] = {"what": "torch.matmul with TF32 off (cuBLAS SGEMM); context only, not this library",
                            "value": 2.0 * M * N * K / (c_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                            "ms_per_step": c_ms, "steps": c_steps}
        step()  # the oracle check below reads this library's output
        torch.cuda.synchronize(dev)
    if name == "tiny_6x6x9":
        entry["us_per_call"] = ms * 1e3
        entry["roofline"]["note"] = "launch-latency bound: 648 FLOP per call"
    # the oracle on sampled rows of the timed output
    rows = sorted({0, M // 2, M - 1} | ({127, 128} if M > 128 else set()))
    C64, S = ref_gemm.gemm_f64(np.ascontiguousarray(A[rows]), B)
    entry["check"] = {"rows": rows, "max_error_over_bound": tolerance.max_error_ratio(dC[rows].cpu().numpy(), C64,
                                                                                       S, K)}
    # end to end: host buffers in, host buffer out, every copy inside the timed region
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    panels = 1 if M * N < 2 ** 20 else 8
    ws_bytes = sg.sgemm_f32_host_workspace_size(M, N, K, panels)
    ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_step():
        sg.sgemm_f32_host(M, N, K, hA, K, hB, N, hC, N, panels, ws, ws_bytes, handle, s_in, s_out)
    for _ in range(2):
        e2e_step()
    e_steps, e_ms = timed_steps(e2e_step, stream, dev, None, min(min_s, 1.0), max_steps=20000)
    entry["e2e"] = {"value": 2.0 * M * N * K / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e_ms,
                    "steps": e_steps, "h2d_bytes_per_step": int(hA.numel() * 4 + hB.numel() * 4),
                    "d2h_bytes_per_step": int(hC.numel() * 4),
                    "call": f"sgemm_f32_host, {panels} row panel(s) requested, copies overlapped with the product"}
    return entry


def max_over_ranks(value, world, device):
    """The largest ``value`` over all ranks (the slowest rank's time); identity for one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_step, steps, world, t_ms):
    """Whole-job throughput: every rank runs ``steps`` full products in ``t_ms`` (the max over ranks)."""
    return flop_per_step * steps * world / (t_ms / 1e3) / 1e12


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    M, N, K, dist, seed, cfg = workload_config(args.workload)
    A, B = gen.operands(M, N, K, seed=seed, dist=dist)
    from oracle import ref_gemm
    # size each step so that warm-up + timed steps take about 90 s in total
    R, dt, cores = oracle_rows_sample(A, B, 90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        ref_gemm.gemm_f64(A[:R], B, with_abs=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ref_gemm.gemm_f64(A[:R], B, with_abs=False)
    t = time.perf_counter() - t0
    value = 2.0 * R * N * K * args.steps / t / 1e12
    sample = f"each step: rows 0..{R - 1} of C ({R}x{N}x{K}), FP64 accumulation, product only"
    line = {
        "impl": "reference", "metric": metric_name(args.workload), "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "note": "the CPU oracle (plain FP64 triple loop, OpenMP over rows) on the host cores; "
                "the pages publish no implementation or measured number to run instead",
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import dense_fp32_matrix_04_gb300 as sg
    from dense_fp32_matrix_04_gb300 import build as sgbuild

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if rank == 0:
        sgbuild.build()
    if world > 1:
        dist.barrier()
    sg.load()

    M, N, K, dist_name, seed, cfg = workload_config(args.workload)
    if world > 1:
        cfg["parallelism"] = f"replicas x{world} (one full product per GPU, no collective)"
    t0 = time.time()
    A, B = gen.operands(M, N, K, seed=seed, dist=dist_name)
    log(f"[bench] inputs {M}x{K}, {K}x{N} generated in {time.time() - t0:.1f} s")
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream

    step, launches_per_step = make_step(sg, args.path, M, N, K, dA, dB, dC, handle, cfg, dev)

    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    sampler = ClockSampler(str(getattr(props, "uuid", "")))

    alg_bytes = 4 * (M * K + K * N + M * N)
    flush = alg_bytes <= 2 * L2_BYTES
    flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev) if flush else None

    torch.cuda.synchronize(dev)
    tw = time.perf_counter()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    per_step_s = (time.perf_counter() - tw) / max(1, args.warmup)
    # the clock record spans a sustained load of about --min-seconds: the same
    # product, untimed, right before the timed steps, with the sampler running
    # through both (the timed region alone may be too short for 200 ms samples)
    soak = int(max(0, -(-(args.min_seconds - per_step_s * args.steps) // max(per_step_s, 1e-6))))
    soak = min(soak, 100000)
    sampler.start()
    for i in range(soak):
        step()
        if i % 64 == 63:
            torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if not flush:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        t_ms = ev0.elapsed_time(ev1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e0, e1 in evs:
            flush_buf.fill_(1)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        t_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    clocks["window"] = (f"{soak} untimed steps of the same product right before the {args.steps} timed steps, "
                        "sampled every 200 ms through both")
    t_ms = max_over_ranks(t_ms, world, dev)

    flop = 2.0 * M * N * K
    value = job_tflops(flop, args.steps, world, t_ms)
    per_launch_s = t_ms / args.steps / 1e3
    peak_alu = sms * FP32_LANES_PER_SM * 2 * MAX_SM_MHZ * 1e6 / 1e12
    hbm_gbs, hbm_src = measured_hbm_gbs()
    t_alu = flop / (peak_alu * 1e12)
    t_hbm = alg_bytes / (hbm_gbs * 1e9)
    if t_alu >= t_hbm:
        roofline = {"bound": "alu", "achieved": flop / per_launch_s / 1e12, "peak": peak_alu, "unit": "TFLOP/s",
                    "peak_basis": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x {MAX_SM_MHZ:.0f} MHz "
                                  "(max SM clock)"}
    else:
        roofline = {"bound": "hbm", "achieved": alg_bytes / per_launch_s / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                    "peak_basis": f"copy bandwidth, {hbm_src}"}
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    roofline["traffic"] = recorded_traffic(args.workload) if args.path == "ffma" else None
    roofline["algorithmic_bytes"] = alg_bytes
    roofline["alu_floor_ms"] = t_alu * 1e3
    roofline["hbm_floor_ms"] = t_hbm * 1e3
    roofline["kernel"] = kernel_name(sg, M, N, K) + (f" + split-K x{cfg['splitk']} with reduction"
                                                 if cfg.get("splitk", 1) > 1 else "")
    if args.path in LADDER:
        roofline["kernel"] = f"{args.path} (the pages' kernel ladder)"
    if args.path == "streamk" and sg.sgemm_f32_streamk_workspace_size(M, N, K) > 0:
        roofline["kernel"] = STREAMK_KERNEL
        roofline["traffic"] = recorded_traffic(args.workload, STREAMK_PROFILES)
    if args.path == "3xtf32":
        tpk, tsrc = tf32_peak_tflops()
        roofline = {"bound": "tensor", "achieved": 3 * flop / per_launch_s / 1e12, "peak": tpk, "unit": "TFLOP/s",
                    "peak_basis": TF32_PEAK_NOTE.format(tsrc=tsrc), "traffic": None,
                    "tensor_pipe_active_ncu": recorded_tensor_pipe(args.workload),
                    "algorithmic_bytes": alg_bytes,
                    "kernel": "split kernels + sgemm_3xtf32_kernel (tcgen05 kind::tf32, persistent, one CTA per "
                              "SM, 128x208 tiles (192..128 where they fill the last round better), 5-stage TMA ring, "
                              "two TMEM accumulators, 3 MMAs per k-slice); achieved counts the 3 TF32 products per "
                              "FP32 product over the whole step, split passes included"}
        roofline["frac"] = roofline["achieved"] / tpk
    if clocks.get("sm_mhz") and roofline["bound"] == "alu":
        p = sms * FP32_LANES_PER_SM * 2 * clocks["sm_mhz"] * 1e6 / 1e12
        roofline["peak_at_sampled_clock"] = p
        roofline["frac_at_sampled_clock"] = roofline["achieved"] / p

    # sampled parity check of the timed output (first and last rows)
    check = None
    if rank == 0:
        from oracle import ref_gemm, tolerance
        rows = [0, M - 1]
        C_rows = dC[rows].cpu().numpy()
        C64, S = ref_gemm.gemm_f64(np.ascontiguousarray(A[rows]), B)
        check = {"rows": rows, "max_error_over_bound": tolerance.max_error_ratio(C_rows, C64, S, K)}

    variants = []
    if args.path == "ffma" and not args.no_variants and K > 0:
        vstep, vl = make_step(sg, "3xtf32", M, N, K, dA, dB, dC, handle, {}, dev)
        for _ in range(3):
            vstep()
        vsteps = max(5, args.steps // 2)
        vt = max_over_ranks(time_steps(vstep, vsteps, stream, dev), world, dev)
        tpk, tsrc = tf32_peak_tflops()
        vval = job_tflops(flop, vsteps, world, vt)
        variants.append({"path": "sgemm_f32_3xtf32 (tensor cores, 3xTF32 split precision)", "value": vval,
                         "unit": "TFLOP/s", "ms_per_step": vt / vsteps, "steps": vsteps, "gpu_launches": vsteps * vl,
                         "roofline": {"bound": "tensor", "achieved": 3 * vval / world, "peak": tpk,
                                      "unit": "TFLOP/s", "frac": 3 * vval / world / tpk,
                                      "peak_basis": TF32_PEAK_NOTE.format(tsrc=tsrc),
                                      "tensor_pipe_active_ncu": recorded_tensor_pipe(args.workload),
                                      "note": "3 TF32 products per FP32 product over the whole step (operand "
                                              "splitting included); the hardware's own tensor-pipe counter "
                                              "(tensor_pipe_active_ncu) is the measured fraction"}})

    # context, not this library: cuBLAS SGEMM through torch.matmul with TF32 off,
    # on the same inputs, timed the same way (outside the timed region)
    context = None
    if args.path == "ffma" and not args.no_context and K > 0:
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        dC2 = torch.empty((M, N), dtype=torch.float32, device=dev)

        def cublas_step():
            torch.matmul(dA, dB, out=dC2)
        for _ in range(3):
            cublas_step()
        csteps = max(5, args.steps // 2)
        ct = max_over_ranks(time_steps(cublas_step, csteps, stream, dev), world, dev)
        torch.backends.cuda.matmul.allow_tf32 = prev
        context = {"what": "torch.matmul with TF32 off (cuBLAS SGEMM); context only, not this library",
                   "value": job_tflops(flop, csteps, world, ct), "unit": "TFLOP/s", "ms_per_step": ct / csteps,
                   "steps": csteps, "l2_flushed_between_steps": False}
        del dC2

    # end to end through the public host-buffer call: sgemm_f32_host copies A and B
    # from pinned host memory and C back, overlapped with the product over row
    # panels; every copy is inside the timed region
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    panels = 8  # a hint: the library rounds panels up to whole waves of tiles
    h_ws_bytes = sg.sgemm_f32_host_workspace_size(M, N, K, panels)
    h_ws = torch.empty(max(h_ws_bytes // 4, 4), dtype=torch.float32, device=dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    if args.path == "ffma":
        def e2e_step():
            sg.sgemm_f32_host(M, N, K, hA, K, hB, N, hC, N, panels, h_ws, h_ws_bytes, handle, s_in, s_out)
    else:
        def e2e_step():
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            step()
            hC.copy_(dC, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    # E2E_ROUNDS rounds of --e2e-steps calls each; the value is the median
    # round: the host-memory copies of one 10-call round at 8192^3 were seen
    # to range from 46 to 63 TFLOP/s on the same buffers, round to round
    rounds = []
    for _ in range(E2E_ROUNDS):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        rounds.append(max_over_ranks(e0.elapsed_time(e1), world, dev))
    te_ms = sorted(rounds)[len(rounds) // 2]
    e2e = {"value": job_tflops(flop, args.e2e_steps, world, te_ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(hA.numel() * 4 + hB.numel() * 4),
           "d2h_bytes_per_step": int(hC.numel() * 4), "steps": args.e2e_steps,
           "rounds": len(rounds), "round_values": [job_tflops(flop, args.e2e_steps, world, t) for t in rounds],
           "statistic": "median round (every copy of every round inside its events)",
           "call": (f"sgemm_f32_host, {panels} row panels, copies overlapped with the product"
                    if args.path == "ffma" else "host copies around the device call, serial")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(A, B, args.cpu_seconds)

    # every other workload, each through sgemm_f32 over its own timed region
    configs = {}
    names = [c for c in args.configs.split(",") if c] if args.path == "ffma" and world == 1 else []
    if names:
        del hA, hB, hC, h_ws
        flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        for name in names:
            t0 = time.time()
            configs[name] = measure_config(sg, name, dev, stream, sms, props, args.min_seconds, flush_buf)
            log(f"[bench] config {name}: {configs[name]['value']:.2f} TFLOP/s "
                f"({configs[name]['roofline']['frac']:.3f} of roofline) in {time.time() - t0:.1f} s")
        del flush_buf

    if rank == 0:
        line = {
            "metric": metric_name(args.workload), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": cfg, "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples",
                                                                "power_w_max", "window")},
            "roofline": roofline, "e2e": e2e, "gpu_launches": args.steps * launches_per_step, "cpu_baseline": cpu,
            "check": check, "device": props.name, "sms": sms, "variants": variants, "context": context,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

"""The benchmark's CPU-side pieces: the reference arm (the CPU oracle) prints
one JSON line with the contract's keys; the workload and roofline helpers."""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_6x6x9",
                          "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny_6x6x9")


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_6x6x9",
                          "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                         env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_workload_config_and_metric_names():
    M, N, K, dist, seed, cfg = bench.workload_config("square_8192")
    assert (M, N, K, dist, seed) == (8192, 8192, 8192, "normal", 2)
    assert "no flush" in cfg["l2"]
    assert bench.metric_name("square_8192") == bench.METRIC
    assert "M=1024" in bench.metric_name("square_1024")
    assert "512 MB buffer is written between timed steps" in bench.workload_config("square_1024")[5]["l2"]


def test_recorded_traffic_follows_the_kernel_sources():
    # each committed ncu summary carries the digest of the kernel headers it was taken on
    t = bench.recorded_traffic()
    assert t is None or t > 805_306_368       # at least the algorithmic bytes when present
    # the ragged product's 125.5 MB fit in L2: ncu (which empties the caches
    # before a captured launch) sees A and B come from DRAM, but part of C may
    # still sit in L2 when the launch ends, so only the operand reads bound it
    r = bench.recorded_traffic("ragged_3001x4999x2047")
    assert r is None or r > 4 * (3001 * 2047 + 2047 * 4999)
    # 6x6x9 moves 576 algorithmic bytes; its capture reads a few kB (a cold launch)
    t0 = bench.recorded_traffic("tiny_6x6x9")
    assert t0 is None or t0 < 1_000_000
    assert bench.recorded_traffic("no_such_workload") is None
    assert len(bench.kernel_source_digest()) == 16
    for name, sources, tile in list(bench.TRAFFIC_PROFILES.values()) + list(bench.STREAMK_PROFILES.values()):
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", name))
        assert len(bench.kernel_source_digest(sources, tile)) == 16
    # the stream-K kernel's profile is looked up in its own table: at least A and B come from DRAM
    sk = bench.recorded_traffic("longk_256x256x65536", bench.STREAMK_PROFILES)
    assert sk is None or sk > 4 * 2 * 256 * 65536
    lk = bench.recorded_traffic("longk_256x256x65536")
    assert lk is None or lk > 4 * 2 * 256 * 65536
    # comments do not enter the digest; code does
    assert bench.code_only("int a; // x\n/* y\n z */ int  b;") == bench.code_only("int a;\nint b; // other")
    assert bench.code_only("int a;") != bench.code_only("int b;")
    # the digest names one tile configuration: another one's line does not enter it
    d_main = bench.kernel_source_digest(bench.KERNEL_SOURCES, "TmaMainTile")
    assert d_main != bench.kernel_source_digest(bench.KERNEL_SOURCES, "TmaNarrowTile")
    assert d_main != bench.kernel_source_digest(bench.KERNEL_SOURCES)


def test_tf32_peak_derivation():
    peak, basis = bench.tf32_peak_tflops()
    assert 400 < peak < 1200 and "1.1/2.25" in basis


def test_config_roofline_takes_the_lower_ceiling():
    # 16384 x 16384 x 32: 15.9 FLOP/B x 6681.5 GB/s = 106.5 TFLOP/s is above the
    # 152-SM FP32 peak of 80.55, so the FP32 pipes bound it
    r = bench.config_roofline(16384, 16384, 32, 0.3, 152, 6681.5, "measured", {"sm_mhz": 2070.0})
    assert r["bound"] == "alu" and abs(r["peak"] - 80.548) < 0.01
    assert abs(r["achieved"] - 2 * 16384 * 16384 * 32 / 0.3e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    assert abs(r["frac_at_sampled_clock"] - r["frac"]) < 1e-12
    # a product of intensity 1.1 FLOP/B is bound by HBM bandwidth
    r = bench.config_roofline(6, 6, 9, 0.004, 152, 6681.5, "measured", {})
    assert r["bound"] == "hbm" and r["peak"] < 80
    assert r["algorithmic_bytes"] == 4 * (6 * 9 + 9 * 6 + 6 * 6)


def test_every_bench_config_is_a_known_workload():
    import gen
    assert set(bench.CONFIG_WORKLOADS) <= set(gen.WORKLOADS)
    assert bench.DEFAULT_WORKLOAD not in bench.CONFIG_WORKLOADS
    assert set(bench.CONFIG_WORKLOADS) | {bench.DEFAULT_WORKLOAD} == set(gen.WORKLOADS)

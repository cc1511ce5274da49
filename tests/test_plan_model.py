"""The launch planner's fitted cost models, checked on the CPU against the
plans measured fastest on a GB300 (152 SMs).

sgemm_f32 chooses, per product, between a plain grid of 128 x 128 tiles, the
same grid with its last partial round of tiles split over thread-block
clusters, and (with fewer main tiles than SMs) narrow 128 x 64 tiles in
clusters.  The choice comes from cost models fitted to timings; the tables
below are those timings (TFLOP/s, CUDA events, medians) and the test asks the
device-free planner (sgemm_f32_plan_model) for each shape.  The rule: the
planner picks the plan measured fastest, or one measured within 2 % of it
(the spread between repeated runs of the same plan on these shapes).
"""

import pytest

import dense_fp32_matrix_04_gb300 as sg
from dense_fp32_matrix_04_gb300 import build

SMS = 152
NEAR = 0.02


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    sg.load()


# The 128 x 128 tile (TMA path) with the cluster split of its last partial
# round of tiles: shape -> (full tiles, cluster size) of the faster plan, with
# the measured rates of the plain grid and of that split.
SPLIT_MEASURED = [
    # M, N, K, (full, cs) measured fastest, plain TF/s, split TF/s
    (2048, 2048, 2048, (152, 4), 51.8, 58.1),
    (2560, 2560, 4096, (304, 4), 56.1, 61.3),
    (3008, 5008, 2048, (912, 8), 56.2, 61.0),
    (4955, 1020, 1024, (304, 8), 42.0, 58.0),
    (6144, 6144, 6144, (2280, 8), 62.9, 65.1),
]

# Shapes whose split measured within 0.3 % of the plain grid: the plain grid
# (no split) is the plan.
NO_SPLIT = [(8192, 8192, 8192), (4096, 4096, 4096), (3072, 3072, 3072), (5120, 5120, 5120), (7168, 7168, 7168),
            (896, 8192, 8192)]

# Fewer main tiles than SMs: the 128 x 128 plan against the narrow-tile plan
# (TFLOP/s), TMA operands and operands read by the cp.async kernel
# (lda = K + 1, ldb = N + 1).
NARROW_TMA = [
    (512, 512, 512, 11.1, 15.7),
    (512, 512, 4096, 22.5, 39.1),
    (768, 768, 768, 29.6, 31.8),
    (1024, 1024, 1024, 38.1, 40.0),
    (1024, 1024, 8192, 50.1, 50.7),
    (1280, 1280, 1280, 44.8, 45.4),
    (1536, 1536, 1536, 52.8, 52.0),
    (2048, 1024, 2048, 47.7, 54.5),
    (1000, 2000, 4096, 46.7, 54.7),
    (640, 640, 8192, 37.6, 48.8),
]
NARROW_CP = [
    (512, 512, 512, 7.5, 14.1),
    (512, 512, 4096, 19.1, 31.6),
    (768, 768, 768, 20.7, 27.0),
    (1024, 1024, 1024, 33.1, 33.6),
    (1536, 1536, 1536, 35.4, 42.6),
    (2048, 1024, 2048, 32.6, 44.7),
    (1000, 2000, 4096, 31.5, 45.2),
    (640, 640, 8192, 30.7, 39.4),
]


def tiles128(M, N):
    return -(-M // 128) * -(-N // 128)


@pytest.mark.parametrize("M,N,K,best,plain,split", SPLIT_MEASURED)
def test_cluster_split_plan_is_the_measured_fastest(M, N, K, best, plain, split):
    tiles, full, cs, tile_n = sg.sgemm_f32_plan_model(M, N, K, SMS, "tma")
    assert split > plain
    assert (tiles, tile_n) == (tiles128(M, N), 128)
    assert (full, cs) == best


@pytest.mark.parametrize("M,N,K", NO_SPLIT)
def test_no_split_where_it_does_not_pay(M, N, K):
    assert sg.sgemm_f32_plan_model(M, N, K, SMS, "tma") == (tiles128(M, N), tiles128(M, N), 1, 128)


@pytest.mark.parametrize("path,row", [("tma", r) for r in NARROW_TMA] + [("cp", r) for r in NARROW_CP])
def test_narrow_tile_choice_matches_the_measurements(path, row):
    M, N, K, wide, narrow = row
    assert tiles128(M, N) < SMS
    tiles, full, cs, tile_n = sg.sgemm_f32_plan_model(M, N, K, SMS, path)
    if (tile_n, cs, full) == (64, 1, tiles):
        # the k-split tile, checked against its own measurements below
        assert path == "tma" and (M, N, K) in {r[:3] for r in KSPLIT_MEASURED}
        return
    picked = narrow if tile_n == 64 else wide
    assert picked >= (1 - NEAR) * max(wide, narrow), (
        f"{M}x{N}x{K} on {path}: planned {'narrow' if tile_n == 64 else '128x128'} ({picked} TF/s) "
        f"against {max(wide, narrow)} TF/s measured for the other plan")
    if tile_n == 64:
        # the narrow tile always runs as clusters that split each tile's k-steps
        assert full == 0 and cs in (2, 4, 8) and tiles == -(-M // 128) * -(-N // 64)


# One round of 128 x 64 tiles: the narrow tile's cluster plan against the
# k-split tile (one CTA per tile, two warp groups on the two halves of every
# k-step), us per product (CUDA events, mean of 400 calls after an L2 flush),
# and whether the k-split tile is the plan (at least 70 % of the SMs filled,
# at most 48 k-steps).
KSPLIT_MEASURED = [
    # M, N, K, cluster plan us, k-split us, taken
    (1024, 1024, 512, 33.8, 30.7, True),
    (1024, 1024, 1024, 54.0, 52.8, True),
    (1024, 1024, 1536, 76.0, 75.3, True),
    (1024, 1216, 1024, 64.3, 52.8, True),
    (896, 1024, 1024, 53.9, 52.7, True),
    (800, 1024, 1024, 53.9, 52.8, True),
    (1000, 1000, 1000, 54.1, 52.9, True),
    (1152, 1024, 1024, 55.1, 52.8, True),
    (960, 960, 960, 54.1, 49.6, True),
    (1280, 960, 1024, 64.3, 52.9, True),
    (1024, 1024, 2048, 95.5, 97.7, False),
    (1024, 1152, 2048, 96.3, 97.9, False),
    (1024, 1024, 4096, 176.9, 182.6, False),
    (768, 1024, 2048, 75.3, 94.5, False),
    (640, 1024, 4096, 115.0, 182.6, False),
    (512, 1024, 8192, 178.7, 357.0, False),
]


@pytest.mark.parametrize("M,N,K,cluster_us,ksplit_us,taken", KSPLIT_MEASURED)
def test_ksplit_tile_where_measured_faster(M, N, K, cluster_us, ksplit_us, taken):
    tiles, full, cs, tile_n = sg.sgemm_f32_plan_model(M, N, K, SMS, "tma")
    ntiles = -(-M // 128) * -(-N // 64)
    if taken:
        assert ksplit_us <= (1 + NEAR) * cluster_us
        assert (tiles, full, cs, tile_n) == (ntiles, ntiles, 1, 64)
    else:
        assert cluster_us <= (1 + NEAR) * ksplit_us
        assert tile_n != 64 or cs > 1
    # only the TMA path has the k-split tile
    for path in ("phased", "cp"):
        t, f, c, n = sg.sgemm_f32_plan_model(M, N, K, SMS, path)
        assert not (n == 64 and c == 1)


def test_narrow_tile_needs_fewer_main_tiles_than_sms():
    # 2048 x 2048 x 512 has 256 main tiles: the narrow tile is not considered
    assert sg.sgemm_f32_plan_model(2048, 2048, 512, SMS, "tma") == (256, 256, 1, 128)


def test_small_k_tile_for_tma_operands_only():
    # 1 <= K <= 64 with TMA operands: the 128 x 64 small-K tile, never split
    assert sg.sgemm_f32_plan_model(16384, 16384, 32, SMS, "tma") == (32768, 32768, 1, 64)
    assert sg.sgemm_f32_plan_model(16384, 16384, 64, SMS, "tma") == (32768, 32768, 1, 64)
    # the same product through the phase maps takes the 128 x 128 tile
    assert sg.sgemm_f32_plan_model(16384, 16384, 32, SMS, "phased") == (16384, 16384, 1, 128)


def test_tiny_products_skip_the_tiles():
    # at most 16384 outputs with 1 <= K <= 128: one thread per output, on every path
    for path in ("tma", "phased", "cp"):
        assert sg.sgemm_f32_plan_model(6, 6, 9, SMS, path) == (1, 1, 1, 0)
        assert sg.sgemm_f32_plan_model(128, 128, 128, SMS, path) == (64, 64, 1, 0)
        assert sg.sgemm_f32_plan_model(128, 128, 129, SMS, path)[3] != 0
        assert sg.sgemm_f32_plan_model(128, 129, 128, SMS, path)[3] != 0
    sg.sgemm_test_tiny_path(False)
    try:
        assert sg.sgemm_f32_plan_model(6, 6, 9, SMS, "tma")[3] == 64   # the small-K tile
    finally:
        sg.sgemm_test_tiny_path(True)


def test_the_plan_follows_the_sm_count():
    # one full round on 152 SMs is a partial one on 148
    assert sg.sgemm_f32_plan_model(2432, 1024, 4096, SMS, "tma") == (152, 152, 1, 128)
    tiles, full, cs, _ = sg.sgemm_f32_plan_model(2432, 1024, 4096, 148, "tma")
    assert tiles == 152 and full == 148 and cs > 1


@pytest.mark.parametrize("args", [(-1, 4, 4, SMS, 0), (4, 4, 4, 0, 0), (4, 4, 4, SMS, 3), (4, 4, 4, SMS, -1)])
def test_model_rejects_bad_arguments(args):
    import ctypes
    M, N, K, sms, path = args
    t, f, c, n = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_int(), ctypes.c_int()
    st = sg.load().sgemm_f32_plan_model(M, N, K, path, sms, ctypes.byref(t), ctypes.byref(f), ctypes.byref(c),
                                        ctypes.byref(n))
    assert st == sg.SGEMM_ERR_INVALID_ARG


# ---------------------------------------------------------------- 3xTF32 layout

def x3_expected_splits(M, N, K, sms, width):
    """The 3xTF32 split rule restated: fewer than sms / 2 tiles of 128 x width
    -> up to 16 k-parts, at least eight 16-deep k-steps each, no empty part."""
    tiles = -(-M // 128) * -(-N // width)
    kt = -(-K // 16)
    if 2 * tiles > sms:
        return 1
    s = min(sms // tiles, kt // 8, 16)
    if s < 2:
        return 1
    per = -(-kt // s)
    return -(-kt // per)


def x3_expected_layout(M, N, K, sms):
    """The 3xTF32 width rule restated: each width w in 208, 192, ..., 128 with
    its own k-parts s costs ceil(tiles * s / sms) rounds x (w + 128) x
    ceil(kt / s); the cheapest wins, ties to the wider tile."""
    kt = -(-K // 16)
    best = None
    for w in (208, 192, 176, 160, 144, 128):
        s = x3_expected_splits(M, N, K, sms, w)
        cost = -(-(-(-M // 128) * -(-N // w) * s) // sms) * (w + 128) * -(-kt // s)
        if best is None or cost < best[0]:
            best = (cost, w, s)
    return best[1], best[2]


def test_3xtf32_layout_follows_the_rule():
    import random
    rng = random.Random(7)
    for _ in range(2000):
        M, N, K = rng.randint(1, 9000), rng.randint(1, 9000), rng.randint(1, 20000)
        sms = rng.choice([148, 152, 160])
        assert sg.sgemm_f32_3xtf32_plan_model(M, N, K, sms) == x3_expected_layout(M, N, K, sms), (M, N, K, sms)


@pytest.mark.parametrize("M,N,K,want", [
    # measured fastest on GB300 (GEMM alone, 340.7 and 300.9 TFLOP/s against 333.3 and 246.4
    # for 128 x 256 with four stages): 128 x 208 with five stages
    (8192, 8192, 8192, (208, 1)), (3001, 4999, 2047, (208, 1)),
    # 600 tiles of 208 fill 3.95 rounds; 1024^3: 48 tiles of 176 x 3 k-parts fill 144 of 152 SMs
    (1024, 1024, 1024, (176, 3))])
def test_3xtf32_layout_on_the_workloads(M, N, K, want):
    assert sg.sgemm_f32_3xtf32_plan_model(M, N, K, SMS) == want


# ---------------------------------------------------------------- stream-K decision

# sgemm_f32 against stream-K at two blocks per SM (TFLOP/s, CUDA events,
# medians; GB300, 152 SMs, L2 flushed between calls): the shapes stream-K
# takes, with both rates, and the shapes it leaves to sgemm_f32
STREAMK_TAKEN = [
    (256, 256, 65536, 22.2, 54.5), (128, 128, 131072, 5.7, 46.6), (384, 384, 16384, 26.4, 47.7),
    (256, 512, 32768, 24.3, 55.6), (384, 384, 4096, 22.5, 28.8), (256, 256, 8192, 18.8, 28.3),
    (128, 1024, 16384, 23.5, 48.0), (512, 512, 32768, 48.4, 58.7), (512, 512, 16384, 47.1, 55.6),
    (1024, 1024, 4096, 48.6, 50.8), (1024, 1024, 8192, 50.8, 56.5), (640, 640, 16384, 50.7, 55.1),
    (1280, 1280, 8192, 53.7, 57.9), (896, 896, 8192, 49.7, 53.8), (512, 2048, 8192, 50.8, 55.9),
    (768, 768, 8192, 54.0, 54.3), (1536, 1536, 4096, 56.1, 56.3),
]
STREAMK_LEFT = [
    (1024, 1024, 1024, 39.8, 32.3), (2048, 2048, 2048, 58.9, 55.9), (640, 640, 4096, 44.0, 40.5),
    (768, 768, 4096, 49.9, 47.7), (1024, 1024, 2048, 44.8, 41.5), (1536, 1536, 1536, 51.8, 47.8),
    (2048, 2048, 8192, 62.4, 60.7), (1280, 1280, 2048, 47.9, 48.2), (300, 700, 10000, 35.2, 35.4),
]


@pytest.mark.parametrize("M,N,K,f32,sk", STREAMK_TAKEN)
def test_streamk_taken_where_measured_faster(M, N, K, f32, sk):
    assert sk >= (1 - NEAR) * f32
    blocks, ws = sg.sgemm_f32_streamk_plan_model(M, N, K, SMS)
    units = tiles128(M, N) * -(-K // 32)
    assert blocks == min(units, 2 * SMS)
    # a counter per tile (in 256-byte blocks) and two 128 x 128 partial tiles per block
    assert ws == -(-tiles128(M, N) * 4 // 256) * 256 + 2 * blocks * 128 * 128 * 4


@pytest.mark.parametrize("M,N,K,f32,sk", STREAMK_LEFT)
def test_streamk_left_to_sgemm_f32_where_not_faster(M, N, K, f32, sk):
    assert sk <= (1 + NEAR) * f32
    assert sg.sgemm_f32_streamk_plan_model(M, N, K, SMS) == (0, 0)


def test_streamk_limits():
    # K <= 64 and tiny products never take stream-K; the grid follows the blocks per SM
    assert sg.sgemm_f32_streamk_plan_model(256, 256, 64, SMS) == (0, 0)
    assert sg.sgemm_f32_streamk_plan_model(100, 100, 100, SMS) == (0, 0)
    assert sg.sgemm_f32_streamk_plan_model(256, 256, 65536, SMS, 1)[0] == SMS
    assert sg.sgemm_f32_streamk_plan_model(128, 128, 96, SMS)[0] == 0          # tiny: 16384 outputs, K <= 128
    sg.sgemm_test_tiny_path(False)
    try:
        assert sg.sgemm_f32_streamk_plan_model(128, 128, 96, SMS)[0] == 3     # one tile of three k-steps
    finally:
        sg.sgemm_test_tiny_path(True)
    import ctypes
    b, w = ctypes.c_longlong(), ctypes.c_size_t()
    for args in [(-1, 4, 4, SMS, 2), (4, 4, 4, 0, 2), (4, 4, 4, SMS, 0)]:
        st = sg.load().sgemm_f32_streamk_plan_model(*args, ctypes.byref(b), ctypes.byref(w))
        assert st == sg.SGEMM_ERR_INVALID_ARG

// The FFMA kernels' shipped tile configurations, one alias per line, each
// with the measurements that chose it.
#pragma once

#include "ffma_tma_sgemm.cuh"

namespace sgemm {

// The shipped configuration: 128 x 128 block tile, 4 warps of 64 x 64, 8 x 16
// outputs per thread accumulated as column pairs with fma.rn.f32x2 in
// column-pair-outer order, 3 stages, k-groups unrolled by four, two CTAs per
// SM.  Chosen by measurement at M = N = K = 8192 among scalar and packed
// forms, per-thread tiles (8x8 .. 16x16), 128 to 512 threads, FFMA orders,
// 2 to 4 stages and unroll depths: 82 % of the FP32 peak against 72 % for the
// best scalar form (16 x 8, row-major order).
using TmaMainTile = TmaTile<8, 16, 2, 2, 3, 1, 2, 4, true>;

// Products with one or two k-steps (K <= 64, e.g. 16384 x 16384 x 32), where
// each block loads once, computes briefly and spends most of its time storing
// C: 128 x 64 tiles, 8 x 8 packed per thread, a single stage and 4 blocks per
// SM (128 registers, no spills) so that the blocks of an SM overlap each
// other's loads, FFMAs and stores; row-outer order with the eight groups of
// four k unrolled (the column-pair-outer order spills at this register
// count).  Measured at 16384 x 16384 x 32: 0.355 ms per product against
// 0.370 ms with 3 blocks per SM (138 registers) and 0.379 ms for the main
// configuration; at K = 64, 0.616 against 0.685 ms.
using TmaSmallKTile = TmaTile<8, 8, 2, 2, 1, 0, 4, 8, true>;

// Products with a single k-step (K <= 32): the same tile with the eight groups
// of four k unrolled by four, half the code of each CTA's only step for four
// CTAs per SM that are rarely at the same point of it.  Measured at 16384 x
// 16384 x 32: 0.349 ms per product against 0.354 ms (unrolled by two: 0.373);
// at K = 64 the full unroll stays faster (0.615 against 0.636 ms).
using TmaSmallK1Tile = TmaTile<8, 8, 2, 2, 1, 0, 4, 4, true>;

// Products with a single k-step, beta == 0 and a C the TMA can address, on the
// kernel that writes C by TMA stores (ffma_tma_smallk.cuh): 128 x 64 tiles of
// two warps, 8 x 16 packed per thread (the main tile's per-thread work, rows
// walked down and up in turn), one stage.  Measured at 16384 x 16384 x 32
// (one product): 0.330 ms against 0.342 ms with per-thread C stores of the
// same tile, 0.345-0.350 ms for TmaSmallK1Tile, 0.334-0.339 ms for 8 x 16 on
// 128 x 64 or 64 x 128 tiles without the row walk and 0.435 ms for 128 x 128
// tiles of four warps at two CTAs per SM.
using TmaSmallKStoreTile = TmaTile<8, 16, 2, 1, 1, 1, 3, 4, true>;

// Products with fewer 128 x 128 tiles than SMs (e.g. 1024^3, 2048 x 1024 x
// 2048) on the TMA kernel: 128 x 64 tiles, 8 x 8 packed per thread, 2 stages and 4 blocks per SM
// (128 registers, no spills), always as thread-block clusters that split each
// tile's k-steps.  Twice the tiles of the main configuration at twice the
// blocks per SM spread the work over the SMs more evenly.  Measured (TFLOP/s,
// against the main tile's plan): 1024^3 39.9 against 38.0, 2048 x 1024 x 2048
// 54.4 against 47.6, 512^3 16.3 against 11.1.
using TmaNarrowTile = TmaTile<8, 8, 2, 2, 2, 1, 4, 8, true>;

// The narrow tile of the cp.async-fed kernel (operands the TMA cannot
// address): the same 128 x 64 tile and arithmetic with 3 stages and 3 blocks
// per SM, since the copy addressing needs more than 128 registers (150-162,
// no spills; at 4 blocks per SM it spills).  Measured with lda = K + 1 and
// ldb = N + 1 (TFLOP/s, against the 128 x 128 cp.async plan): 2048 x 1024 x
// 2048 44.6 against 32.6, 1536^3 43.6 against 35.4, 512^3 14.9 against 7.5.
using TmaNarrowCpTile = TmaTile<8, 8, 2, 2, 3, 1, 3, 8, true>;

// One round of 128 x 64 tiles (70-100 % of the SM count, at most 48 k-steps)
// on the TMA kernel of ffma_tma_ksplit.cuh: one CTA per tile of two groups of
// two warps, each group taking one half of every k-step, 8 x 16 packed per
// thread with the row walk, 3 stages.  This is the per-group tile.  Measured
// against the narrow tile's cluster plan (us per product, CUDA events, mean of
// 400 calls after an L2 flush): 1024^3 52.8 against 54.0, 1024 x 1216 x 1024
// 52.8 against 64.3, 960^3 49.6 against 54.1, 1024 x 1024 x 512 30.7 against
// 33.8; at 64 k-steps the cluster plan wins (1024 x 1024 x 2048: 95.5
// against 97.7).  A variant whose groups took alternate k-steps (each with its
// own two stages of a 4-stage ring) ran 4 % slower at 1024^3.
using TmaKSplitTile = TmaTile<8, 16, 2, 1, 3, 1, 1, 4, true>;

}  // namespace sgemm

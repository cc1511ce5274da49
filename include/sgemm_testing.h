/*
 * libsgemm -- TEST-ONLY interface.
 *
 * Nothing here is part of the product interface in sgemm.h, and a program
 * that computes products has no reason to include this header.  It holds the
 * hooks that the library's own tests use to reach code paths an ordinary call
 * never takes (a bounded wait that runs out, a kernel that the plan would not
 * pick for these operands), and the device-free form of the launch planner.
 */
#ifndef SGEMM_TESTING_H
#define SGEMM_TESTING_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Switches that change how every later product in this process is launched.
 * They take effect only when the environment variable SGEMM_TEST_SWITCHES is
 * "1" at the time of the call; otherwise the call changes nothing and returns
 * SGEMM_ERR_INVALID_ARG, so a program that does not set the variable cannot
 * turn a kernel's copies off by accident.
 *
 * flags bit 0: the TMA-fed kernels never issue their copies, so every block's
 * bounded wait runs out (the timeout path, checked without any fault); bit 1:
 * route every product to the cp.async kernel, so both kernels can be checked
 * on the same inputs; bits 4..7: the cluster size of the cluster split,
 * forced (0 = automatic, 1 = never split, 2 .. 8 = split the tiles beyond
 * whole multiples of the SM count with that size); bit 8: with a forced size,
 * split every tile; bit 9: no programmatic overlap of the cluster-split launch
 * with the plain one before it; bit 10: never use the narrow tile (a forced
 * cluster size also keeps the 128 x 128 tile); bit 11: read 16-byte aligned
 * operands through the phase maps too (every shift 0), so the phased kernel
 * can be checked on any inputs; bit 12: sgemm_f32_streamk takes stream-K
 * whenever its operands allow it; bits 13..14: its grid holds that many blocks
 * per SM (0 = every block that can be resident, two per SM).
 * wait_limit_ns: the bound of each wait (default 2 s).
 * flags = 0 and wait_limit_ns = 2000000000 restore the defaults.
 * SGEMM_ERR_INVALID_ARG if flags < 0, wait_limit_ns == 0, or the environment
 * variable is not "1".
 */
int sgemm_test_switches(int flags, unsigned long long wait_limit_ns);

/*
 * Turns the one-thread-per-output kernel that sgemm_f32 uses for tiny
 * products (at most 16384 outputs, 1 <= K <= 128) on (enable = 1, the default)
 * or off (0: they take the tiled kernels like larger products), for every
 * later product in this process.  The library's tests turn it off so that
 * their small shapes reach the tiled kernels' edge handling, and on where
 * they test the tiny kernel itself.  Same environment condition as
 * sgemm_test_switches; SGEMM_ERR_INVALID_ARG otherwise or if enable is not 0
 * or 1.
 */
int sgemm_test_tiny_path(int enable);

/*
 * The planner of sgemm_f32 without a device: the plan sgemm_f32_plan reports
 * (same outputs, same meaning) for the kernel path `path` -- 0: operands the
 * TMA can address (the TMA kernel, its small-K tile for 1 <= K <= 64);
 * 1: operands whose rows are only 4-byte aligned, read through phase maps
 * (sgemm_f32 takes it when M >= 4 and K >= 4); 2: the cp.async-fed kernel
 * (which sgemm_f32 takes for the remaining unaligned products) -- computed
 * for a GPU with `sms` SMs on which clusters of 2, 4 and 8 blocks can all be
 * resident, with every test switch off (the tiny-product path follows
 * sgemm_test_tiny_path).  It lets the cost models that choose
 * between the plain grid, the cluster split and the narrow tile be checked
 * on a machine without a GPU.  Launches nothing and makes no CUDA call.
 * SGEMM_ERR_INVALID_ARG for a NULL output, a negative size, sms < 1 or an
 * unknown path.
 */
int sgemm_f32_plan_model(int M, int N, int K, int path, int sms, long long *tiles, long long *full_tiles,
                         int *cluster_size, int *tile_n);

/*
 * How sgemm_f32_3xtf32 lays out an M x N x K product on a GPU with `sms`
 * SMs, without a device: *tile_n = the width of its 128-row output tiles
 * (208 down to 128 in steps of 16, the width with the lowest estimated cost:
 * rounds of tiles over the SMs x (width + 128) x k-steps per part) and
 * *splits = the number of parts that divide the k-steps of a small grid
 * (1: none).  SGEMM_ERR_INVALID_ARG for a NULL output, a negative size or
 * sms < 1.
 */
int sgemm_f32_3xtf32_plan_model(int M, int N, int K, int sms, int *tile_n, int *splits);

/*
 * How sgemm_f32_streamk runs an M x N x K product of 16-byte aligned
 * operands on a GPU with `sms` SMs where `blocks_per_sm` blocks of its kernel
 * can be resident, without a device: *blocks = the stream-K grid (0: the call
 * runs as sgemm_f32) and *workspace_bytes = what sgemm_f32_streamk_workspace_size
 * would return there.  Every cluster size is assumed resident and every test
 * switch off (the tiny-product path follows sgemm_test_tiny_path).
 * SGEMM_ERR_INVALID_ARG for a NULL output, a negative size, sms < 1 or
 * blocks_per_sm < 1.
 */
int sgemm_f32_streamk_plan_model(int M, int N, int K, int sms, int blocks_per_sm, long long *blocks,
                                 size_t *workspace_bytes);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_TESTING_H */

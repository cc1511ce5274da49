/*
 * libsgemm -- single-precision matrix product C = A * B on one NVIDIA GB300
 * (sm_103a), hand-written CUDA kernels behind a plain C interface.
 *
 * The operation is the one the tutorial pages build step by step: every
 * output element is the length-K dot product of a row of A and a column of B
 * ("SGEMM: Shared Memory Tiling Visualizer", tiled kernel listing;
 * "Shared Memory Tiling", 'The naive kernel' and 'The tiled kernel'), for
 * general M, N, K with boundary masking (the visualizer's zero-filled tile
 * loads) and strided row-major operands.  There is no alpha, beta or epilogue
 * operation: C is overwritten with the product.
 *
 * Layout (all matrices FP32, row-major, caller-owned DEVICE memory):
 *   A: M x K, element (i, k) at A[i * lda + k], lda >= max(1, K)
 *   B: K x N, element (k, j) at B[k * ldb + j], ldb >= max(1, N)
 *   C: M x N, element (i, j) at C[i * ldc + j], ldc >= max(1, N)
 * Pointers must be 4-byte aligned; a pointer may be NULL only when its matrix
 * has no elements.  Every call is asynchronous on `stream` (0 = the legacy
 * default stream): the library allocates no memory, never synchronises, and
 * does not touch host memory behind the caller's back.  Entries of C outside
 * the M x N block (the gap between N and ldc) are never written.
 *
 * CUDA graphs: the first call on a device does one-time set-up (kernel
 * shared-memory limits, a cluster occupancy query); after one such call,
 * sgemm_f32, sgemm_f32_splitk, sgemm_f32_3xtf32 and sgemm_gemm launch only
 * kernels (and, for sgemm_gemm, device-to-device copies) on `stream`, so they
 * can be captured into a graph and replayed on new data in the same buffers.
 *
 * Numerics: each element is an FP32 sum of FP32 products in some order, with
 * round-to-nearest fused multiply-adds; the result satisfies
 * |C - C_exact| <= 2 * K * 2^-24 * sum_k |a_ik| |b_kj| elementwise, and is
 * exact whenever all partial sums are exactly representable (e.g. small
 * integers).  K == 0 writes zeros (an empty sum).
 *
 * Errors: every entry point validates its arguments on the host before any
 * CUDA call and returns a status; on any status other than SGEMM_OK nothing
 * was launched.  SGEMM_ERR_LAUNCH carries a CUDA launch failure (including a
 * device without an sm_103a image); errors of earlier asynchronous work on the
 * stream are not this library's and surface at the caller's next
 * synchronisation.
 */
#ifndef SGEMM_H
#define SGEMM_H

#include <stddef.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1, /* negative size, short leading dimension, NULL or misaligned pointer */
    SGEMM_ERR_ALIAS = 2,       /* C overlaps A or B */
    SGEMM_ERR_LAUNCH = 3,      /* the CUDA launch (or its attribute set-up) failed */
    SGEMM_ERR_DEVICE = 4,      /* the device reported an error (cudaGetDevice / attributes) */
    SGEMM_ERR_TIMEOUT = 5,     /* a kernel gave up on a bounded wait (reported by sgemm_device_status) */
    SGEMM_ERR_SCRATCH_LIMIT = 6 /* sgemm_f32_splitk_noalloc: the partials do not fit its static scratch */
} sgemm_status;

/*
 * C = A * B ("Shared Memory Tiling", the tiled kernel and 'What tiling does
 * not fix'; "SGEMM: 2D Register Tiling Visualizer", the outer-product listing).
 * Register-tiled FP32 FFMA kernels with thread-block tiles staged in shared
 * memory through a multi-stage pipeline:
 *   - A and B with 16-byte aligned bases and leading dimensions (multiples of
 *     4 floats), K >= 1: 128 x 128 block tiles copied by the tensor memory
 *     accelerator (TMA) with hardware zero-fill at the edges, 8 x 16 outputs
 *     per thread accumulated with packed two-wide FP32 FMAs; K <= 64 takes
 *     128 x 64 tiles of a single stage, and a single k-step (K <= 32) with a
 *     16-byte aligned C whose row length N is a multiple of 4 writes its C
 *     tiles by TMA stores from shared memory;
 *   - otherwise, with M >= 4 and K >= 4: the same tiles and packed FMAs, each
 *     operand read by the TMA through four tensor maps, one per residue of
 *     the row index mod 4 (those rows are 4 * ld floats apart, a multiple of
 *     16 bytes), in boxes 4 floats wider than the tile; each row is shifted
 *     into place in shared memory before the FMAs.  A phase map starts at the
 *     16-byte boundary at or below its first row, so up to 3 floats in front
 *     of a row (the previous row's tail, or for the first row the bytes
 *     before A or B in the same 16-byte granule) are read and never used;
 *   - otherwise (M < 4, K < 4, or K == 0): the same tiles, fragment reads and
 *     packed FMAs, fed by cp.async copies (16-byte copies for an operand whose
 *     rows are 16-byte aligned, 4-byte copies otherwise).  A last, partial row of
 *     tiles reads the 128 rows of A that end at row M and stores only its
 *     own; B's right edge is a per-thread copy size; only the last, partial
 *     k-step and products with M < 128 take per-element masks.  The copy
 *     strides are 32-bit: an operand needing 16 * lda (A) or 4 * ldb (B)
 *     >= 2^31 takes 4-byte copies, and an A whose rows are not 16-byte
 *     aligned with 4 * lda >= 2^31 is computed by the pages' register-tiled
 *     ladder kernel (64-bit indexing, much slower).
 * On every path, when a grid would leave SMs idle (few tiles, or a last
 * partial round of tiles over the SMs), those tiles are each shared by a
 * thread-block cluster of 2, 4 or 8 blocks that split its k-steps and add their
 * partial sums through distributed shared memory in a fixed rank order: no
 * workspace, and the same bits on every run.  With fewer 128 x 128 tiles than
 * SMs, any path may instead use narrow 128 x 64 tiles (8 x 8 outputs per
 * thread; four blocks per SM on the TMA and phased paths, three on the
 * cp.async path, the latter only when 16 * lda and 8 * ldb fit in 32 bits),
 * all in such clusters
 * (sgemm_f32_plan reports the choice).  On the TMA path, products whose
 * narrow tiles fill one round over the SMs to at least 70 % with at most 48
 * k-steps (e.g. 1024^3) instead run one block per narrow tile, of two groups
 * of warps that each take one half of every k-step and add their sums in
 * shared memory (no cluster).  Tiny products -- at most 16384
 * outputs, 1 <= K <= 128, on any path -- skip the tiles: one thread per output
 * computes its dot product straight from memory (the pages' naive kernel),
 * which for them costs a fraction of the tiled kernels' set-up.
 * Returns an sgemm_status.  M == 0 or N == 0: SGEMM_OK, nothing launched.
 * The TMA kernels' waits are bounded: if a copy never lands, its blocks give
 * up, write nothing, and the next sgemm_device_status() returns
 * SGEMM_ERR_TIMEOUT.
 */
int sgemm_f32(int M, int N, int K,
              const float *A, int lda,
              const float *B, int ldb,
              float *C, int ldc,
              cudaStream_t stream);

/*
 * How sgemm_f32 launches an M x N x K product on the current device, for
 * operands the TMA can address (tma_operands != 0: A, B 16-byte aligned with
 * leading dimensions that are multiples of 4) or not (0): *tiles = the number
 * of output tiles, 128 rows by *tile_n columns; the first *full_tiles of them
 * run as a plain grid, the rest as clusters of *cluster_size blocks that
 * split each tile's k-steps (*cluster_size == 1: no cluster split,
 * *full_tiles == *tiles).  *tile_n is 64 for TMA operands with 1 <= K <= 64
 * (never split) and for the narrow tile, which a product with fewer 128 x 128
 * tiles than SMs takes when its cost model says so (then every tile is in a
 * cluster, or, for the two-group k-split blocks of TMA operands,
 * *cluster_size == 1 and *full_tiles == *tiles); 128 otherwise.  Non-TMA operands with M >= 4 and K >= 4 take the
 * phased TMA kernel's plan; smaller ones the cp.async kernel's, which assumes
 * 16 * lda and 8 * ldb fit in 32 bits (otherwise the 128 x 128 plan runs).  The result
 * reflects the switches of the test-only interface (sgemm_testing.h), which
 * are all off unless a test turned them on.  Tiny products (at most 16384
 * outputs, 1 <= K <= 128) report *tile_n = 0, *cluster_size = 1 and
 * *tiles = *full_tiles = the blocks of 256 outputs of the one-thread-per-output
 * kernel.  Launches nothing.
 * SGEMM_ERR_INVALID_ARG for a NULL output or negative size; SGEMM_ERR_DEVICE
 * if the device cannot be queried.
 */
int sgemm_f32_plan(int M, int N, int K, int tma_operands, long long *tiles, long long *full_tiles,
                   int *cluster_size, int *tile_n);

/*
 * Split-K form of sgemm_f32 for grids with fewer output tiles than the GPU has
 * SMs (e.g. 1024 x 1024 x 1024): the K dimension is cut into `splits` ranges
 * of whole k-steps, each computed by its own set of thread blocks into a
 * partial M x N product in `workspace`, and a second kernel adds the partials
 * in increasing split order into C (deterministic; each element is still an
 * FP32 sum of FP32 products, within the bound stated above, and exact for
 * small-integer inputs).  The tiled kernels and their choice are those of
 * sgemm_f32 ("Shared Memory Tiling", 'The tiled kernel': the k loop over
 * tiles, here divided among thread blocks).
 *   splits: 1 .. 64; values above the number of k-steps are lowered to it;
 *           splits == 1 is exactly sgemm_f32 and needs no workspace.
 *   workspace: caller-owned device memory of at least
 *           sgemm_f32_splitk_workspace_size(M, N, splits) bytes, 16-byte
 *           aligned, not overlapping A, B or C; its contents on entry do not
 *           matter and on return are unspecified.
 * SGEMM_ERR_INVALID_ARG for a bad split count or a missing, misaligned or
 * short workspace; SGEMM_ERR_ALIAS if the workspace overlaps an operand.  If
 * a product kernel gives up on a bounded wait (SGEMM_ERR_TIMEOUT from
 * sgemm_device_status), it fills its partial tile with NaN instead, and the
 * reduction, which still runs, makes the elements of C in that tile NaN.
 */
int sgemm_f32_splitk(int M, int N, int K,
                     const float *A, int lda,
                     const float *B, int ldb,
                     float *C, int ldc,
                     int splits, float *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* Workspace bytes sgemm_f32_splitk needs: splits * M * (N rounded up to 4) * 4
 * for splits > 1, else 0. */
size_t sgemm_f32_splitk_workspace_size(int M, int N, int splits);

/*
 * A split count for M x N x K on the current device: enough splits for the
 * grid of 128 x 128 output tiles to reach two blocks per SM, with at least
 * four 32-deep k-steps per split (1 when the tiles already fill the GPU).
 */
int sgemm_f32_splitk_suggest(int M, int N, int K, int *splits);

/*
 * Stream-K form of sgemm_f32 for products with few output tiles over a long
 * K (e.g. 256 x 256 x 65536), where even thread-block clusters of eight
 * blocks per tile would leave SMs idle -- the load imbalance "Shared Memory
 * Tiling" ('What tiling does not fix') points at.  The product is cut into
 * units of one 128 x 128 tile and one 32-deep k-step, and every block that
 * can be resident (two per SM) takes an equal contiguous run of them across
 * tile boundaries, with the tiled kernel of sgemm_f32 (TMA-fed tiles, packed
 * FP32 FMAs).  The blocks that share a tile write their partial tiles to the
 * workspace; once all have, each adds up its own slice of the tile over them
 * in an order fixed by the shape (so every run gives the same bits) and
 * stores it.  Each element is an FP32 sum of FP32 products within the bound
 * stated above, and exact for small integers.
 *   Stream-K runs when A and B are 16-byte aligned with leading dimensions
 *   that are multiples of 4, K > 64, the product is not a tiny one (see
 *   sgemm_f32), and either sgemm_f32's own plan would start fewer blocks than
 *   the device has SMs (its one-round k-split blocks count as filling them),
 *   or there are fewer 128 x 128 tiles than SMs and each block gets at least
 *   24 units.  Every other product runs exactly as
 *   sgemm_f32 does and reads no workspace.  The kernel is launched
 *   cooperatively (all of its blocks resident at once).
 *   workspace: caller-owned device memory of at least
 *     sgemm_f32_streamk_workspace_size(M, N, K) bytes (0 when the product
 *     does not take stream-K; about 40 MB on a GPU with 152 SMs), 16-byte
 *     aligned, not overlapping A, B or C: one counter per tile, which the call
 *     zeroes (a memset on `stream`) before its kernel, and two partial tiles
 *     per block.  Its contents on entry do not matter.  Calls that share a
 *     workspace must not overlap on the GPU.
 * Errors as for sgemm_f32_splitk.  Every wait is bounded -- on the copies, and
 * on the other blocks that share a tile; a block that gives up stops, so the
 * tiles it shares are not stored (C keeps its old values there) and
 * sgemm_device_status reports SGEMM_ERR_TIMEOUT.
 */
int sgemm_f32_streamk(int M, int N, int K,
                      const float *A, int lda,
                      const float *B, int ldb,
                      float *C, int ldc,
                      float *workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* Workspace bytes sgemm_f32_streamk needs for an M x N x K product of
 * 16-byte aligned operands on the current device (0 when it runs as
 * sgemm_f32). */
size_t sgemm_f32_streamk_workspace_size(int M, int N, int K);

/*
 * C = A * B in FP32 accuracy on the tensor cores ("3xTF32").  Each operand is
 * split into a TF32 high part and a TF32 low part (rounded to nearest), and
 * C = A_hi B_hi + A_hi B_lo + A_lo B_hi is accumulated in FP32 by tcgen05
 * matrix instructions with the accumulator in tensor memory.  The tiling,
 * pipelining and edge masking are those of the tiled kernel ("Shared Memory
 * Tiling", the tiled kernel and 'What tiling does not fix'), with the inner
 * product on the tensor cores instead of the FP32 cores: one persistent
 * block per SM walks 128-row output tiles (208 columns wide, or 192 down to
 * 128 when a narrower tile fills the last round of tiles over the SMs better),
 * with two accumulators so that one tile's stores overlap the next tile's
 * products.
 *
 * Accuracy: each product carries a relative error of about 3 * 2^-22 from the
 * split, on top of the FP32 accumulation; the result is held to the same bound
 * as sgemm_f32, |C - C_exact| <= 2 K 2^-24 sum_k |a_ik| |b_kj|, which this
 * leaves room for once K is a few dozen (tested at K = 9 and up).  Small
 * integers are split exactly (A_lo = 0), so integer products whose partial
 * sums stay below 2^24 are exact.
 *
 * A grid of fewer than half as many 128 x 208 output tiles as the device has
 * SMs (e.g. 1024 x 1024 x 1024) has its k-steps divided into up to 16 parts;
 * their partial tiles land in the workspace and are added in part order into
 * C (deterministic, the same bound).
 *
 * workspace: caller-owned device memory of at least
 * sgemm_f32_3xtf32_workspace_size(M, N, K) bytes, 16-byte aligned, not
 * overlapping A, B or C; it receives A_hi, A_lo (M x K) and B_hi, B_lo
 * transposed (N x K), with rows padded to a multiple of 4 floats, then the
 * partial tiles of a divided product.  Any alignment of A, B and C is
 * accepted.  K <= 2,097,120.  K == 0 writes zeros and needs no workspace.
 * Errors as for sgemm_f32_splitk; the copy waits are bounded and report
 * through sgemm_device_status (after a timeout of a divided product, the
 * elements of C in the tiles that gave up are NaN).
 */
int sgemm_f32_3xtf32(int M, int N, int K,
                     const float *A, int lda,
                     const float *B, int ldb,
                     float *C, int ldc,
                     float *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* Workspace bytes sgemm_f32_3xtf32 needs on the current device: 4 (2M + 2N)
 * (K rounded up to 4), rounded up to 256, plus splits * M * (N rounded up to
 * 4) * 4 when the product is divided. */
size_t sgemm_f32_3xtf32_workspace_size(int M, int N, int K);

/*
 * sgemm_f32_splitk without a workspace argument, for callers that cannot
 * allocate device memory: code that runs inside a host application which owns
 * the whole device-memory budget (a plug-in handed only its input and output
 * buffers), or a latency-critical loop where an allocation, which may
 * synchronise the device and take unbounded time, is not allowed.  The
 * SGEMM pages have no counterpart to this entry point; it only changes
 * where the split-K partial products live.
 *
 * The partials go to one fixed array in device memory that the library
 * reserves when it is loaded: 8,388,608 floats (32 MiB) on every device that
 * loads the library, held until the process exits.  Requests with
 * splits * M * (N rounded up to 4) above that (after splits is lowered to the
 * number of k-steps) return SGEMM_ERR_SCRATCH_LIMIT and launch nothing;
 * splits == 1 needs no scratch.  This function allocates nothing and calls no
 * allocating routine.  Its first call on each device looks up the array's
 * device address (a CUDA runtime query, done once per device with that device
 * current); make that first call before any stream capture.
 *
 * Every call on a device shares the one array, and the array keeps the last
 * call's partials.  Nothing in it needs to start at zero: the product kernels
 * of a call write every partial sum that its reduction adds into C (rows < M,
 * columns < N of each split's slab) before the reduction runs.  The reduction
 * also reads the padding columns of a slab (N up to the next multiple of 4),
 * which may hold an earlier call's values; it discards them.  A product kernel
 * that gives up on a bounded wait fills its partial tile with NaN, so an
 * earlier call's partials never reach C (those elements of C are NaN).  Calls
 * whose kernels overlap on the GPU (on different streams, or from different
 * threads) race on the array and give wrong results: order them on one stream
 * or with events.  Arguments, results and the other error codes are as for
 * sgemm_f32_splitk.
 */
int sgemm_f32_splitk_noalloc(int M, int N, int K,
                             const float *A, int lda,
                             const float *B, int ldb,
                             float *C, int ldc,
                             int splits, cudaStream_t stream);

/*
 * General form: C = alpha * op(A) op(B) + beta * C, BLAS-style, row-major.
 * The pages' product is the case alpha = 1, beta = 0, no transposes; the
 * rest is the usual superset (the pages use none of it).
 *   transa: SGEMM_OP_N -- A is M x K (lda >= K); SGEMM_OP_T -- A is stored
 *           K x M (lda >= M) and op(A) = A^T.
 *   transb: SGEMM_OP_N -- B is K x N (ldb >= N); SGEMM_OP_T -- B is stored
 *           N x K (ldb >= K) and op(B) = B^T.
 *   beta == 0: C is not read (NaN in C does not propagate).
 *   alpha == 0 or K == 0: A and B are not read; C = beta * C.
 *   algo: SGEMM_ALGO_FFMA -- the FP32 FFMA kernels of sgemm_f32; an operand
 *           given transposed is first copied row-major with padded rows into
 *           the workspace (one memory-bound pass), so that the product runs
 *           on the TMA-fed kernels.  An operand whose base or leading
 *           dimension is not 16-byte aligned is read in place through phase
 *           maps, as by sgemm_f32; only when M or K is below 4 is it copied
 *           into the workspace as well.
 *         SGEMM_ALGO_3XTF32 -- the tensor-core path of sgemm_f32_3xtf32; its
 *           operand split reads either orientation directly.
 *   workspace: at least sgemm_gemm_workspace_size(...) bytes, caller-owned
 *           device memory, 16-byte aligned, not overlapping A, B or C; the
 *           FFMA form reads it only for transposed operands, and for
 *           unaligned ones when M or K is below 4 (and may be given NULL
 *           otherwise).
 * Accuracy: |C - C_exact| <= 2 (K + 2) 2^-24 (|alpha| sum_k |a||b| + |beta||c|).
 * K <= 2,097,120 (and N <= 2,097,120 when B is transposed); other errors as
 * for sgemm_f32_3xtf32.
 */
typedef enum { SGEMM_OP_N = 0, SGEMM_OP_T = 1 } sgemm_op;
typedef enum { SGEMM_ALGO_FFMA = 0, SGEMM_ALGO_3XTF32 = 1 } sgemm_algo;

int sgemm_gemm(int algo, int transa, int transb, int M, int N, int K,
               float alpha, const float *A, int lda,
               const float *B, int ldb,
               float beta, float *C, int ldc,
               float *workspace, size_t workspace_bytes,
               cudaStream_t stream);

/* Workspace bytes sgemm_gemm needs for this algorithm and operand orientation. */
size_t sgemm_gemm_workspace_size(int algo, int transa, int transb, int M, int N, int K);

/*
 * C = A * B with A, B and C in HOST memory: the end-to-end form of sgemm_f32.
 * B is copied to the device once, in up to 8 column blocks of growing width;
 * then, panel by
 * panel of at most `panels` row panels of C (each rounded up to whole waves of
 * 128 x 128 output tiles on this device, so fewer panels may result), the rows
 * of A are copied in on h2d_stream, the product runs on `stream` with the
 * kernels of sgemm_f32, and the rows of C are copied back on d2h_stream, so
 * that copies of one panel overlap the product of another.  The first panel's
 * product runs block by block as the blocks of B land.  Each product is an
 * sgemm_f32 launch on the device copies: every element is held to the same
 * bound, and its bits equal sgemm_f32's on the whole product except where the
 * cluster split divides that element's k-steps differently for a panel than
 * for the whole (never when neither splits).
 *   workspace: caller-owned device memory of at least
 *     sgemm_f32_host_workspace_size(M, N, K, panels) bytes (B, two A panels
 *     and two C panels), 16-byte aligned; the library allocates nothing.
 *   streams: three caller-owned streams (distinct for overlap); the copies
 *     start only after the work already queued on `stream` (so back-to-back
 *     calls may share one workspace); the call is asynchronous and its work
 *     is complete when `stream` reaches the point after the call (synchronise
 *     `stream`, not the copy streams).  A, B and
 *     C must stay valid until then; pinned (page-locked) host memory is needed
 *     for the copies to overlap.  A thread's first call on a device creates 17
 *     CUDA events that its later calls there reuse (released at process exit).
 *   K == 0: C's rows are zeroed on the host before returning.
 * Errors: SGEMM_ERR_INVALID_ARG (sizes, strides, NULL, panels < 1, short or
 * misaligned workspace), SGEMM_ERR_LAUNCH (a copy, event or launch failed).
 */
int sgemm_f32_host(int M, int N, int K,
                   const float *A, int lda,
                   const float *B, int ldb,
                   float *C, int ldc,
                   int panels, float *workspace, size_t workspace_bytes,
                   cudaStream_t stream, cudaStream_t h2d_stream, cudaStream_t d2h_stream);

/* Device workspace bytes sgemm_f32_host needs for this shape and panel count
 * on the current device (it queries the SM count; 0 if that fails). */
size_t sgemm_f32_host_workspace_size(int M, int N, int K, int panels);

/*
 * The pages' kernel ladder, as GPU kernels: the reference points the tuned
 * kernels are measured against, and the kernels whose executed global loads
 * the pages count.  Every level computes C = A * B with the same contract,
 * shapes, strides, masks and errors as sgemm_f32 (plain loads: any 4-byte
 * alignment), one FP32 FMA chain per output in increasing k.
 *   SGEMM_LADDER_NAIVE: one thread per output, operands read straight from
 *     global memory, 2MNK loads ("Shared Memory Tiling", 'The naive kernel').
 *   SGEMM_LADDER_TILED_16 / _32: T x T thread blocks staging T x T tiles of A
 *     and B in shared memory with zero-filled edges, 2MNK/T loads for
 *     T-divisible shapes ("SGEMM: Shared Memory Tiling Visualizer", the tiled
 *     kernel); _32_PADDED uses [32][33] tiles ("Shared Memory Tiling",
 *     'Conflict-free layout').
 *   SGEMM_LADDER_REGISTER_2D: 64 x 64 x 8 block tiles, 4 x 4 outputs per
 *     thread from register outer products ("SGEMM: 2D Register Tiling
 *     Visualizer", the listing).
 * Row-block counts above 65535 (M > 65535 x 16 / 32 / 64) return
 * SGEMM_ERR_INVALID_ARG.
 */
typedef enum {
    SGEMM_LADDER_NAIVE = 0,
    SGEMM_LADDER_TILED_16 = 1,
    SGEMM_LADDER_TILED_32 = 2,
    SGEMM_LADDER_TILED_32_PADDED = 3,
    SGEMM_LADDER_REGISTER_2D = 4
} sgemm_ladder_level;

int sgemm_f32_ladder(int level, int M, int N, int K,
                     const float *A, int lda,
                     const float *B, int ldb,
                     float *C, int ldc,
                     cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears this device's error word, which
 * kernels set when a bounded wait runs out.  SGEMM_OK if no kernel gave up
 * since the last call, SGEMM_ERR_TIMEOUT if one did, SGEMM_ERR_DEVICE if a
 * CUDA call failed (including an earlier asynchronous error on the stream).
 */
int sgemm_device_status(cudaStream_t stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char *sgemm_status_string(int status);

/* Library interface version: 100 * major + minor. */
int sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_H */

// The C interface of libsgemm: argument checks, kernel choice and launch.
// Declarations and the full contract are in include/sgemm.h (and the
// test-only entry points in include/sgemm_testing.h).
//
// How sgemm_f32 chooses a kernel (launch_product), in order:
//   1. tiny products (<= 16384 outputs, K <= 128): one thread per output
//      (ffma_tiny.cuh);
//   2. operands the TMA can address (16-byte aligned bases and rows):
//      K <= 32 with beta == 0 and N % 4 == 0 -> the TMA-store small-K tile
//      (ffma_tma_smallk.cuh); K <= 64 -> the 8 x 8 small-K tile; otherwise the
//      main 128 x 128 tile (ffma_tma_sgemm.cuh), planned by split_plan;
//   3. rows only 4-byte aligned, M >= 4 and K >= 4: the same tiles read through
//      four phase maps per operand (ffma_tma_phased.cuh), planned likewise;
//   4. otherwise the cp.async-fed kernel (ffma_cp_packed.cuh), or for A rows
//      more than 2 GiB apart the pages' register-tiled ladder kernel.
// split_plan (the fitted cost models; split_plan_model is the device-free
// part) decides between a plain grid, a plain grid plus the cluster split of
// its last partial round of tiles, and narrow 128 x 64 tiles in clusters.
// The other entry points reuse these launches: split-K and its allocation-free
// form (partials + splitk_reduce.cuh), stream-K (ffma_tma_streamk.cuh), the
// 3xTF32 product (tf32_split.cuh + tf32x3_tcgen05.cuh, x3_width choosing the
// tile width), sgemm_gemm (repacks transposed or unaligned operands when the
// FFMA path needs it) and the host-buffer pipeline at the end of the file.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "../../include/sgemm.h"
#include "../../include/sgemm_testing.h"
#include "ffma_cp_packed.cuh"
#include "ffma_tma_phased.cuh"
#include "ffma_tma_sgemm.cuh"
#include "ffma_tma_smallk.cuh"
#include "ffma_tma_ksplit.cuh"
#include "ffma_tma_streamk.cuh"
#include "ffma_tiny.cuh"
#include "ladder.cuh"
#include "splitk_reduce.cuh"
#include "tf32_split.cuh"
#include "tf32x3_tcgen05.cuh"
#include "tiles.cuh"

// Device error word: kernels that give up on a bounded wait record a code here;
// sgemm_device_status() reads and clears it.  One instance per device context.
__device__ int g_sgemm_device_error;

// Fixed scratch for sgemm_f32_splitk_noalloc: room for the split-K partial
// products of callers that cannot allocate device memory.  8,388,608 floats
// (32 MiB), reserved on every device that loads this library until the
// process exits.  Shared by all calls on a device.
constexpr long long kNoallocScratchFloats = 8388608;
static __device__ __align__(256) float g_splitk_noalloc_scratch[kNoallocScratchFloats];

namespace {

using TmaTile = sgemm::TmaMainTile;
using TmaSmallK = sgemm::TmaSmallKTile;
using TmaSmallK1 = sgemm::TmaSmallK1Tile;
using TmaNarrow = sgemm::TmaNarrowTile;
using TmaNarrowCp = sgemm::TmaNarrowCpTile;
using TmaKSplit = sgemm::TmaKSplitTile;
using TmaPhased = sgemm::PhasedTile<sgemm::TmaMainTile>;
using PhasedNarrow = sgemm::PhasedTile<sgemm::TmaNarrowTile>;
using X3Tile = sgemm::Tf32x3MainTile;

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;

// test-only switches (sgemm_test_switches); bit 0 is read by the TMA kernels.
// Bit 1: route every product to the cp.async-fed kernel.  Bits 4..7: cluster
// size forced on the cluster split of the main tile (0 = the automatic plan,
// 1 = never split, 2 .. 8 = split the tiles beyond whole multiples of the SM
// count with that cluster size); bit 8: put every tile in the cluster-split
// launch; bit 9: no programmatic overlap; bit 10: never use the narrow tile;
// bit 11: read 16-byte aligned operands through the phase maps as well (the
// main tile of the phased kernel instead of the TMA kernel).
constexpr int kDebugForceCpAsync = 2;
constexpr int kDebugClusterShift = 4;
constexpr int kDebugClusterAll = 256;
constexpr int kDebugNoOverlap = 512;  // launch the cluster-split grid without programmatic overlap
constexpr int kDebugNoNarrow = 1024;
constexpr int kDebugForcePhased = 2048;
constexpr int kDebugForceStreamK = 4096;  // sgemm_f32_streamk: stream-K whatever the tile count
constexpr int kDebugStreamKPerSmShift = 13;  // bits 13..14: stream-K blocks per SM (0 = all resident)
std::atomic<int> g_debug_flags{0};
// test-only (sgemm_test_tiny_path): tiny products take the one-thread-per-output kernel
std::atomic<int> g_tiny_path{1};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

struct DeviceInfo {
    int dev = 0;
    int sms = 0;
    int *err_word = nullptr;
};

// Per-device facts queried once: SM count and the device address of the error word.
int device_info(DeviceInfo &out) {
    static std::mutex mu;
    static DeviceInfo info[kMaxDevices];
    static bool ready[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        DeviceInfo d;
        d.dev = dev;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SGEMM_ERR_DEVICE;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err_word), g_sgemm_device_error) != cudaSuccess)
            return SGEMM_ERR_DEVICE;
        info[dev] = d;
        ready[dev] = true;
    }
    out = info[dev];
    return SGEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major rows x cols FP32 matrix with leading dimension ld, read in boxes of
// box_rows x box_cols; out-of-bounds elements read as zero.
bool encode_2d(CUtensorMap *map, const float *ptr, int rows, int cols, int ld, int box_rows, int box_cols,
               CUtensorMapSwizzle swizzle) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four phase maps of a rows x cols operand (leading dimension ld, rows
// >= 4, base 4-byte aligned): phase s holds rows s, s + 4, ..., 4 ld floats
// apart; it starts at the 16-byte boundary d_s floats below row s, is
// cols + d_s wide (zero past the operand's last column and last row) and is
// read in boxes of box_rows x (box_cols + 4).  Returns d_0 .. d_3, two bits
// each, or -1 when a map cannot be encoded.
int encode_phases(CUtensorMap (&maps)[4], const float *ptr, int rows, int cols, int ld, int box_rows, int box_cols) {
    auto fn = encode_fn();
    if (!fn || rows < 4) return -1;
    int shifts = 0;
    for (int s = 0; s < 4; ++s) {
        const uintptr_t row = reinterpret_cast<uintptr_t>(ptr) + (uintptr_t)s * (uintptr_t)ld * sizeof(float);
        const int d = (int)((row >> 2) & 3);
        const cuuint64_t dims[2] = {(cuuint64_t)cols + (cuuint64_t)d, (cuuint64_t)((rows - s + 3) / 4)};
        const cuuint64_t strides[1] = {(cuuint64_t)4 * (cuuint64_t)ld * sizeof(float)};
        const cuuint32_t box[2] = {(cuuint32_t)box_cols + 4, (cuuint32_t)box_rows};
        const cuuint32_t elem[2] = {1, 1};
        if (fn(&maps[s], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, reinterpret_cast<void *>(row - 4 * (uintptr_t)d), dims,
               strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return -1;
        shifts |= d << (2 * s);
    }
    return shifts;
}

// Raise a kernel's dynamic shared-memory limit once (per device: `done` is the
// caller's flag for this kernel and device).
template <class Kernel>
bool smem_attr_once(std::atomic<int> &done, Kernel kernel, int bytes) {
    if (done.load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done.store(1, std::memory_order_release);
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// C = alpha * op(A) op(B) + beta * C.  The product kernels take A as M x K and
// B as K x N row-major; transa / transb mean A is stored K x M and B N x K
// (only the 3xTF32 split pass reads those orientations directly).
struct Problem {
    int M, N, K;
    const float *A;
    int lda;
    const float *B;
    int ldb;
    float *C;
    int ldc;
    float alpha = 1.f, beta = 0.f;
    bool transa = false, transb = false;
};

// The TMA kernel needs 16-byte aligned bases and row strides and K >= 1.
bool use_tma(const Problem &p) {
    return p.K > 0 && aligned16(p.A) && p.lda % 4 == 0 && aligned16(p.B) && p.ldb % 4 == 0 &&
           !(g_debug_flags.load() & (kDebugForceCpAsync | kDebugForcePhased));
}

// Operands the TMA kernel cannot address (rows only 4-byte aligned) go through
// four phase maps each, which need at least four rows of A and of B.
bool use_phased(const Problem &p) {
    const int dbg = g_debug_flags.load();
    return p.M >= 4 && p.K >= 4 && !(dbg & kDebugForceCpAsync) && ((dbg & kDebugForcePhased) || !use_tma(p));
}

int k_tiles(const Problem &p) { return (p.K + TmaTile::BK - 1) / TmaTile::BK; }

// The cp.async kernel holds its per-copy row strides in 32-bit registers: 16
// rows of A (16-byte copies) or 4 (4-byte copies), 4 rows of B (16-byte) or 1.
// An operand whose stride would not fit takes the narrower copies; A with
// 4 * lda >= 2^31 (rows more than 2 GiB apart) cannot take that kernel at all.
constexpr int64_t kIntMax = 0x7fffffff;
bool cp_vec_a(const Problem &p) { return aligned16(p.A) && p.lda % 4 == 0 && 16 * (int64_t)p.lda <= kIntMax; }
bool cp_vec_b(const Problem &p) { return aligned16(p.B) && p.ldb % 4 == 0 && 4 * (int64_t)p.ldb <= kIntMax; }
bool cp_fits(const Problem &p) { return 4 * (int64_t)p.lda <= kIntMax; }
// The narrow tile's B copies step 8 rows (16-byte) or 2 (4-byte): it is used
// only when every stride of either width fits.
bool cp_narrow_fits(const Problem &p) { return 16 * (int64_t)p.lda <= kIntMax && 8 * (int64_t)p.ldb <= kIntMax; }

template <class T, bool VC, int ROLE, bool PLAIN = false>
bool tma_attr(int dev) {
    static std::atomic<int> done[kMaxDevices];
    return smem_attr_once(done[dev], sgemm::sgemm_ffma_tma_kernel<T, VC, ROLE, PLAIN>, T::SMEM_BYTES);
}

template <class T, bool VC, int ROLE>
bool phased_attr(int dev) {
    static std::atomic<int> done[kMaxDevices];
    return smem_attr_once(done[dev], sgemm::sgemm_ffma_tma_phased_kernel<T, VC, ROLE>, T::SMEM_BYTES);
}

template <class T>
struct IsPhased : std::false_type {};
template <class T>
struct IsPhased<sgemm::PhasedTile<T>> : std::true_type {};

// The cluster-split launch configuration: `clusters` clusters of cs CTAs and,
// after a plain grid of the same product, programmatic overlap with that grid.
template <class T>
cudaLaunchConfig_t split_config(int64_t clusters, int cs, bool overlap, cudaStream_t stream,
                                cudaLaunchAttribute (&attr)[2]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(clusters * cs));
    cfg.blockDim = dim3(T::THREADS);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 2 : 1;
    return cfg;
}

// Whether clusters of `cs` CTAs of the cluster-split kernel can be resident on
// this device at all; queried once per device and size on the kernel of T
// (the TMA, cp.async-fed or phased form).
template <class T, bool VA, bool VB, int ROLE>
bool cp_packed_attr(int dev);

template <class T, bool CP = false>
bool cluster_fits(int dev, int cs) {
    static std::atomic<int> known[kMaxDevices][9];  // 0 unknown, 1 yes, 2 no
    if (cs < 2 || cs > 8) return false;
    std::atomic<int> &slot = known[dev][cs];
    int k = slot.load(std::memory_order_acquire);
    if (k == 0) {
        bool smem_ok;
        if constexpr (CP) smem_ok = cp_packed_attr<T, false, false, sgemm::kRoleSplit>(dev);
        else if constexpr (IsPhased<T>::value) smem_ok = phased_attr<T, true, sgemm::kRoleSplit>(dev);
        else smem_ok = tma_attr<T, true, sgemm::kRoleSplit>(dev);
        if (!smem_ok) return false;
        cudaLaunchAttribute attr[2];
        const cudaLaunchConfig_t cfg = split_config<T>(1, cs, false, 0, attr);
        int n = 0;
        cudaError_t e;
        if constexpr (CP)
            e = cudaOccupancyMaxActiveClusters(&n, sgemm::sgemm_ffma_cp_kernel<T, false, false, sgemm::kRoleSplit>,
                                               &cfg);
        else if constexpr (IsPhased<T>::value)
            e = cudaOccupancyMaxActiveClusters(&n, sgemm::sgemm_ffma_tma_phased_kernel<T, true, sgemm::kRoleSplit>,
                                               &cfg);
        else
            e = cudaOccupancyMaxActiveClusters(&n, sgemm::sgemm_ffma_tma_kernel<T, true, sgemm::kRoleSplit>, &cfg);
        const bool ok = e == cudaSuccess && n > 0;
        if (!ok) (void)cudaGetLastError();
        k = ok ? 1 : 2;
        slot.store(k, std::memory_order_release);
    }
    return k == 1;
}

// How a product on the main tile (TMA or cp.async-fed) is launched: tiles
// [0, full) as a plain grid, tiles [full, tiles) as clusters of `cs` CTAs that
// split each tile's k-steps (cs == 1: no cluster split).
struct SplitPlan {
    int64_t tiles = 0;
    int64_t full = 0;
    int cs = 1;
    bool narrow = false;  // tiles are the narrow tile's (128 x 64), all of them in clusters of cs
    bool ksplit = false;  // narrow tiles, one CTA each of two warp groups on alternate k-steps (cs == 1)
};

// The k-split tile (ffma_tma_ksplit.cuh) takes TMA products with fewer main
// tiles than SMs whose 128 x 64 tiles fill one round over the SMs to at least
// kKSplitFillPct (70 %), with at most kKSplitMaxSteps (48) k-steps: there it
// beat the narrow tile's cluster plan by 1-22 % on GB300 (1024^3: 52.8
// against 54.0 us; 1024 x 1216 x 1024: 52.8 against 64.3), and lost beyond
// those bounds (96 tiles on 152 SMs; 64 k-steps: 97.7 against 95.5 us).
constexpr int64_t kKSplitFillPct = 70;
constexpr int64_t kKSplitMaxSteps = 48;

// Cost model of the main tile, fitted to measurements on GB300 of products from
// 512 x 512 x 8192 to 8192^3: two CTAs on an SM each advance one k-step per
// unit of time; one CTA alone on an SM advances two (the SM's throughput is
// the same); and each CTA spends kCtaOverheadSteps units outside its k-loop
// (pipeline fill, epilogue, partial-sum exchange), hidden behind the other
// CTA's work when two share the SM.
constexpr double kCtaOverheadSteps = 2.0;

// Time for an SM to run L CTAs of w k-steps each, two at a time and the last
// one alone when L is odd.
double sm_time(int64_t L, double w) {
    return (double)(L / 2) * (w + kCtaOverheadSteps) + (double)(L % 2) * (0.5 * w + kCtaOverheadSteps);
}

// Cost model of the narrow tile in the same units (those of the main tile on
// the same path): an SM advances `steps` of its CTAs' k-steps (each half a
// main k-step of work) per unit while three or more of them are resident,
// `two` times that with two, half with one alone, and spends `round` units per
// round of up to `per_sm` CTAs.  Fitted on GB300 to products with fewer main
// tiles than SMs: 17 of them from 512^3 to 2048 x 2048 x 512 for the TMA path,
// 14 with lda = K + 1 (ldb = N + 1, or N + 4) for the cp.async path.  Over
// those the plan it picks ran within 6 % (TMA) and 3 % (cp.async) of the
// fastest of the main plan and clusters of 2, 4 and 8 narrow CTAs.
struct NarrowModel {
    double steps, two, round;
    int per_sm;
};
constexpr NarrowModel kNarrowTma{4.4, 0.9, 1.25, 4};
constexpr NarrowModel kNarrowCp{5.9, 0.75, 1.5, 3};

// Time for an SM to run L narrow CTAs of w k-steps each.
double narrow_sm_time(const NarrowModel &m, int64_t L, double w) {
    if (L <= 1) return w / (0.5 * m.steps) + m.round;
    if (L == 2) return 2.0 * w / (m.two * m.steps) + m.round;
    return (double)L * w / m.steps + m.round * (double)((L + m.per_sm - 1) / m.per_sm);
}

// Which narrow tile a product may take: none, the TMA kernel's, the cp.async
// kernel's, or the phased TMA kernel's (run, like the TMA kernel's, at four
// CTAs per SM, and planned with its model).
enum class Narrow { kNone, kTma, kCp, kPhased };

// The cluster split fills SMs that a grid would leave idle.  With P SMs, the
// `rem` tiles beyond whole multiples of P (all of them when there are fewer
// than P) are shared by clusters of c = 2, 4 or 8 CTAs -- c chosen by the cost
// model among those leaving at least four 32-deep k-steps per CTA, ties to the
// larger c -- when the estimate beats the plain grid by 4 % or more.  With
// fewer main tiles than SMs, the narrow tile of the product's path (`narrow`)
// in clusters of 2, 4 or 8 (the c with the lowest estimate, ties to the
// larger c) is taken instead when its estimate is lower still.
//
// The model itself touches no device: `sms` is the SM count, `dbg` the
// test-only switches, and fits(narrow, c) says whether clusters of c CTAs of
// the narrow tile (narrow == true) or of the 128 x 128 tile can be resident.
template <class Fits>
SplitPlan split_plan_model(int M, int N, int K, int64_t sms, Narrow narrow, int dbg, Fits fits) {
    using T = TmaTile;
    SplitPlan plan;
    plan.tiles = (int64_t)((M + T::BM - 1) / T::BM) * ((N + T::BN - 1) / T::BN);
    plan.full = plan.tiles;
    const int64_t P = sms;
    const int64_t kt = (K + T::BK - 1) / T::BK;
    if (P <= 0 || plan.tiles == 0) return plan;
    const int forced = (dbg >> kDebugClusterShift) & 15;
    const int64_t rem = plan.tiles % P;
    int64_t full = plan.tiles - rem;
    int cs = 1;
    if (forced) {
        cs = forced;
        if (dbg & kDebugClusterAll) full = 0;
    } else if (rem > 0) {
        const double plain = sm_time((plan.tiles + P - 1) / P, (double)kt);
        double best = plain;
        for (int c = 2; c <= 8 && kt >= 4 * c; c *= 2) {
            const double t = sm_time(full / P, (double)kt) + sm_time((rem * c + P - 1) / P, (double)((kt + c - 1) / c));
            if (t <= best) best = t, cs = c;
        }
        if (cs > 1 && best > 0.96 * plain) cs = 1, best = plain;
        if (narrow != Narrow::kNone && !(dbg & kDebugNoNarrow) && plan.tiles < P) {
            static_assert(TmaNarrow::BM == TmaNarrowCp::BM && TmaNarrow::BN == TmaNarrowCp::BN, "one narrow tile shape");
            using TN = TmaNarrow;
            const NarrowModel &m = narrow == Narrow::kCp ? kNarrowCp : kNarrowTma;
            const int64_t ntiles = (int64_t)((M + TN::BM - 1) / TN::BM) * ((N + TN::BN - 1) / TN::BN);
            static_assert(TmaKSplit::BM == TN::BM && TmaKSplit::BN == TN::BN, "one narrow tile shape");
            if (narrow == Narrow::kTma && ntiles <= P && 100 * ntiles >= kKSplitFillPct * P && kt <= kKSplitMaxSteps) {
                plan.tiles = plan.full = ntiles;
                plan.cs = 1;
                plan.narrow = plan.ksplit = true;
                return plan;
            }
            int ncs = 0;
            double nbest = 0.0;
            for (int c = 2; c <= 8 && kt >= 4 * c; c *= 2) {
                const double t = narrow_sm_time(m, (ntiles * c + P - 1) / P, (double)((kt + c - 1) / c));
                if ((ncs == 0 || t <= nbest) && fits(true, c)) nbest = t, ncs = c;
            }
            if (ncs > 0 && nbest < best) {
                plan.tiles = ntiles;
                plan.full = 0;
                plan.cs = ncs;
                plan.narrow = true;
                return plan;
            }
        }
    }
    if (cs < 2 || cs > 8 || full == plan.tiles) return plan;
    if (!fits(false, cs)) return plan;
    plan.full = full;
    plan.cs = cs;
    return plan;
}

// The plan on the current device: the model with this device's SM count, the
// test-only switches, and cluster sizes checked against the kernel of the
// product's path.
SplitPlan split_plan(int M, int N, int K, const DeviceInfo &info, Narrow narrow, bool phased = false) {
    auto fits = [&](bool narrow_tile, int c) {
        if (narrow_tile)
            return narrow == Narrow::kTma      ? cluster_fits<TmaNarrow>(info.dev, c)
                   : narrow == Narrow::kPhased ? cluster_fits<PhasedNarrow>(info.dev, c)
                                               : cluster_fits<TmaNarrowCp, true>(info.dev, c);
        return phased ? cluster_fits<TmaPhased>(info.dev, c) : cluster_fits<TmaTile>(info.dev, c);
    };
    return split_plan_model(M, N, K, info.sms, narrow, g_debug_flags.load(), fits);
}

// Launch the TMA kernel over grouped tiles [tile_base, tile_base + tiles): a
// plain (tiles x splits) grid, the same as the first of a plain + split pair
// (primary), or tiles clusters of cs CTAs (cs > 1).
template <class T, bool PLAIN>
int launch_tma_as(const Problem &p, float alpha, float beta, bool vc, int splits, float *partials, int ldp,
                  int64_t tile_base, int64_t tiles, int cs, bool primary, cudaStream_t stream, const DeviceInfo &info) {
    alignas(64) CUtensorMap ta, tb;
    if (!encode_2d(&ta, p.A, p.M, p.K, p.lda, T::BM, T::BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tb, p.B, p.K, p.N, p.ldb, T::BK, T::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return SGEMM_ERR_LAUNCH;
    const unsigned long long wait = g_wait_limit_ns.load();
    const int dbg = g_debug_flags.load();
    using sgemm::sgemm_ffma_tma_kernel;
    // the narrow tiles only ever run as clusters
    constexpr bool kClustersOnly = std::is_same_v<T, TmaNarrow> || std::is_same_v<T, TmaNarrowCp>;
    if constexpr (kClustersOnly) {
        if (cs <= 1) return SGEMM_ERR_LAUNCH;
    } else if (cs <= 1) {
        const dim3 grid((unsigned)tiles, (unsigned)splits);
        if (primary) {
            if constexpr (!T::CSPLIT_OK) {
                return SGEMM_ERR_LAUNCH;  // only a tile that supports the cluster split has a split to precede
            } else {
                if (!(vc ? tma_attr<T, true, sgemm::kRolePrimary, PLAIN>(info.dev)
                         : tma_attr<T, false, sgemm::kRolePrimary, PLAIN>(info.dev)))
                    return SGEMM_ERR_LAUNCH;
                auto kernel = vc ? sgemm_ffma_tma_kernel<T, true, sgemm::kRolePrimary, PLAIN>
                                 : sgemm_ffma_tma_kernel<T, false, sgemm::kRolePrimary, PLAIN>;
                kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(ta, tb, p.M, p.N, p.K, alpha, beta, p.C, p.ldc,
                                                                    partials, ldp, (int)tile_base, info.err_word, wait,
                                                                    dbg);
            }
        } else {
            if (!(vc ? tma_attr<T, true, sgemm::kRolePlain, PLAIN>(info.dev)
                     : tma_attr<T, false, sgemm::kRolePlain, PLAIN>(info.dev)))
                return SGEMM_ERR_LAUNCH;
            auto kernel = vc ? sgemm_ffma_tma_kernel<T, true, sgemm::kRolePlain, PLAIN>
                             : sgemm_ffma_tma_kernel<T, false, sgemm::kRolePlain, PLAIN>;
            kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(ta, tb, p.M, p.N, p.K, alpha, beta, p.C, p.ldc,
                                                                partials, ldp, (int)tile_base, info.err_word, wait, dbg);
        }
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
    if constexpr (!T::CSPLIT_OK) {
        return SGEMM_ERR_LAUNCH;
    } else {
        if (!(vc ? tma_attr<T, true, sgemm::kRoleSplit, PLAIN>(info.dev)
                 : tma_attr<T, false, sgemm::kRoleSplit, PLAIN>(info.dev)))
            return SGEMM_ERR_LAUNCH;
        auto kernel =
            vc ? sgemm_ffma_tma_kernel<T, true, sgemm::kRoleSplit, PLAIN>
               : sgemm_ffma_tma_kernel<T, false, sgemm::kRoleSplit, PLAIN>;
        // behind a plain grid of the same product: start on the SMs it frees as it drains
        const bool overlap = tile_base > 0 && !(dbg & kDebugNoOverlap);
        cudaLaunchAttribute attr[2];
        const cudaLaunchConfig_t cfg = split_config<T>(tiles, cs, overlap, stream, attr);
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, p.M, p.N, p.K, alpha, beta, p.C, p.ldc,
                                                 (float *)nullptr, 0, (int)tile_base, info.err_word, wait, dbg);
        return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
}

// Launch the TMA kernel of tile T (see launch_tma_as); the main tile takes its
// PLAIN form when alpha = 1 and beta = 0.
template <class T>
int launch_tma(const Problem &p, float alpha, float beta, bool vc, int splits, float *partials, int ldp,
               int64_t tile_base, int64_t tiles, int cs, bool primary, cudaStream_t stream, const DeviceInfo &info) {
    if constexpr (std::is_same_v<T, TmaTile>) {
        if (alpha == 1.f && beta == 0.f)
            return launch_tma_as<T, true>(p, alpha, beta, vc, splits, partials, ldp, tile_base, tiles, cs, primary,
                                          stream, info);
    }
    return launch_tma_as<T, false>(p, alpha, beta, vc, splits, partials, ldp, tile_base, tiles, cs, primary, stream,
                                   info);
}

// One k-step (K <= 32) with C's rows 16-byte aligned: the small-K tile unrolled
// by four, as a plain grid of `tiles` tiles (its scalar-store form would spill,
// so it is built only with 16-byte C stores).
int launch_smallk1(const Problem &p, float alpha, float beta, int64_t tiles, cudaStream_t stream,
                   const DeviceInfo &info) {
    using T = TmaSmallK1;
    static_assert(T::BM == TmaSmallK::BM && T::BN == TmaSmallK::BN, "one small-K tile shape");
    alignas(64) CUtensorMap ta, tb;
    if (!encode_2d(&ta, p.A, p.M, p.K, p.lda, T::BM, T::BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tb, p.B, p.K, p.N, p.ldb, T::BK, T::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return SGEMM_ERR_LAUNCH;
    if (!tma_attr<T, true, sgemm::kRolePlain>(info.dev)) return SGEMM_ERR_LAUNCH;
    sgemm::sgemm_ffma_tma_kernel<T, true, sgemm::kRolePlain><<<(unsigned)tiles, T::THREADS, T::SMEM_BYTES, stream>>>(
        ta, tb, p.M, p.N, p.K, alpha, beta, p.C, p.ldc, nullptr, 0, 0, info.err_word, g_wait_limit_ns.load(),
        g_debug_flags.load());
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// One k-step (K <= 32), beta == 0 and a C the TMA can address (16-byte aligned
// base and rows, N a multiple of 4): the 8 x 16-per-thread small-K tile whose
// C tile is written by a TMA store, as a plain grid of 128 x 64 tiles.
int launch_smallk_store(const Problem &p, float alpha, cudaStream_t stream, const DeviceInfo &info) {
    using T = sgemm::TmaSmallKStoreTile;
    using S = sgemm::SmallKStore<T>;
    alignas(64) CUtensorMap ta, tb, tc;
    if (!encode_2d(&ta, p.A, p.M, p.K, p.lda, T::BM, T::BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tb, p.B, p.K, p.N, p.ldb, T::BK, T::BN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tc, p.C, p.M, p.N, p.ldc, T::BM, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return SGEMM_ERR_LAUNCH;
    static std::atomic<int> done[kMaxDevices];
    if (!smem_attr_once(done[info.dev], sgemm::sgemm_ffma_tma_smallk_store_kernel<T>, S::SMEM_BYTES))
        return SGEMM_ERR_LAUNCH;
    const int64_t tiles = (int64_t)((p.M + T::BM - 1) / T::BM) * ((p.N + T::BN - 1) / T::BN);
    sgemm::sgemm_ffma_tma_smallk_store_kernel<T><<<(unsigned)tiles, T::THREADS, S::SMEM_BYTES, stream>>>(
        ta, tb, tc, p.M, p.N, p.K, alpha, info.err_word, g_wait_limit_ns.load(), g_debug_flags.load());
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// One round of 128 x 64 tiles on the k-split kernel (ffma_tma_ksplit.cuh):
// one CTA per tile, two groups of warps on alternate k-steps.
int launch_ksplit(const Problem &p, float alpha, float beta, bool vc, int64_t tiles, cudaStream_t stream,
                  const DeviceInfo &info) {
    using T = TmaKSplit;
    alignas(64) CUtensorMap ta, tb;
    if (!encode_2d(&ta, p.A, p.M, p.K, p.lda, T::BM, T::BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tb, p.B, p.K, p.N, p.ldb, T::BK, T::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return SGEMM_ERR_LAUNCH;
    static std::atomic<int> done[kMaxDevices][4];
    using sgemm::sgemm_ffma_tma_ksplit_kernel;
    const bool plain = alpha == 1.f && beta == 0.f;
    auto kernel = plain ? (vc ? sgemm_ffma_tma_ksplit_kernel<T, true, true>
                              : sgemm_ffma_tma_ksplit_kernel<T, false, true>)
                        : (vc ? sgemm_ffma_tma_ksplit_kernel<T, true, false>
                              : sgemm_ffma_tma_ksplit_kernel<T, false, false>);
    if (!smem_attr_once(done[info.dev][(vc ? 1 : 0) + (plain ? 2 : 0)], kernel, T::SMEM_BYTES)) return SGEMM_ERR_LAUNCH;
    kernel<<<(unsigned)tiles, 2 * T::THREADS, T::SMEM_BYTES, stream>>>(ta, tb, p.M, p.N, p.K, alpha, beta, p.C, p.ldc,
                                                                      info.err_word, g_wait_limit_ns.load(),
                                                                      g_debug_flags.load());
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// Launch the phased TMA kernel (operands whose rows are only 4-byte aligned)
// over grouped tiles [tile_base, tile_base + tiles), with the same roles as
// launch_tma.
template <class T>
int launch_phased(const Problem &p, float alpha, float beta, bool vc, int splits, float *partials, int ldp,
                  int64_t tile_base, int64_t tiles, int cs, bool primary, cudaStream_t stream, const DeviceInfo &info) {
    static_assert(IsPhased<T>::value && T::CSPLIT_OK, "a tile read through phase maps");
    alignas(64) sgemm::PhasedMaps maps;
    const int da = encode_phases(maps.a, p.A, p.M, p.K, p.lda, T::A_PHASE_ROWS, T::BK);
    const int db = encode_phases(maps.b, p.B, p.K, p.N, p.ldb, T::B_PHASE_ROWS, T::BN);
    if (da < 0 || db < 0) return SGEMM_ERR_LAUNCH;
    const unsigned long long wait = g_wait_limit_ns.load();
    const int dbg = g_debug_flags.load();
    using sgemm::sgemm_ffma_tma_phased_kernel;
    // the narrow tile only ever runs as clusters
    constexpr bool kClustersOnly = std::is_same_v<T, PhasedNarrow>;
    if constexpr (kClustersOnly) {
        if (cs <= 1) return SGEMM_ERR_LAUNCH;
    } else if (cs <= 1) {
        const dim3 grid((unsigned)tiles, (unsigned)splits);
        if (primary) {
            if (!(vc ? phased_attr<T, true, sgemm::kRolePrimary>(info.dev)
                     : phased_attr<T, false, sgemm::kRolePrimary>(info.dev)))
                return SGEMM_ERR_LAUNCH;
            auto kernel = vc ? sgemm_ffma_tma_phased_kernel<T, true, sgemm::kRolePrimary>
                             : sgemm_ffma_tma_phased_kernel<T, false, sgemm::kRolePrimary>;
            kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(maps, (uint32_t)da, (uint32_t)db, p.M, p.N, p.K, alpha,
                                                                beta, p.C, p.ldc, partials, ldp, (int)tile_base,
                                                                info.err_word, wait, dbg);
        } else {
            if (!(vc ? phased_attr<T, true, sgemm::kRolePlain>(info.dev)
                     : phased_attr<T, false, sgemm::kRolePlain>(info.dev)))
                return SGEMM_ERR_LAUNCH;
            auto kernel = vc ? sgemm_ffma_tma_phased_kernel<T, true, sgemm::kRolePlain>
                             : sgemm_ffma_tma_phased_kernel<T, false, sgemm::kRolePlain>;
            kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(maps, (uint32_t)da, (uint32_t)db, p.M, p.N, p.K, alpha,
                                                                beta, p.C, p.ldc, partials, ldp, (int)tile_base,
                                                                info.err_word, wait, dbg);
        }
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
    if (!(vc ? phased_attr<T, true, sgemm::kRoleSplit>(info.dev) : phased_attr<T, false, sgemm::kRoleSplit>(info.dev)))
        return SGEMM_ERR_LAUNCH;
    auto kernel = vc ? sgemm_ffma_tma_phased_kernel<T, true, sgemm::kRoleSplit>
                     : sgemm_ffma_tma_phased_kernel<T, false, sgemm::kRoleSplit>;
    const bool overlap = tile_base > 0 && !(dbg & kDebugNoOverlap);
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = split_config<T>(tiles, cs, overlap, stream, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, maps, (uint32_t)da, (uint32_t)db, p.M, p.N, p.K, alpha, beta,
                                             p.C, p.ldc, (float *)nullptr, 0, (int)tile_base, info.err_word, wait, dbg);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

template <class T, bool VA, bool VB, int ROLE>
bool cp_packed_attr(int dev) {
    static std::atomic<int> done[kMaxDevices];
    return smem_attr_once(done[dev], sgemm::sgemm_ffma_cp_kernel<T, VA, VB, ROLE>, T::SMEM_BYTES);
}

// The packed cp.async kernel for the given operand alignment and launch role.
template <class T, int ROLE>
bool cp_packed_kernel(bool va, bool vb, int dev,
                      void (*&kernel)(int, int, int, float, const float *, int, const float *, int, float, float *, int,
                                      int, float *, int, int)) {
    if (va && vb) kernel = sgemm::sgemm_ffma_cp_kernel<T, true, true, ROLE>;
    else if (va) kernel = sgemm::sgemm_ffma_cp_kernel<T, true, false, ROLE>;
    else if (vb) kernel = sgemm::sgemm_ffma_cp_kernel<T, false, true, ROLE>;
    else kernel = sgemm::sgemm_ffma_cp_kernel<T, false, false, ROLE>;
    return va ? (vb ? cp_packed_attr<T, true, true, ROLE>(dev) : cp_packed_attr<T, true, false, ROLE>(dev))
              : (vb ? cp_packed_attr<T, false, true, ROLE>(dev) : cp_packed_attr<T, false, false, ROLE>(dev));
}

// Launch the packed cp.async kernel (operands TMA cannot address) over grouped
// tiles [tile_base, tile_base + tiles), with the same roles as launch_tma.
template <class T>
int launch_cp(const Problem &p, float alpha, float beta, bool vc, int splits, float *partials, int ldp,
              int64_t tile_base, int64_t tiles, int cs, bool primary, cudaStream_t stream, const DeviceInfo &info) {
    const bool va = cp_vec_a(p);
    const bool vb = cp_vec_b(p);
    const int dbg = g_debug_flags.load();
    void (*kernel)(int, int, int, float, const float *, int, const float *, int, float, float *, int, int, float *,
                   int, int) = nullptr;
    constexpr bool kClustersOnly = std::is_same_v<T, TmaNarrow> || std::is_same_v<T, TmaNarrowCp>;
    if constexpr (kClustersOnly) {
        if (cs <= 1) return SGEMM_ERR_LAUNCH;
    } else if (cs <= 1) {
        const bool attr = primary ? cp_packed_kernel<T, sgemm::kRolePrimary>(va, vb, info.dev, kernel)
                                  : cp_packed_kernel<T, sgemm::kRolePlain>(va, vb, info.dev, kernel);
        if (!attr) return SGEMM_ERR_LAUNCH;
        const dim3 grid((unsigned)tiles, (unsigned)splits);
        kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(p.M, p.N, p.K, alpha, p.A, p.lda, p.B, p.ldb, beta, p.C,
                                                            p.ldc, vc ? 1 : 0, partials, ldp, (int)tile_base);
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
    if (!cp_packed_kernel<T, sgemm::kRoleSplit>(va, vb, info.dev, kernel)) return SGEMM_ERR_LAUNCH;
    const bool overlap = tile_base > 0 && !(dbg & kDebugNoOverlap);
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = split_config<T>(tiles, cs, overlap, stream, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p.M, p.N, p.K, alpha, p.A, p.lda, p.B, p.ldb, beta, p.C,
                                             p.ldc, vc ? 1 : 0, (float *)nullptr, 0, (int)tile_base);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// Launch the product: on the TMA kernels when the operands allow it (the
// small-K tile for K <= 64), on the phased TMA kernel when their rows are only
// 4-byte aligned (M, K >= 4), otherwise on the cp.async-fed kernel.  splits > 1
// writes partial sums to `partials` (splits slabs of M x ldp) instead of C;
// splits == 1 follows the cluster-split plan.
// Products for which one thread per output beats the tiled kernels' set-up:
// at most kTinyOutputs outputs with at most kTinyK terms each.  Measured on
// GB300 (µs per call, one thread per output against the tiled plan): 6x6x9
// 3.7-4.1 against 6.6; 32x32x64 6.1 against 7.2 (10.3 with odd strides);
// 128x128x128 9.7 against 16.4; 256x128x128 10.2 against 16.4; at K = 256
// the two are even (14.3-16.4) and at K = 512 the tiled plan is twice as fast.
constexpr int kTinyOutputs = 16384;
constexpr int kTinyK = 128;
bool tiny_product(const Problem &p) {
    return (int64_t)p.M * p.N <= kTinyOutputs && p.K <= kTinyK && p.K > 0 && g_tiny_path.load();
}

int launch_product(const Problem &p, int splits, float *partials, int ldp, cudaStream_t stream,
                   const DeviceInfo &info) {
    const bool vc = splits > 1 || (aligned16(p.C) && p.ldc % 4 == 0);
    // partial slabs hold the raw products; alpha and beta act in the reduction
    const float alpha = splits > 1 ? 1.f : p.alpha, beta = splits > 1 ? 0.f : p.beta;
    if (splits == 1 && tiny_product(p)) {
        sgemm::sgemm_ffma_tiny_kernel<<<(unsigned)((p.M * p.N + sgemm::kTinyThreads - 1) / sgemm::kTinyThreads),
                                        sgemm::kTinyThreads, 0, stream>>>(p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, p.C,
                                                                           p.ldc, alpha, beta);
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
    const bool tma = use_tma(p);
    const bool phased = !tma && use_phased(p);
    if (!tma && !phased && !cp_fits(p)) {
        // rows of A more than 2 GiB apart and not 16-byte aligned: the register-
        // tiled kernel of the pages' ladder, which indexes in 64 bits (C = A B;
        // the entry points that get here pass alpha = 1, beta = 0, one split)
        if (splits != 1 || p.alpha != 1.f || p.beta != 0.f || (p.M + 63) / 64 > 65535) return SGEMM_ERR_INVALID_ARG;
        sgemm::ladder_register_kernel<64, 64, 8, 4, 4><<<dim3((p.N + 63) / 64, (p.M + 63) / 64), 256, 0, stream>>>(
            p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, p.C, p.ldc);
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
    if (tma && splits == 1 && p.K <= 2 * TmaSmallK::BK) {
        const int64_t tiles =
            (int64_t)((p.M + TmaSmallK::BM - 1) / TmaSmallK::BM) * ((p.N + TmaSmallK::BN - 1) / TmaSmallK::BN);
        static_assert(sgemm::TmaSmallKStoreTile::BM == TmaSmallK::BM && sgemm::TmaSmallKStoreTile::BN == TmaSmallK::BN,
                      "one small-K tile shape");
        // the TMA store writes a row's right edge in 16-byte units: only rows of a
        // multiple of 4 floats end on a unit boundary (otherwise the store would
        // also write the gap between N and ldc)
        if (p.K <= TmaSmallK1::BK && vc && beta == 0.f && p.N % 4 == 0) return launch_smallk_store(p, alpha, stream, info);
        if (p.K <= TmaSmallK1::BK && vc) return launch_smallk1(p, alpha, beta, tiles, stream, info);
        return launch_tma<TmaSmallK>(p, alpha, beta, vc, 1, partials, ldp, 0, tiles, 1, false, stream, info);
    }
    // grouped tiles [base, base + n) as a (n x s) grid, or n clusters of cs CTAs
    auto launch = [&](int64_t base, int64_t n, int s, int cs, bool primary) {
        return tma      ? launch_tma<TmaTile>(p, alpha, beta, vc, s, partials, ldp, base, n, cs, primary, stream, info)
               : phased ? launch_phased<TmaPhased>(p, alpha, beta, vc, s, partials, ldp, base, n, cs, primary, stream,
                                                   info)
                        : launch_cp<TmaTile>(p, alpha, beta, vc, s, partials, ldp, base, n, cs, primary, stream, info);
    };
    if (splits > 1) {
        const int64_t tiles = (int64_t)((p.M + TmaTile::BM - 1) / TmaTile::BM) * ((p.N + TmaTile::BN - 1) / TmaTile::BN);
        return launch(0, tiles, splits, 1, false);
    }
    const Narrow narrow = tma ? Narrow::kTma
                          : phased ? Narrow::kPhased
                                   : (cp_narrow_fits(p) ? Narrow::kCp : Narrow::kNone);
    const SplitPlan plan = split_plan(p.M, p.N, p.K, info, narrow, phased);
    if (plan.ksplit) return launch_ksplit(p, alpha, beta, vc, plan.tiles, stream, info);
    if (plan.narrow)
        return tma      ? launch_tma<TmaNarrow>(p, alpha, beta, vc, 1, partials, ldp, 0, plan.tiles, plan.cs, false,
                                                stream, info)
               : phased ? launch_phased<PhasedNarrow>(p, alpha, beta, vc, 1, partials, ldp, 0, plan.tiles, plan.cs,
                                                      false, stream, info)
                        : launch_cp<TmaNarrowCp>(p, alpha, beta, vc, 1, partials, ldp, 0, plan.tiles, plan.cs, false,
                                                 stream, info);
    if (plan.full > 0) {
        const int st = launch(0, plan.full, 1, 1, plan.cs > 1);
        if (st != SGEMM_OK || plan.full == plan.tiles) return st;
    }
    return launch(plan.full, plan.tiles - plan.full, 1, plan.cs, false);
}

int launch_reduce(const Problem &p, int splits, const float *partials, int ldp, cudaStream_t stream,
                  const DeviceInfo &info) {
    const int64_t quads = (int64_t)p.M * ((p.N + 3) / 4);
    const int64_t want = (quads + 255) / 256;
    const int blocks = (int)(want < (int64_t)info.sms * 8 ? want : (int64_t)info.sms * 8);
    if (aligned16(p.C) && p.ldc % 4 == 0)
        sgemm::splitk_reduce_kernel<true>
            <<<blocks, 256, 0, stream>>>(p.M, p.N, splits, partials, ldp, p.alpha, p.beta, p.C, p.ldc);
    else
        sgemm::splitk_reduce_kernel<false>
            <<<blocks, 256, 0, stream>>>(p.M, p.N, splits, partials, ldp, p.alpha, p.beta, p.C, p.ldc);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// ---- stream-K (sgemm_f32_streamk)

using StreamKTile = TmaTile;

template <class T, bool VC>
bool streamk_attr(int dev) {
    static std::atomic<int> done[kMaxDevices];
    return smem_attr_once(done[dev], sgemm::sgemm_ffma_tma_streamk_kernel<T, VC>, T::SMEM_BYTES);
}

// CTAs of the stream-K kernel resident at once on this device (SMs x blocks
// per SM), queried once per device; 0 if the query fails.
template <class T>
int64_t streamk_resident(const DeviceInfo &info) {
    static std::atomic<int> per_sm[kMaxDevices];
    int n = per_sm[info.dev].load(std::memory_order_acquire);
    if (n == 0) {
        if (!streamk_attr<T, true>(info.dev) || !streamk_attr<T, false>(info.dev)) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sgemm::sgemm_ffma_tma_streamk_kernel<T, true>,
                                                          T::THREADS, T::SMEM_BYTES) != cudaSuccess ||
            n < 1) {
            (void)cudaGetLastError();
            return 0;
        }
        per_sm[info.dev].store(n, std::memory_order_release);
    }
    return (int64_t)n * info.sms;
}

// How sgemm_f32_streamk runs a product: stream-K over a grid of `ctas` CTAs
// (use == true), or sgemm_f32's own launch (no workspace).  Stream-K is taken
// for TMA-addressable operands with K > 64 (not tiny products) when
//  * sgemm_f32's plan (plain tiles, cluster split, narrow tiles) would start
//    fewer CTAs than the device has SMs -- few output tiles over a long K,
//    where at most eight CTAs can share a tile; or
//  * the product has fewer 128 x 128 tiles than SMs and every resident block
//    gets at least kStreamKMinUnits (tile, k-step) units.
// It then runs every resident block (two per SM).  Measured on GB300
// (TFLOP/s, sgemm_f32 against stream-K at two blocks per SM): 256 x 256 x
// 65536 22.2 / 54.5, 128 x 128 x 131072 5.7 / 46.6, 384 x 384 x 4096 22.5 /
// 28.8, 512 x 512 x 16384 47.1 / 55.6 (26.9 units per block), 1024 x 1024 x
// 4096 48.6 / 50.8 (26.9), 1024 x 1024 x 8192 50.8 / 56.5, 1280 x 1280 x 8192
// 53.7 / 57.9; below the threshold sgemm_f32 holds its own or wins: 1024 x
// 1024 x 2048 44.8 / 41.5 (13.5 units), 1536^3 51.8 / 47.8 (22.7), 768 x 768
// x 4096 49.9 / 47.7 (15.2), 1024^3 39.8 / 32.3 (6.7); with more tiles than
// SMs stream-K was not faster either (2048 x 2048 x 8192 62.4 / 60.7).
constexpr int64_t kStreamKMinUnits = 24;

struct StreamKPlan {
    bool use = false;
    int64_t tiles = 0, ctas = 0;
    size_t counter_bytes = 0, bytes = 0;
};

// The decision and the grid without a device: `sms` SMs, `resident` blocks of
// the stream-K kernel resident at once, `dbg` the test-only switches, fits()
// as for split_plan_model.
template <class Fits>
StreamKPlan streamk_plan_model(int M, int N, int K, int64_t sms, int64_t resident, int dbg, Fits fits) {
    using T = StreamKTile;
    StreamKPlan plan;
    if ((int64_t)M * N == 0 || K <= 2 * TmaSmallK::BK || resident <= 0) return plan;
    plan.tiles = (int64_t)((M + T::BM - 1) / T::BM) * ((N + T::BN - 1) / T::BN);
    const int64_t units = plan.tiles * ((K + T::BK - 1) / T::BK);
    if (!(dbg & kDebugForceStreamK)) {
        const SplitPlan sp = split_plan_model(M, N, K, sms, Narrow::kTma, dbg, fits);
        // (the k-split plan fills at least 70 % of the SMs with one round of
        // tiles, and beat stream-K there: 1024^3)
        const int64_t ctas = sp.ksplit ? sms : sp.narrow ? sp.tiles * sp.cs : sp.full + (sp.tiles - sp.full) * sp.cs;
        const bool long_k = plan.tiles < sms && units >= kStreamKMinUnits * resident;
        if (ctas >= sms && !long_k) return plan;
    }
    const int forced = (dbg >> kDebugStreamKPerSmShift) & 3;
    if (forced > 0 && forced * sms < resident) resident = forced * sms;
    plan.use = true;
    plan.ctas = units < resident ? units : resident;
    plan.counter_bytes = (size_t)((plan.tiles * 4 + 255) / 256 * 256);
    plan.bytes = plan.counter_bytes + (size_t)(2 * plan.ctas) * T::BM * T::BN * 4;
    return plan;
}

StreamKPlan streamk_plan(const Problem &p, const DeviceInfo &info) {
    if (!use_tma(p) || tiny_product(p)) return StreamKPlan{};
    const int64_t resident = streamk_resident<StreamKTile>(info);
    auto fits = [&](bool narrow_tile, int c) {
        return narrow_tile ? cluster_fits<TmaNarrow>(info.dev, c) : cluster_fits<TmaTile>(info.dev, c);
    };
    return streamk_plan_model(p.M, p.N, p.K, info.sms, resident, g_debug_flags.load(), fits);
}

int launch_streamk(const Problem &p, const StreamKPlan &plan, void *workspace, cudaStream_t stream,
                   const DeviceInfo &info) {
    using T = StreamKTile;
    alignas(64) CUtensorMap ta, tb;
    if (!encode_2d(&ta, p.A, p.M, p.K, p.lda, T::BM, T::BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tb, p.B, p.K, p.N, p.ldb, T::BK, T::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return SGEMM_ERR_LAUNCH;
    int *counters = static_cast<int *>(workspace);
    unsigned char *slots = static_cast<unsigned char *>(workspace) + plan.counter_bytes;
    if (cudaMemsetAsync(counters, 0, (size_t)plan.tiles * 4, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    const bool vc = aligned16(p.C) && p.ldc % 4 == 0;
    auto kernel = vc ? sgemm::sgemm_ffma_tma_streamk_kernel<T, true> : sgemm::sgemm_ffma_tma_streamk_kernel<T, false>;
    // cooperative: the CTAs that share a tile wait for one another's partial
    // tiles at the end of their runs, so all of them must be resident at once
    // (the grid is at most the resident count; the launch fails otherwise)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.ctas);
    cfg.blockDim = dim3(T::THREADS);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, p.M, p.N, p.K, p.alpha, p.beta, p.C, p.ldc, counters,
                                             slots, info.err_word, (unsigned long long)g_wait_limit_ns.load(),
                                             g_debug_flags.load());
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

// Byte range [lo, hi) spanned by a rows x cols matrix with leading dimension ld.
void span(const void *ptr, int64_t rows, int64_t cols, int64_t ld, uintptr_t &lo, uintptr_t &hi) {
    lo = reinterpret_cast<uintptr_t>(ptr);
    hi = (rows > 0 && cols > 0) ? lo + (uintptr_t)(((rows - 1) * ld + cols) * (int64_t)sizeof(float)) : lo;
}

bool overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Host-side checks shared by every entry point; nothing here touches the GPU.
int validate(const Problem &p) {
    if (p.M < 0 || p.N < 0 || p.K < 0) return SGEMM_ERR_INVALID_ARG;
    if (p.lda < (p.K > 1 ? p.K : 1) || p.ldb < (p.N > 1 ? p.N : 1) || p.ldc < (p.N > 1 ? p.N : 1))
        return SGEMM_ERR_INVALID_ARG;
    const bool a_nonempty = (int64_t)p.M * p.K > 0, b_nonempty = (int64_t)p.K * p.N > 0;
    const bool c_nonempty = (int64_t)p.M * p.N > 0;
    if ((a_nonempty && !p.A) || (b_nonempty && !p.B) || (c_nonempty && !p.C)) return SGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p.A) | reinterpret_cast<uintptr_t>(p.B) | reinterpret_cast<uintptr_t>(p.C)) & 3u)
        return SGEMM_ERR_INVALID_ARG;
    if (!c_nonempty) return SGEMM_OK;
    // the largest tile grid (the small-K tile's 128 x 64 tiles) must fit gridDim.x
    const int64_t tiles =
        (int64_t)((p.M + TmaSmallK::BM - 1) / TmaSmallK::BM) * ((p.N + TmaSmallK::BN - 1) / TmaSmallK::BN);
    if (tiles > 0x7fffffff) return SGEMM_ERR_INVALID_ARG;
    uintptr_t c0, c1, a0, a1, b0, b1;
    span(p.C, p.M, p.N, p.ldc, c0, c1);
    span(p.A, p.M, p.K, p.lda, a0, a1);
    span(p.B, p.K, p.N, p.ldb, b0, b1);
    if ((a_nonempty && overlap(c0, c1, a0, a1)) || (b_nonempty && overlap(c0, c1, b0, b1))) return SGEMM_ERR_ALIAS;
    return SGEMM_OK;
}

int ld_partials(int N) { return ((N + 3) / 4) * 4; }

int64_t ld4(int n) { return ((int64_t)n + 3) / 4 * 4; }

// Workspace of the FFMA form of sgemm_gemm: room for row-major copies of both
// operands (A -> M x K, B -> K x N, rows padded to 4 floats), used for an
// operand given transposed or not 16-byte aligned (base or leading dimension).
size_t gemm_ffma_workspace(int, int, int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return ((size_t)M * (size_t)ld4(K) + (size_t)K * (size_t)ld4(N)) * sizeof(float);
}

size_t partials_bytes(int M, int N, int splits) {
    if (splits <= 1 || M <= 0 || N <= 0) return 0;
    return (size_t)splits * (size_t)M * (size_t)ld_partials(N) * sizeof(float);
}

// Row length of the split operands in the 3xTF32 workspace (16-byte rows for TMA).
int64_t x3_kpad(int K) { return ((int64_t)K + 3) / 4 * 4; }

// Split count of the 3xTF32 product on 128 x bn tiles: its kernel runs one
// CTA per SM, so a grid of fewer than half as many tiles as SMs has its
// k-steps divided among CTA rows (up to 16, keeping at least eight 16-deep
// k-steps each), and the partial tiles are added in row order by the split-K
// reduction.
int x3_splits(int M, int N, int K, int sms, int bn) {
    using T = X3Tile;
    if (M <= 0 || N <= 0 || K <= 0 || sms <= 0) return 1;
    const int64_t tiles = (int64_t)((M + T::BM - 1) / T::BM) * ((N + bn - 1) / bn);
    const int64_t kt = (K + T::BK - 1) / T::BK;
    if (2 * tiles > sms) return 1;
    int64_t s = sms / tiles;
    if (s > kt / 8) s = kt / 8;
    if (s > 16) s = 16;
    if (s < 2) return 1;
    const int64_t per = (kt + s - 1) / s;  // no empty splits
    return (int)((kt + per - 1) / per);
}

// Tile width of the 3xTF32 product.  With one CTA per SM, a grid of U units
// (tiles x k-parts) takes ceil(U / sms) rounds, and a round of 128 x w tiles
// costs about (w + 128) units per k-step: the copies of a k-step move 128 rows
// of A (hi and lo) whatever the width, and w rows of B.  Fitted to the sweep
// on GB300 (GEMM alone): against the 208-wide tile, 192 is predicted 1.06x /
// 1.19x slower at 8192^3 / 3001 x 4999 x 2047 and measured 1.05x / 1.17x;
// 160 predicted 1.11x / 1.29x, measured 1.12x / 1.29x.  Each width is costed
// with its own k-parts (x3_splits) as rounds x (w + 128) x the k-steps of a
// part; the lowest cost wins, ties to the wider tile.
int x3_width(int M, int N, int K, int sms) {
    using T = X3Tile;
    if (M <= 0 || N <= 0 || K <= 0 || sms <= 0) return T::BN;
    const int64_t tm = (M + T::BM - 1) / T::BM;
    const int64_t kt = (K + T::BK - 1) / T::BK;
    int best = T::BN;
    int64_t best_cost = -1;
    for (int bn : sgemm::kTf32x3Widths) {
        const int s = x3_splits(M, N, K, sms, bn);
        const int64_t units = tm * ((N + bn - 1) / bn) * s;
        const int64_t rounds = (units + sms - 1) / sms;
        const int64_t cost = rounds * (bn + 128) * ((kt + s - 1) / s);
        if (best_cost < 0 || cost < best_cost) best = bn, best_cost = cost;
    }
    return best;
}

int64_t up256(int64_t b) { return (b + 255) / 256 * 256; }

// Workspace of a 3xTF32 product: the split operands (A_hi, A_lo: M x K_pad;
// B_hi^T, B_lo^T: N x K_pad), then the partial tiles of a split-K product.
size_t x3_workspace_bytes(int M, int N, int K, int sms) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const int64_t ops = 4 * x3_kpad(K) * (2 * (int64_t)M + 2 * (int64_t)N);
    return (size_t)(up256(ops) + (int64_t)partials_bytes(M, N, x3_splits(M, N, K, sms, x3_width(M, N, K, sms))));
}

int device_sms() {
    DeviceInfo info;
    return device_info(info) == SGEMM_OK ? info.sms : 0;
}

// The tensor-core part of a 3xTF32 product on 128 x T::BN tiles, from the
// split operands ah, al (M x kp) and bh, bl (N x kp); `partials` is the
// workspace after them.
template <class T>
int launch_3xtf32_gemm(const Problem &p, const float *ah, const float *al, const float *bh, const float *bl,
                       int64_t kp, float *partials, cudaStream_t stream, const DeviceInfo &info) {
    alignas(64) CUtensorMap tah, tal, tbh, tbl;
    const CUtensorMapSwizzle sw = T::ROW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_2d(&tah, ah, p.M, p.K, (int)kp, T::BM, T::BK, sw) ||
        !encode_2d(&tal, al, p.M, p.K, (int)kp, T::BM, T::BK, sw) ||
        !encode_2d(&tbh, bh, p.N, p.K, (int)kp, T::BN, T::BK, sw) ||
        !encode_2d(&tbl, bl, p.N, p.K, (int)kp, T::BN, T::BK, sw))
        return SGEMM_ERR_LAUNCH;
    const bool vc = aligned16(p.C) && p.ldc % 4 == 0;
    static std::atomic<int> done_v[kMaxDevices], done_s[kMaxDevices];
    if (!smem_attr_once(done_v[info.dev], sgemm::sgemm_3xtf32_kernel<T, true>, T::SMEM_BYTES) ||
        (!vc && !smem_attr_once(done_s[info.dev], sgemm::sgemm_3xtf32_kernel<T, false>, T::SMEM_BYTES)))
        return SGEMM_ERR_LAUNCH;
    auto kernel = vc ? sgemm::sgemm_3xtf32_kernel<T, true> : sgemm::sgemm_3xtf32_kernel<T, false>;
    const int64_t tiles = (int64_t)((p.M + T::BM - 1) / T::BM) * ((p.N + T::BN - 1) / T::BN);
    const int splits = x3_splits(p.M, p.N, p.K, info.sms, T::BN);
    // persistent: one CTA per SM (at most one per unit) walks the tiles x splits units
    const int64_t units = tiles * splits;
    const unsigned grid = (unsigned)(units < info.sms ? units : info.sms);
    const int ldp = ld_partials(p.N);
    if (splits > 1) {
        // the kernel writes raw partial tiles; alpha and beta act in the reduction
        sgemm::sgemm_3xtf32_kernel<T, true><<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(
            tah, tal, tbh, tbl, p.M, p.N, p.K, splits, 1.f, 0.f, partials, ldp, partials, ldp, info.err_word,
            g_wait_limit_ns.load(), g_debug_flags.load());
        if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
        return launch_reduce(p, splits, partials, ldp, stream, info);
    }
    kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(tah, tal, tbh, tbl, p.M, p.N, p.K, 1, p.alpha, p.beta, p.C,
                                                        p.ldc, nullptr, 0, info.err_word, g_wait_limit_ns.load(),
                                                        g_debug_flags.load());
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// The launches of a 3xTF32 product: split A, split and transpose B, then the
// tensor-core kernel over 128 x w output tiles (w from x3_width), and for
// small grids the split-K reduction.
int launch_3xtf32(const Problem &p, float *ws, cudaStream_t stream, const DeviceInfo &info) {
    const int64_t kp = x3_kpad(p.K);
    float *ah = ws, *al = ws + (int64_t)p.M * kp;
    float *bh = al + (int64_t)p.M * kp, *bl = bh + (int64_t)p.N * kp;
    // A_hi, A_lo are M x K rows and B_hi, B_lo are N x K rows: a row split of an
    // operand already stored that way, a transposing split otherwise; both in
    // one launch
    auto job = [&](int rows, const float *src, int ld, bool transpose, float *hi, float *lo) {
        sgemm::SplitJob j{src, ld, rows, p.K, hi, lo, (int)kp, transpose ? 1 : 0, 0, 1, 1};
        if (transpose) {
            j.gx = (rows + 31) / 32;  // 32 output rows by 32 k per block
            j.gy = (p.K + 31) / 32;
        } else {
            j.vec = aligned16(src) && ld % 4 == 0;
            j.gx = ((p.K + 3) / 4 + 255) / 256;  // 256 quads of k per block
            j.gy = rows < 65535 ? rows : 65535;   // rows strided by gy
        }
        return j;
    };
    const sgemm::SplitJob ja = job(p.M, p.A, p.lda, p.transa, ah, al);   // A^T stored K x M: transposing
    const sgemm::SplitJob jb = job(p.N, p.B, p.ldb, !p.transb, bh, bl);  // B stored K x N: transposing
    const int64_t blocks = (int64_t)ja.gx * ja.gy + (int64_t)jb.gx * jb.gy;
    if (blocks > 0x7fffffff) return SGEMM_ERR_INVALID_ARG;
    sgemm::split_tf32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(ja, jb);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    float *partials = ws + up256(4 * kp * (2 * (int64_t)p.M + 2 * (int64_t)p.N)) / 4;
    switch (x3_width(p.M, p.N, p.K, info.sms)) {
        case 192: return launch_3xtf32_gemm<sgemm::Tf32x3WidthTile<192>>(p, ah, al, bh, bl, kp, partials, stream, info);
        case 176: return launch_3xtf32_gemm<sgemm::Tf32x3WidthTile<176>>(p, ah, al, bh, bl, kp, partials, stream, info);
        case 160: return launch_3xtf32_gemm<sgemm::Tf32x3WidthTile<160>>(p, ah, al, bh, bl, kp, partials, stream, info);
        case 144: return launch_3xtf32_gemm<sgemm::Tf32x3WidthTile<144>>(p, ah, al, bh, bl, kp, partials, stream, info);
        case 128: return launch_3xtf32_gemm<sgemm::Tf32x3WidthTile<128>>(p, ah, al, bh, bl, kp, partials, stream, info);
        default: return launch_3xtf32_gemm<X3Tile>(p, ah, al, bh, bl, kp, partials, stream, info);
    }
}

// Device address of g_splitk_noalloc_scratch on the current device, looked up
// once per device (the host-side name of the array is only a stand-in).
int noalloc_scratch(float **out) {
    static std::mutex mu;
    static float *ptr[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev]) {
        float *p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_splitk_noalloc_scratch) != cudaSuccess || !p)
            return SGEMM_ERR_DEVICE;
        ptr[dev] = p;
    }
    *out = ptr[dev];
    return SGEMM_OK;
}

}  // namespace

extern "C" {

const char *sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG: bad size, leading dimension, pointer or workspace";
        case SGEMM_ERR_ALIAS: return "SGEMM_ERR_ALIAS: C (or the workspace) overlaps another operand";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: CUDA launch failed";
        case SGEMM_ERR_DEVICE: return "SGEMM_ERR_DEVICE: CUDA device query failed";
        case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a kernel gave up on a bounded wait";
        case SGEMM_ERR_SCRATCH_LIMIT:
            return "SGEMM_ERR_SCRATCH_LIMIT: splits * M * (N rounded up to 4) exceeds the 8,388,608-float static scratch";
        default: return "SGEMM_ERR_UNKNOWN";
    }
}

int sgemm_version(void) { return 102; }

int sgemm_f32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
              cudaStream_t stream) {
    const Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    const int st = validate(p);
    if (st != SGEMM_OK || (int64_t)M * N == 0) return st;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    return launch_product(p, 1, nullptr, 0, stream, info);
}

}  // extern "C"

namespace {

// sgemm_f32_plan's outputs for one product on path `path` (0: TMA operands,
// 1: phased, 2: cp.async); plan_fn(narrow, phased, status) gives the split
// plan of that path (on a device, or from the model alone).
template <class PlanFn>
int report_plan(int M, int N, int K, int path, PlanFn plan_fn, long long *tiles, long long *full_tiles,
                int *cluster_size, int *tile_n) {
    if (!tiles || !full_tiles || !cluster_size || !tile_n || M < 0 || N < 0 || K < 0 || path < 0 || path > 2)
        return SGEMM_ERR_INVALID_ARG;
    *tiles = *full_tiles = 0;
    *cluster_size = 1;
    *tile_n = TmaTile::BN;
    if ((int64_t)M * N == 0) return SGEMM_OK;
    if (tiny_product(Problem{M, N, K, nullptr, 1, nullptr, 1, nullptr, 1})) {
        // one thread per output, in blocks of 256
        *tiles = *full_tiles = ((long long)M * N + sgemm::kTinyThreads - 1) / sgemm::kTinyThreads;
        *tile_n = 0;
        return SGEMM_OK;
    }
    if (K <= 2 * TmaSmallK::BK && K > 0 && path == 0) {
        *tiles = *full_tiles =
            (long long)((M + TmaSmallK::BM - 1) / TmaSmallK::BM) * ((N + TmaSmallK::BN - 1) / TmaSmallK::BN);
        *tile_n = TmaSmallK::BN;
        return SGEMM_OK;
    }
    int st = SGEMM_OK;
    const SplitPlan plan = plan_fn(path == 0 ? Narrow::kTma : path == 1 ? Narrow::kPhased : Narrow::kCp, path == 1, st);
    if (st != SGEMM_OK) return st;
    *tiles = plan.tiles;
    *full_tiles = plan.full;
    *cluster_size = plan.cs;
    *tile_n = plan.narrow ? TmaNarrow::BN : TmaTile::BN;
    return SGEMM_OK;
}

}  // namespace

extern "C" {

int sgemm_f32_plan(int M, int N, int K, int tma_operands, long long *tiles, long long *full_tiles, int *cluster_size,
                   int *tile_n) {
    const int dbg = g_debug_flags.load();
    const bool cp = !tma_operands || (dbg & (kDebugForceCpAsync | kDebugForcePhased)) != 0;
    const bool phased = cp && M >= 4 && K >= 4 && !(dbg & kDebugForceCpAsync);
    auto on_device = [&](Narrow narrow, bool ph, int &st) {
        DeviceInfo info;
        if (device_info(info) != SGEMM_OK) {
            st = SGEMM_ERR_DEVICE;
            return SplitPlan{};
        }
        return split_plan(M, N, K, info, narrow, ph);
    };
    return report_plan(M, N, K, !cp ? 0 : phased ? 1 : 2, on_device, tiles, full_tiles, cluster_size, tile_n);
}

int sgemm_f32_3xtf32_plan_model(int M, int N, int K, int sms, int *tile_n, int *splits) {
    if (!tile_n || !splits || M < 0 || N < 0 || K < 0 || sms < 1) return SGEMM_ERR_INVALID_ARG;
    *tile_n = x3_width(M, N, K, sms);
    *splits = x3_splits(M, N, K, sms, *tile_n);
    return SGEMM_OK;
}

int sgemm_f32_plan_model(int M, int N, int K, int path, int sms, long long *tiles, long long *full_tiles,
                         int *cluster_size, int *tile_n) {
    if (sms < 1) return SGEMM_ERR_INVALID_ARG;
    auto model = [&](Narrow narrow, bool, int &) {
        return split_plan_model(M, N, K, sms, narrow, 0, [](bool, int) { return true; });
    };
    return report_plan(M, N, K, path, model, tiles, full_tiles, cluster_size, tile_n);
}

int sgemm_f32_streamk_plan_model(int M, int N, int K, int sms, int blocks_per_sm, long long *blocks,
                                 size_t *workspace_bytes) {
    if (!blocks || !workspace_bytes || M < 0 || N < 0 || K < 0 || sms < 1 || blocks_per_sm < 1)
        return SGEMM_ERR_INVALID_ARG;
    *blocks = 0;
    *workspace_bytes = 0;
    if (tiny_product(Problem{M, N, K, nullptr, 1, nullptr, 1, nullptr, 1})) return SGEMM_OK;
    const StreamKPlan plan =
        streamk_plan_model(M, N, K, sms, (int64_t)sms * blocks_per_sm, 0, [](bool, int) { return true; });
    if (plan.use) {
        *blocks = plan.ctas;
        *workspace_bytes = plan.bytes;
    }
    return SGEMM_OK;
}

size_t sgemm_f32_splitk_workspace_size(int M, int N, int splits) { return partials_bytes(M, N, splits); }

int sgemm_f32_splitk_suggest(int M, int N, int K, int *splits) {
    if (!splits || M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    *splits = 1;
    if ((int64_t)M * N == 0 || K == 0) return SGEMM_OK;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    // MIN_BLOCKS TMA tiles per SM at a time: split until the (tiles x splits)
    // grid fills the SMs, keeping at least four 32-deep k-steps per split
    const int64_t tiles = (int64_t)((M + TmaTile::BM - 1) / TmaTile::BM) * ((N + TmaTile::BN - 1) / TmaTile::BN);
    const int64_t kt = (K + TmaTile::BK - 1) / TmaTile::BK;
    int64_t s = (int64_t)info.sms * TmaTile::MIN_BLOCKS / (tiles > 0 ? tiles : 1);
    if (s > kt / 4) s = kt / 4;
    if (s > kMaxSplits) s = kMaxSplits;
    *splits = (int)(s < 1 ? 1 : s);
    return SGEMM_OK;
}

int sgemm_f32_splitk(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                     int splits, float *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    int st = validate(p);
    if (st != SGEMM_OK) return st;
    if (splits < 1 || splits > kMaxSplits) return SGEMM_ERR_INVALID_ARG;
    if ((int64_t)M * N == 0) return SGEMM_OK;
    // more splits than k-steps would leave empty slabs: cap at the k-step count
    const int kt = k_tiles(p);
    if (splits > kt) splits = kt > 0 ? kt : 1;
    if (!use_tma(p) && !use_phased(p) && !cp_fits(p)) splits = 1;
    if (splits > 1) {
        const size_t need = partials_bytes(M, N, splits);
        if (!workspace || !aligned16(workspace) || workspace_bytes < need) return SGEMM_ERR_INVALID_ARG;
        const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + need;
        uintptr_t lo, hi;
        span(C, M, N, ldc, lo, hi);
        if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
        span(A, M, K, lda, lo, hi);
        if ((int64_t)M * K > 0 && overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
        span(B, K, N, ldb, lo, hi);
        if ((int64_t)K * N > 0 && overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    }
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    if (splits == 1) return launch_product(p, 1, nullptr, 0, stream, info);
    const int ldp = ld_partials(N);
    st = launch_product(p, splits, workspace, ldp, stream, info);
    if (st != SGEMM_OK) return st;
    return launch_reduce(p, splits, workspace, ldp, stream, info);
}

int sgemm_f32_splitk_noalloc(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                             int ldc, int splits, cudaStream_t stream) {
    const Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    int st = validate(p);
    if (st != SGEMM_OK) return st;
    if (splits < 1 || splits > kMaxSplits) return SGEMM_ERR_INVALID_ARG;
    if ((int64_t)M * N == 0) return SGEMM_OK;
    const int kt = k_tiles(p);
    if (splits > kt) splits = kt > 0 ? kt : 1;
    if (!use_tma(p) && !use_phased(p) && !cp_fits(p)) splits = 1;
    const int ldp = ld_partials(N);
    if (splits > 1 && (long long)splits * M * ldp > kNoallocScratchFloats) return SGEMM_ERR_SCRATCH_LIMIT;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    if (splits == 1) return launch_product(p, 1, nullptr, 0, stream, info);
    float *scratch = nullptr;
    if (noalloc_scratch(&scratch) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    // every (split, row < M, column < N) partial that the reduction adds into C
    // is written by the product kernels first (as NaN by a block that gave up
    // on a wait); the padding columns it also reads are discarded, so nothing
    // needs clearing
    st = launch_product(p, splits, scratch, ldp, stream, info);
    if (st != SGEMM_OK) return st;
    return launch_reduce(p, splits, scratch, ldp, stream, info);
}

size_t sgemm_f32_streamk_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return 0;
    // the plan depends on the operands only through use_tma: size it for
    // 16-byte aligned operands, the only ones stream-K runs on (no pointer is
    // dereferenced)
    alignas(16) static const float aligned_probe[4] = {0.f, 0.f, 0.f, 0.f};
    const Problem p{M, N, K, aligned_probe, (K + 3) / 4 * 4, aligned_probe, (N + 3) / 4 * 4, nullptr, N};
    const StreamKPlan plan = streamk_plan(p, info);
    return plan.use ? plan.bytes : 0;
}

int sgemm_f32_streamk(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                      float *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    const int st = validate(p);
    if (st != SGEMM_OK || (int64_t)M * N == 0) return st;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    const StreamKPlan plan = streamk_plan(p, info);
    if (!plan.use) return launch_product(p, 1, nullptr, 0, stream, info);
    if (!workspace || !aligned16(workspace) || workspace_bytes < plan.bytes) return SGEMM_ERR_INVALID_ARG;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + plan.bytes;
    uintptr_t lo, hi;
    span(C, M, N, ldc, lo, hi);
    if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    span(A, M, K, lda, lo, hi);
    if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    span(B, K, N, ldb, lo, hi);
    if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    return launch_streamk(p, plan, workspace, stream, info);
}

size_t sgemm_f32_3xtf32_workspace_size(int M, int N, int K) { return x3_workspace_bytes(M, N, K, device_sms()); }

int sgemm_f32_3xtf32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                     float *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    const int st = validate(p);
    if (st != SGEMM_OK || (int64_t)M * N == 0) return st;
    if (K > 65535 * 32) return SGEMM_ERR_INVALID_ARG;
    if (K == 0) return sgemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream);  // an empty sum: zeros
    const size_t need = x3_workspace_bytes(M, N, K, device_sms());
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return SGEMM_ERR_INVALID_ARG;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + need;
    uintptr_t lo, hi;
    span(C, M, N, ldc, lo, hi);
    if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    span(A, M, K, lda, lo, hi);
    if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    span(B, K, N, ldb, lo, hi);
    if (overlap(w0, w1, lo, hi)) return SGEMM_ERR_ALIAS;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    return launch_3xtf32(p, workspace, stream, info);
}

int sgemm_f32_ladder(int level, int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                     int ldc, cudaStream_t stream) {
    const Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    const int st = validate(p);
    if (st != SGEMM_OK) return st;
    if (level < SGEMM_LADDER_NAIVE || level > SGEMM_LADDER_REGISTER_2D) return SGEMM_ERR_INVALID_ARG;
    if ((int64_t)M * N == 0) return SGEMM_OK;
    const int rows_per_block = level == SGEMM_LADDER_REGISTER_2D ? 64 : (level == SGEMM_LADDER_NAIVE || level == SGEMM_LADDER_TILED_16) ? 16 : 32;
    if ((M + rows_per_block - 1) / rows_per_block > 65535) return SGEMM_ERR_INVALID_ARG;
    switch (level) {
        case SGEMM_LADDER_NAIVE:
            sgemm::ladder_naive_kernel<<<dim3((N + 15) / 16, (M + 15) / 16), dim3(16, 16), 0, stream>>>(
                M, N, K, A, lda, B, ldb, C, ldc);
            break;
        case SGEMM_LADDER_TILED_16:
            sgemm::ladder_tiled_kernel<16, 0><<<dim3((N + 15) / 16, (M + 15) / 16), dim3(16, 16), 0, stream>>>(
                M, N, K, A, lda, B, ldb, C, ldc);
            break;
        case SGEMM_LADDER_TILED_32:
            sgemm::ladder_tiled_kernel<32, 0><<<dim3((N + 31) / 32, (M + 31) / 32), dim3(32, 32), 0, stream>>>(
                M, N, K, A, lda, B, ldb, C, ldc);
            break;
        case SGEMM_LADDER_TILED_32_PADDED:
            sgemm::ladder_tiled_kernel<32, 1><<<dim3((N + 31) / 32, (M + 31) / 32), dim3(32, 32), 0, stream>>>(
                M, N, K, A, lda, B, ldb, C, ldc);
            break;
        default:
            sgemm::ladder_register_kernel<64, 64, 8, 4, 4><<<dim3((N + 63) / 64, (M + 63) / 64), 256, 0, stream>>>(
                M, N, K, A, lda, B, ldb, C, ldc);
    }
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

size_t sgemm_gemm_workspace_size(int algo, int transa, int transb, int M, int N, int K) {
    if (algo == SGEMM_ALGO_3XTF32) return x3_workspace_bytes(M, N, K, device_sms());
    return gemm_ffma_workspace(transa, transb, M, N, K);
}

int sgemm_gemm(int algo, int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda,
               const float *B, int ldb, float beta, float *C, int ldc, float *workspace, size_t workspace_bytes,
               cudaStream_t stream) {
    if ((algo != SGEMM_ALGO_FFMA && algo != SGEMM_ALGO_3XTF32) || (transa != SGEMM_OP_N && transa != SGEMM_OP_T) ||
        (transb != SGEMM_OP_N && transb != SGEMM_OP_T))
        return SGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    // stored shapes of A and B
    const int a_rows = transa ? K : M, a_cols = transa ? M : K;
    const int b_rows = transb ? N : K, b_cols = transb ? K : N;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1) || ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_ARG;
    const bool a_nonempty = (int64_t)M * K > 0, b_nonempty = (int64_t)K * N > 0, c_nonempty = (int64_t)M * N > 0;
    if ((a_nonempty && !A) || (b_nonempty && !B) || (c_nonempty && !C)) return SGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 3u)
        return SGEMM_ERR_INVALID_ARG;
    if (!c_nonempty) return SGEMM_OK;
    const int64_t tiles = (int64_t)((M + TmaSmallK::BM - 1) / TmaSmallK::BM) * ((N + TmaSmallK::BN - 1) / TmaSmallK::BN);
    if (tiles > 0x7fffffff || K > 65535 * 32 || (transb && N > 65535 * 32)) return SGEMM_ERR_INVALID_ARG;
    uintptr_t c0, c1, a0, a1, b0, b1;
    span(C, M, N, ldc, c0, c1);
    span(A, a_rows, a_cols, lda, a0, a1);
    span(B, b_rows, b_cols, ldb, b0, b1);
    if ((a_nonempty && overlap(c0, c1, a0, a1)) || (b_nonempty && overlap(c0, c1, b0, b1))) return SGEMM_ERR_ALIAS;

    DeviceInfo info;
    if (alpha == 0.f || K == 0) {
        // nothing to multiply: C = beta * C (A and B are not read)
        if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
        const int64_t want = ((int64_t)M * N + 255) / 256;
        const int blocks = (int)(want < (int64_t)info.sms * 8 ? want : (int64_t)info.sms * 8);
        sgemm::scale_kernel<<<blocks, 256, 0, stream>>>(M, N, beta, C, ldc);
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }
    // the FFMA form needs its workspace only for transposed operands, and for
    // operands whose rows are not 16-byte aligned when M or K is below 4 (from
    // four rows up the phased TMA kernel reads them where they are)
    const bool small = M < 4 || K < 4;
    const bool a_copy = transa || (small && (!aligned16(A) || lda % 4 != 0));
    const bool b_copy = transb || (small && (!aligned16(B) || ldb % 4 != 0));
    const size_t need = algo == SGEMM_ALGO_3XTF32 || a_copy || b_copy
                            ? sgemm_gemm_workspace_size(algo, transa, transb, M, N, K)
                            : 0;
    if (need > 0) {
        if (!workspace || !aligned16(workspace) || workspace_bytes < need) return SGEMM_ERR_INVALID_ARG;
        const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + need;
        if (overlap(w0, w1, c0, c1) || (a_nonempty && overlap(w0, w1, a0, a1)) ||
            (b_nonempty && overlap(w0, w1, b0, b1)))
            return SGEMM_ERR_ALIAS;
    }
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;

    Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    p.alpha = alpha;
    p.beta = beta;
    if (algo == SGEMM_ALGO_3XTF32) {
        p.transa = transa == SGEMM_OP_T;
        p.transb = transb == SGEMM_OP_T;
        return launch_3xtf32(p, workspace, stream, info);
    }
    // FFMA: transposed operands are first copied row-major into the workspace,
    // and (below four rows) operands whose base or rows are not 16-byte aligned
    // are copied there with padded rows, so that the product runs on the
    // TMA-fed kernel
    float *w = workspace;
    if (a_copy) {
        const int ld = (int)ld4(K);
        if (transa)
            sgemm::transpose_kernel<<<dim3((M + 31) / 32, (K + 31) / 32), 256, 0, stream>>>(K, M, A, lda, w, ld);
        else if (cudaMemcpy2DAsync(w, (size_t)ld * sizeof(float), A, (size_t)lda * sizeof(float),
                                   (size_t)K * sizeof(float), M, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        p.A = w;
        p.lda = ld;
    }
    w = workspace + (int64_t)M * ld4(K);
    if (b_copy) {
        const int ld = (int)ld4(N);
        if (transb)
            sgemm::transpose_kernel<<<dim3((K + 31) / 32, (N + 31) / 32), 256, 0, stream>>>(N, K, B, ldb, w, ld);
        else if (cudaMemcpy2DAsync(w, (size_t)ld * sizeof(float), B, (size_t)ldb * sizeof(float),
                                   (size_t)N * sizeof(float), K, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        p.B = w;
        p.ldb = ld;
    }
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return launch_product(p, 1, nullptr, 0, stream, info);
}

// ---------------------------------------------------------------- host buffers, pipelined

namespace {

// B is copied in up to kHostBChunks column blocks so that the first row panel's
// products can start on the first block instead of waiting for all of B.
constexpr int kHostBChunks = 8;

struct HostPlan {
    int rows;          // rows of C per panel (a multiple of the 128-row tile)
    int panels;
    int chunks;                        // column blocks of B (whole 128-column tiles each)
    int chunk_c0[kHostBChunks + 1];    // first column of each block; chunk_c0[chunks] = N
    int64_t lda_d;     // device row pitch of the A panels (floats)
    int64_t ldn_d;     // device row pitch of B and of the C panels
    size_t b_bytes, a_bytes, c_bytes, total;
};

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Panel height: about M / panels rows, rounded up to whole waves of output
// tiles (the panels run one after another, so a panel that ends in a partly
// filled wave leaves SMs idle at every panel boundary).
HostPlan host_plan(int M, int N, int K, int panels, int sms) {
    HostPlan h{};
    if (panels < 1) panels = 1;
    const int64_t tiles_n = (N + TmaTile::BN - 1) / TmaTile::BN;
    const int64_t slots = (int64_t)(sms > 0 ? sms : 1) * TmaTile::MIN_BLOCKS;
    const int64_t wave_rows = (int64_t)TmaTile::BM * (slots / gcd64(slots, tiles_n > 0 ? tiles_n : 1));
    int64_t rows = ((int64_t)M + panels - 1) / panels;
    rows = (rows + wave_rows - 1) / wave_rows * wave_rows;
    if (rows > M) rows = M;
    if (rows < 1) rows = 1;
    h.rows = (int)rows;
    h.panels = (int)((M + rows - 1) / rows);
    // column blocks of B for the first panel: the first two just wide enough
    // that the first panel's product over one still gives every SM a tile, then
    // doubling widths (each block's copy is shorter than the product over the
    // block before it, and wide blocks run at two CTAs per SM), the last one
    // taking the rest
    const int64_t tiles_m0 = (rows + TmaTile::BM - 1) / TmaTile::BM;
    const int64_t fill = ((int64_t)(sms > 0 ? sms : 1) + tiles_m0 - 1) / tiles_m0;
    int64_t w = fill < 1 ? 1 : fill;
    int64_t t0 = 0;
    h.chunks = 0;
    while (t0 < tiles_n && h.chunks < kHostBChunks) {
        h.chunk_c0[h.chunks++] = (int)(t0 * TmaTile::BN);
        int64_t width = h.chunks <= 2 ? w : w << (h.chunks - 2);
        if (h.chunks == kHostBChunks || t0 + width > tiles_n) width = tiles_n - t0;
        t0 += width;
    }
    if (h.chunks == 0) h.chunk_c0[h.chunks++] = 0;
    h.chunk_c0[h.chunks] = N;
    h.lda_d = ld4(K);
    h.ldn_d = ld4(N);
    h.b_bytes = (size_t)K * h.ldn_d * sizeof(float);
    h.a_bytes = (size_t)rows * h.lda_d * sizeof(float);
    h.c_bytes = (size_t)rows * h.ldn_d * sizeof(float);
    // B once, two A panels and two C panels (double buffering), each 256-byte aligned
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    h.total = up(h.b_bytes) + 2 * up(h.a_bytes) + 2 * up(h.c_bytes);
    return h;
}

// The host pipeline's events, created on a thread's first call for a device
// and reused by its later calls there: a stream wait takes the event's latest
// record at the moment it is enqueued, so recording the same event again in a
// later call is safe.  They live until the process exits.
constexpr int kHostEvents = 1 + kHostBChunks + 8;

int host_events(int dev, cudaEvent_t *&out) {
    struct Pool {
        cudaEvent_t ev[kHostEvents];
        bool ready = false;
    };
    thread_local Pool pool[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    Pool &p = pool[dev];
    if (!p.ready) {
        for (int i = 0; i < kHostEvents; ++i) {
            if (cudaEventCreateWithFlags(&p.ev[i], cudaEventDisableTiming) != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(p.ev[j]);
                return SGEMM_ERR_LAUNCH;
            }
        }
        p.ready = true;
    }
    out = p.ev;
    return SGEMM_OK;
}

}  // namespace

size_t sgemm_f32_host_workspace_size(int M, int N, int K, int panels) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return 0;
    return host_plan(M, N, K, panels, info.sms).total;
}

int sgemm_f32_host(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                   int panels, float *workspace, size_t workspace_bytes, cudaStream_t stream,
                   cudaStream_t h2d_stream, cudaStream_t d2h_stream) {
    if (M < 0 || N < 0 || K < 0 || panels < 1) return SGEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_ARG;
    if (((int64_t)M * K > 0 && !A) || ((int64_t)K * N > 0 && !B) || ((int64_t)M * N > 0 && !C))
        return SGEMM_ERR_INVALID_ARG;
    if ((int64_t)M * N == 0) return SGEMM_OK;
    if (K == 0) {
        // an empty sum: zero the host rows directly
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) C[i * ldc + j] = 0.f;
        return SGEMM_OK;
    }
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    const HostPlan h = host_plan(M, N, K, panels, info.sms);
    if (!workspace || !aligned16(workspace) || workspace_bytes < h.total) return SGEMM_ERR_INVALID_ARG;

    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    char *base = reinterpret_cast<char *>(workspace);
    float *dB = reinterpret_cast<float *>(base);
    float *dA[2] = {reinterpret_cast<float *>(base + up(h.b_bytes)),
                    reinterpret_cast<float *>(base + up(h.b_bytes) + up(h.a_bytes))};
    float *dC[2] = {reinterpret_cast<float *>(base + up(h.b_bytes) + 2 * up(h.a_bytes)),
                    reinterpret_cast<float *>(base + up(h.b_bytes) + 2 * up(h.a_bytes) + up(h.c_bytes))};

    // events: call start; each column block of B landed; A panel landed; A
    // panel consumed; C panel ready; C panel copied out
    cudaEvent_t *ev = nullptr;
    int st = host_events(info.dev, ev);
    cudaEvent_t ev_start = nullptr, *ev_b = nullptr, *ev_a = nullptr, *ev_a_free = nullptr, *ev_c = nullptr,
                *ev_c_free = nullptr;
    if (st == SGEMM_OK) {
        ev_start = ev[0];
        ev_b = ev + 1;
        ev_a = ev + 1 + kHostBChunks;
        ev_a_free = ev_a + 2;
        ev_c = ev_a + 4;
        ev_c_free = ev_a + 6;
    }
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && st == SGEMM_OK) st = SGEMM_ERR_LAUNCH;
        return st == SGEMM_OK;
    };
    if (st == SGEMM_OK) {
        // everything already queued on `stream` (an earlier call on the same
        // workspace included) comes before this call's copies
        ok(cudaEventRecord(ev_start, stream));
        ok(cudaStreamWaitEvent(h2d_stream, ev_start, 0));
        ok(cudaStreamWaitEvent(d2h_stream, ev_start, 0));
    }
    // the first A panel, then B in column blocks (the first panel's products
    // follow the blocks as they land), then the other A panels
    auto copy_a = [&](int p) {
        const int b = p & 1;
        const int r0 = p * h.rows;
        const int rows = (M - r0) < h.rows ? (M - r0) : h.rows;
        // copy A rows r0 .. r0 + rows - 1 once the product two panels back has read its buffer
        if (p >= 2) ok(cudaStreamWaitEvent(h2d_stream, ev_a_free[b], 0));
        ok(cudaMemcpy2DAsync(dA[b], h.lda_d * sizeof(float), A + (int64_t)r0 * lda, (size_t)lda * sizeof(float),
                             (size_t)K * sizeof(float), rows, cudaMemcpyHostToDevice, h2d_stream));
        ok(cudaEventRecord(ev_a[b], h2d_stream));
    };
    if (st == SGEMM_OK) copy_a(0);
    for (int j = 0; j < h.chunks && st == SGEMM_OK; ++j) {
        const int c0 = h.chunk_c0[j];
        const int cols = h.chunk_c0[j + 1] - c0;
        ok(cudaMemcpy2DAsync(dB + c0, h.ldn_d * sizeof(float), B + c0, (size_t)ldb * sizeof(float),
                             (size_t)cols * sizeof(float), K, cudaMemcpyHostToDevice, h2d_stream));
        ok(cudaEventRecord(ev_b[j], h2d_stream));
    }
    for (int p = 0; p < h.panels && st == SGEMM_OK; ++p) {
        const int b = p & 1;
        const int r0 = p * h.rows;
        const int rows = (M - r0) < h.rows ? (M - r0) : h.rows;
        if (p >= 1) copy_a(p);
        // the product, once its A panel has landed and its C buffer has been copied out
        ok(cudaStreamWaitEvent(stream, ev_a[b], 0));
        if (p >= 2) ok(cudaStreamWaitEvent(stream, ev_c_free[b], 0));
        if (st != SGEMM_OK) break;
        // panel 0: one product per column block of B, each once its block has
        // landed; later panels: one product over all of B (every block has landed)
        const int parts = p == 0 ? h.chunks : 1;
        for (int j = 0; j < parts && st == SGEMM_OK; ++j) {
            const int c0 = p == 0 ? h.chunk_c0[j] : 0;
            const int cols = p == 0 ? h.chunk_c0[j + 1] - c0 : N;
            if (p == 0) ok(cudaStreamWaitEvent(stream, ev_b[j], 0));
            if (st != SGEMM_OK) break;
            const Problem prob{rows, cols, K, dA[b], (int)h.lda_d, dB + c0, (int)h.ldn_d, dC[b] + c0, (int)h.ldn_d};
            const int ls = launch_product(prob, 1, nullptr, 0, stream, info);
            if (ls != SGEMM_OK) st = ls;
        }
        if (st != SGEMM_OK) break;
        ok(cudaEventRecord(ev_a_free[b], stream));
        ok(cudaEventRecord(ev_c[b], stream));
        // copy the C panel back to the host rows
        ok(cudaStreamWaitEvent(d2h_stream, ev_c[b], 0));
        ok(cudaMemcpy2DAsync(C + (int64_t)r0 * ldc, (size_t)ldc * sizeof(float), dC[b], h.ldn_d * sizeof(float),
                             (size_t)N * sizeof(float), rows, cudaMemcpyDeviceToHost, d2h_stream));
        ok(cudaEventRecord(ev_c_free[b], d2h_stream));
    }
    // `stream` completes only after the last copy out (and the copy streams' work)
    if (st == SGEMM_OK) {
        const int last = (h.panels - 1) & 1;
        ok(cudaStreamWaitEvent(stream, ev_c_free[last], 0));
        if (h.panels >= 2) ok(cudaStreamWaitEvent(stream, ev_c_free[last ^ 1], 0));
    }
    return st;
}

int sgemm_device_status(cudaStream_t stream) {
    DeviceInfo info;
    if (device_info(info) != SGEMM_OK) return SGEMM_ERR_DEVICE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SGEMM_ERR_DEVICE;
    int code = 0;
    if (cudaMemcpy(&code, info.err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SGEMM_ERR_DEVICE;
    if (code != 0) {
        const int zero = 0;
        if (cudaMemcpy(info.err_word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return SGEMM_ERR_DEVICE;
        return SGEMM_ERR_TIMEOUT;
    }
    return SGEMM_OK;
}

int sgemm_test_tiny_path(int enable) {
    const char *on = std::getenv("SGEMM_TEST_SWITCHES");
    if (!on || std::strcmp(on, "1") != 0 || (enable != 0 && enable != 1)) return SGEMM_ERR_INVALID_ARG;
    g_tiny_path.store(enable);
    return SGEMM_OK;
}

int sgemm_test_switches(int flags, unsigned long long wait_limit_ns) {
    const char *on = std::getenv("SGEMM_TEST_SWITCHES");
    if (!on || std::strcmp(on, "1") != 0) return SGEMM_ERR_INVALID_ARG;
    if (flags < 0 || wait_limit_ns == 0) return SGEMM_ERR_INVALID_ARG;
    g_debug_flags.store(flags);
    g_wait_limit_ns.store(wait_limit_ns);
    return SGEMM_OK;
}

}  // extern "C"

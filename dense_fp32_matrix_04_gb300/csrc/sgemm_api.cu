// The C interface of libsgemm: argument checks, variant choice and launch.
// Declarations and the full contract are in include/sgemm.h.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/sgemm.h"
#include "ffma_sgemm.cuh"
#include "ffma_tma_sgemm.cuh"

// Device error word: kernels that give up on a bounded wait record a code here;
// sgemm_device_status() reads and clears it.  One instance per device context.
__device__ int g_sgemm_device_error;

namespace {

using sgemm::FfmaTile;

// 128 x 128 CTA tile, 16-deep k-steps, 4 pipeline stages, 2 CTAs per SM.
using MainTile = FfmaTile<128, 128, 16, 4, 2>;

constexpr int kMaxDevices = 64;

// test-only switches (sgemm_debug_set); bit 0 is read by the TMA kernel
constexpr int kDebugForceCpAsync = 2;
std::atomic<int> g_debug_flags{0};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

struct DeviceInfo {
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
// box_rows x box_cols; OOB elements read as zero.
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

using TmaMain = sgemm::TmaMainTile;

template <bool VC>
int launch_tma(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
               cudaStream_t stream, const DeviceInfo &info, int dev) {
    using T = TmaMain;
    alignas(64) CUtensorMap ta, tb;
    if (!encode_2d(&ta, A, M, K, lda, T::BM, T::BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tb, B, K, N, ldb, T::BK, T::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return SGEMM_ERR_LAUNCH;
    auto kernel = sgemm::sgemm_ffma_tma_kernel<T, VC>;
    static std::atomic<int> done[kMaxDevices];
    if (!done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        done[dev].store(1, std::memory_order_release);
    }
    const int64_t tiles = (int64_t)((M + T::BM - 1) / T::BM) * ((N + T::BN - 1) / T::BN);
    kernel<<<(unsigned)tiles, T::THREADS, T::SMEM_BYTES, stream>>>(ta, tb, M, N, K, C, ldc, info.err_word,
                                                                   g_wait_limit_ns.load(), g_debug_flags.load());
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

// Per device and per kernel instantiation: has the dynamic shared-memory limit been raised?
template <class T, bool VB, bool VC>
std::atomic<int> &smem_attr_done(int dev) {
    static std::atomic<int> done[kMaxDevices];
    return done[dev];
}

template <class T, bool VB, bool VC>
int launch_ffma(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    auto kernel = sgemm::sgemm_ffma_kernel<T, VB, VC>;
    std::atomic<int> &done = smem_attr_done<T, VB, VC>(dev);
    if (!done.load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) !=
            cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        done.store(1, std::memory_order_release);
    }
    const int64_t tiles = (int64_t)((M + T::BM - 1) / T::BM) * ((N + T::BN - 1) / T::BN);
    kernel<<<(unsigned)tiles, T::THREADS, T::SMEM_BYTES, stream>>>(M, N, K, A, lda, B, ldb, C, ldc);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte range [lo, hi) spanned by a rows x cols matrix with leading dimension ld.
void span(const void *p, int64_t rows, int64_t cols, int64_t ld, uintptr_t &lo, uintptr_t &hi) {
    lo = reinterpret_cast<uintptr_t>(p);
    hi = (rows > 0 && cols > 0) ? lo + (uintptr_t)(((rows - 1) * ld + cols) * (int64_t)sizeof(float)) : lo;
}

bool overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

}  // namespace

extern "C" {

const char *sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG: bad size, leading dimension or pointer";
        case SGEMM_ERR_ALIAS: return "SGEMM_ERR_ALIAS: C overlaps A or B";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: CUDA launch failed";
        case SGEMM_ERR_DEVICE: return "SGEMM_ERR_DEVICE: CUDA device query failed";
        case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a kernel gave up on a bounded wait";
        default: return "SGEMM_ERR_UNKNOWN";
    }
}

int sgemm_version(void) { return 100; }

int sgemm_f32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
              cudaStream_t stream) {
    // ---- host-side checks; nothing below touches the GPU until they pass
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_ARG;
    const bool a_nonempty = (int64_t)M * K > 0, b_nonempty = (int64_t)K * N > 0, c_nonempty = (int64_t)M * N > 0;
    if ((a_nonempty && !A) || (b_nonempty && !B) || (c_nonempty && !C)) return SGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 3u)
        return SGEMM_ERR_INVALID_ARG;
    if (!c_nonempty) return SGEMM_OK;
    const int64_t tiles = (int64_t)((M + MainTile::BM - 1) / MainTile::BM) * ((N + MainTile::BN - 1) / MainTile::BN);
    if (tiles > 0x7fffffff) return SGEMM_ERR_INVALID_ARG;
    uintptr_t c0, c1, a0, a1, b0, b1;
    span(C, M, N, ldc, c0, c1);
    span(A, M, K, lda, a0, a1);
    span(B, K, N, ldb, b0, b1);
    if ((a_nonempty && overlap(c0, c1, a0, a1)) || (b_nonempty && overlap(c0, c1, b0, b1))) return SGEMM_ERR_ALIAS;

    // ---- variant
    const bool vb = aligned16(B) && (ldb % 4 == 0);
    const bool vc = aligned16(C) && (ldc % 4 == 0);
    const bool va = aligned16(A) && (lda % 4 == 0);
    if (K > 0 && va && vb && !(g_debug_flags.load() & kDebugForceCpAsync)) {
        // TMA-fed kernel: needs 16-byte aligned bases and row strides
        DeviceInfo info;
        int dev = 0;
        if (device_info(info) != SGEMM_OK || cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_DEVICE;
        return vc ? launch_tma<true>(M, N, K, A, lda, B, ldb, C, ldc, stream, info, dev)
                  : launch_tma<false>(M, N, K, A, lda, B, ldb, C, ldc, stream, info, dev);
    }
    if (vb && vc) return launch_ffma<MainTile, true, true>(M, N, K, A, lda, B, ldb, C, ldc, stream);
    if (vb) return launch_ffma<MainTile, true, false>(M, N, K, A, lda, B, ldb, C, ldc, stream);
    if (vc) return launch_ffma<MainTile, false, true>(M, N, K, A, lda, B, ldb, C, ldc, stream);
    return launch_ffma<MainTile, false, false>(M, N, K, A, lda, B, ldb, C, ldc, stream);
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

int sgemm_debug_set(int flags, unsigned long long wait_limit_ns) {
    if (flags < 0 || wait_limit_ns == 0) return SGEMM_ERR_INVALID_ARG;
    g_debug_flags.store(flags);
    g_wait_limit_ns.store(wait_limit_ns);
    return SGEMM_OK;
}

}  // extern "C"

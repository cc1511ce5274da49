// Thin inline-PTX wrappers used by the SGEMM kernels (sm_103a).
#pragma once

#include <cstdint>

namespace sgemm {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 4-byte asynchronous global->shared copy; src_bytes == 0 zero-fills the slot
// without reading global memory (the masked load of a boundary tile).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// 16-byte asynchronous copy that bypasses L1; bytes src_bytes..15 are zero-filled.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void stg128(float *p, float a, float b, float c, float d) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}


// ---------------------------------------------------------------- packed FP32 pairs (sm_100+)

// Two FP32 values in one 64-bit register pair: low half = first value.
__device__ __forceinline__ uint64_t f32x2_dup(float a) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};\n" : "=l"(r) : "f"(a));
    return r;
}
__device__ __forceinline__ float2 f32x2_unpack(uint64_t v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
// d = a * b + d on both halves, each an IEEE round-to-nearest single-precision FMA.
__device__ __forceinline__ void f32x2_fma(uint64_t &d, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;\n" : "+l"(d) : "l"(a), "l"(b));
}

// ---------------------------------------------------------------- thread-block clusters (sm_90+)

// Rank of this CTA in its cluster, and the cluster's CTA count (1 and 0 when
// the launch has no cluster dimension).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
    return r;
}
// Index of this CTA's cluster along x in the grid.
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;\n" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster arrives (release) and waits
// (acquire): shared-memory writes made before it are visible to the other
// CTAs' distributed shared-memory reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Address, in the cluster's shared window, of the word at CTA-local shared
// address `addr` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ ulonglong2 dsmem_ld_v2u64(uint32_t cluster_addr) {
    ulonglong2 v;
    asm volatile("ld.shared::cluster.v2.u64 {%0, %1}, [%2];\n" : "=l"(v.x), "=l"(v.y) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// ---------------------------------------------------------------- programmatic dependent launch (sm_90+)

// Let the next grid in the stream, if it was launched with programmatic stream
// serialization, start once every CTA of this grid has passed this point.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n");
}
// Wait until the grids this one may overlap have completed and their memory
// operations are visible (returns at once when there are none).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier / TMA (sm_90+)

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// One non-blocking probe of the phase with the given parity; true once it has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Bounded wait: gives up after `limit_ns` of wall time or 2^30 probes, whichever
// comes first, and reports whether the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t probe = 1; probe < (1u << 30); ++probe) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((probe & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// 2-D tiled TMA load of the box at (x, y) (x innermost) into shared memory,
// completing `bytes` of transaction count on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tensor_map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            dst),
        "l"(tensor_map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const void *tensor_map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(tensor_map) : "memory");
}

}  // namespace sgemm

// ptx.cuh -- thin inline-PTX wrappers for sm_103a: shared-memory barriers
// (mbarrier), the tensor-memory accelerator (cp.async.bulk.tensor), the global
// nanosecond timer and packed FP32x2 fused multiply-add.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace sg {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA) and other threads.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// The barrier operations take the barrier either as a pointer or as its
// 32-bit shared-window address (`_at` forms), which keeps a kernel's barrier
// addresses in one 32-bit register each.
__device__ __forceinline__ void mbar_arrive_at(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) { mbar_arrive_at(smem_addr(bar)); }

__device__ __forceinline__ void mbar_arrive_expect_tx_at(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    mbar_arrive_expect_tx_at(smem_addr(bar), bytes);
}

// true once the phase with the given parity has completed
__device__ __forceinline__ bool mbar_try_wait_at(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    return mbar_try_wait_at(smem_addr(bar), parity);
}

// Bounded wait: spins on try_wait and gives up after `timeout_ns` of global time.
// Returns false on expiry.  The clock is read only after a failed try, so the
// fast path costs one try_wait.
__device__ __forceinline__ bool mbar_wait_at(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait_at(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_at(bar, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    return mbar_wait_at(smem_addr(bar), parity, timeout_ns);
}

// Shared-memory data access by 32-bit shared-window address (the memory
// clobber keeps them in program order with the warp's other shared accesses).
__device__ __forceinline__ void sts128(uint32_t addr, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ float lds32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Thread-block clusters: this CTA's rank, a full barrier of the cluster
// (release / acquire: shared-memory writes before it are visible to every CTA
// of the cluster after it), the cluster-window address of the same shared
// variable in CTA `rank`, and a 32-bit load through such an address.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Volatile 32-bit shared-memory flag access by shared-window address.
__device__ __forceinline__ int ld_shared_flag(uint32_t addr) {
    int v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_flag(uint32_t addr, int v) {
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------- async copies
// 4-byte asynchronous copy global -> shared; with src_bytes 0 nothing is read
// and the destination is zero-filled.  Completion: cp_async_commit groups the
// copies issued since the last commit, cp_async_wait<n> waits until at most n
// groups of this thread are pending.
__device__ __forceinline__ void cp_async4(uint32_t smem_dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- TMA
// Bring the 128-byte line that holds `ptr` into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes on `bar`.
// x is the innermost (contiguous) coordinate; it must be a multiple of 4 floats.
__device__ __forceinline__ void tma_load_2d_at(uint32_t smem_dst, const CUtensorMap *map,
                                               uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
// 3-D form: (x, y) as above and z the batch.
__device__ __forceinline__ void tma_load_3d_at(uint32_t smem_dst, const CUtensorMap *map,
                                               uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    tma_load_2d_at(smem_addr(smem_dst), map, smem_addr(bar), x, y);
}

// ---------------------------------------------------------------- FP32x2
// d = a * b + c on both lanes, round to nearest even (one instruction on sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    return __ffma2_rn(a, b, c);
}

}  // namespace sg

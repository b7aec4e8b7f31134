// tf32x3_pair.cuh -- the 3xTF32 GEMM on a pair of SMs per tile (a 2-CTA
// cluster, tcgen05 `cta_group::2`).  Same split and the same three MMAs per
// 8-deep k step as tf32x3.cuh, but one MMA covers a 256 x 256 tile of the pair:
// each CTA holds 128 rows of A and half of B's columns in its shared memory,
// the MMA (issued by CTA 0) reads both CTAs' halves, and each CTA's TMEM
// receives its 128 rows x 256 columns of the accumulator.  Per SM a 16-deep
// stage is 32 KB instead of 48 KB, so the ring holds 6 stages: the copies have
// about three times as long to arrive as in the single-CTA kernel, whose MMAs
// wait for them.
//
// Roles (256 threads per CTA, one CTA per SM):
//   warp 0    both CTAs: thread 0 copies its CTA's A_hi, A_lo (128 x 16) and
//             B_hi, B_lo halves (128 x 16) into its own ring; the copies signal
//             CTA 0's full barrier, which counts both CTAs' bytes;
//   warp 1    both CTAs allocate TMEM (512 columns, the pair's collective
//             allocation); in CTA 0 thread 32 issues the MMAs and commits each
//             stage to the empty barriers of both CTAs, each finished tile to
//             both CTAs' accumulator barriers;
//   warps 4-7 both CTAs: the epilogue of the CTA's 128 rows, as in tf32x3.cuh;
//             each warp hands the accumulator back on CTA 0's barrier.
// Every barrier wait is bounded; an expiry sets the abort flag of both CTAs.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "tf32x3.cuh"

namespace sg {
namespace t3 {

constexpr int P_BM = 256, P_BN = 256;       // the pair's tile
constexpr int P_ROWS = 128;                  // A rows and B columns (rows of B^T) per CTA
constexpr int P_STAGES = 6;
constexpr int P_A = P_ROWS * BK;             // floats of A_hi (or A_lo) per CTA and stage: 8 KB
constexpr int P_B = P_ROWS * BK;             // floats of B_hi (or B_lo) per CTA and stage: 8 KB
constexpr int P_STAGE_FLOATS = 2 * P_A + 2 * P_B;
constexpr uint32_t P_STAGE_BYTES = P_STAGE_FLOATS * 4u;                    // 32 KB
constexpr uint32_t P_STAGE_BYTES_HALF = P_STAGE_BYTES - uint32_t(P_B) * 4u;  // B halves of 64 rows
constexpr size_t P_SMEM_BYTES =
    size_t(P_STAGES) * P_STAGE_BYTES + size_t(EPI_FLOATS) * 4 + 1024 + 256;
static_assert(P_SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(P_SMEM_BYTES > 232448 / 2, "one CTA per SM");

// Instruction descriptor of the pair's MMA: D f32, A and B tf32 K-major,
// M = 256 (128 rows in each CTA), N = 256; and N = 128 for half-width tiles.
constexpr uint32_t P_IDESC = (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(P_BN >> 3) << 17) |
                             (uint32_t(P_BM >> 4) << 24);
constexpr uint32_t P_IDESC_HALF = (P_IDESC & ~(0x3Fu << 17)) | (uint32_t((P_BN / 2) >> 3) << 17);

// Arrive (with an expected byte count) on a barrier of either CTA of the pair.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
                     bar),
                 "r"(bytes)
                 : "memory");
}
// 2-D tile copy into this CTA's shared memory whose completion (bytes) is
// counted on a barrier of either CTA of the pair (`cta_group::2`: here CTA 0's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const CUtensorMap *map,
                                                 uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
// Bounded wait on a barrier of this CTA with cluster-scope acquire: what the
// other CTA (or its copies) did before arriving is visible afterwards.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    const uint32_t a = smem_addr(bar);
    auto try_once = [&] {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        return done != 0;
    };
    if (try_once()) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (try_once()) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}
__device__ __forceinline__ void st_cluster_flag(uint32_t addr, int v) {
    asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_cluster_u32(uint32_t addr) {
    int v;
    asm volatile("ld.relaxed.cluster.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D (both CTAs' TMEM) = A * B (+ D): A and B halves from both CTAs' shared memory
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this shared offset in both CTAs when every MMA
// this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"((unsigned short)3)
        : "memory");
}

// Work of pair q (of Q pairs): its whole 256 x 256 tiles t = q, q + Q, ...
// below `full`, then, when the last partial wave holds at most Q/2 tiles, that
// wave cut into 256 x 128 tiles h = q, q + Q, ... below 2 * (tiles - full).
struct PairPlan {
    int full, halves, mine_full, mine;

    __device__ void init(const Params &p) {
        const int Q = gridDim.x / 2, q = blockIdx.x / 2;
        const int tiles = p.tiles_m * p.tiles_n;
        const int tail = tiles % Q;
        full = (tail != 0 && 2 * tail <= Q) ? tiles - tail : tiles;
        halves = 2 * (tiles - full);
        mine_full = q < full ? (full - 1 - q) / Q + 1 : 0;
        const int mine_half = q < halves ? (halves - 1 - q) / Q + 1 : 0;
        mine = mine_full + mine_half;
    }

    __device__ void item(const Params &p, int j, int &tm, int &col0, int &ncols) const {
        const int Q = gridDim.x / 2, q = blockIdx.x / 2;
        int tn;
        if (j < mine_full) {
            tile_coords(q + j * Q, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            col0 = tn * P_BN;
            ncols = P_BN;
        } else {
            const int h = q + (j - mine_full) * Q;
            tile_coords(full + h / 2, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            col0 = tn * P_BN + (h & 1) * (P_BN / 2);
            ncols = P_BN / 2;
        }
    }
};


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    sgemm_3xtf32_pair_kernel(const __grid_constant__ CUtensorMap tmAh,
                             const __grid_constant__ CUtensorMap tmAl,
                             const __grid_constant__ CUtensorMap tmBh,
                             const __grid_constant__ CUtensorMap tmBl,
                             const __grid_constant__ CUtensorMap tmBh2,
                             const __grid_constant__ CUtensorMap tmBl2, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    float *ring = reinterpret_cast<float *>(base);
    float *epi = ring + P_STAGES * P_STAGE_FLOATS;
    uint64_t *full = reinterpret_cast<uint64_t *>(epi + EPI_FLOATS);
    uint64_t *empty = full + P_STAGES;
    uint64_t *acc_full = empty + P_STAGES;   // [2] MMA -> epilogue (both CTAs)
    uint64_t *acc_empty = acc_full + 2;      // [2] epilogue -> MMA (CTA 0's)
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base + 1);
    volatile int *issued_slot = abort_flag + 1;   // stages this CTA's producer filled

    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(&full[s], 2);    // CTA 0's counts one arrival, with bytes, per CTA
            mbar_init(&empty[s], 1);   // the MMA commit, multicast to both CTAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 2 * EPI_WARPS);   // CTA 0's: both CTAs' epilogue warps
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *issued_slot = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_base, TMEM_COLS);
    tc_fence_before();
    cluster_barrier();   // both CTAs' barriers, flags and TMEM exist before any remote use
    tc_fence_after();
    const uint32_t taddr = *tmem_base;
    const uint32_t peer_abort = dsmem_map(smem_addr((const void *)abort_flag), rank ^ 1u);
    auto set_abort = [&] {
        *abort_flag = 1;
        st_cluster_flag(peer_abort, 1);
    };

    PairPlan plan;
    plan.init(p);
    const int my_tiles = plan.mine;
    const int k_tiles = (p.K + BK - 1) / BK;

    if (warp == 0) {
        // ================================================================ copies (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tmAh);
            tma_prefetch_desc(&tmAl);
            tma_prefetch_desc(&tmBh);
            tma_prefetch_desc(&tmBl);
            tma_prefetch_desc(&tmBh2);
            tma_prefetch_desc(&tmBl2);
            const uint32_t ring_s = smem_addr(ring);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
                int tm, col0, ncols;
                plan.item(p, j, tm, col0, ncols);
                const bool half = ncols != P_BN;
                const int arow = tm * P_BM + int(rank) * P_ROWS;      // this CTA's rows of A
                const int brow = col0 + int(rank) * (ncols / 2);     // its columns of B
                for (int kb = 0; kb < k_tiles; ++kb) {
                    if (*abort_flag) break;
                    // first use of a stage: parity 1 counts as complete
                    if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns)) {
                        atomicOr(&g_error_word, ERR_EMPTY_WAIT);
                        set_abort();
                        break;
                    }
                    const uint32_t st = ring_s + uint32_t(stage * P_STAGE_FLOATS) * 4u;
                    const uint32_t fb = dsmem_map(smem_addr(&full[stage]), 0u);
                    mbar_arrive_expect_tx_cluster(fb, half ? P_STAGE_BYTES_HALF : P_STAGE_BYTES);
                    tma_load_2d_pair(st, &tmAh, fb, kb * BK, arow);
                    tma_load_2d_pair(st + uint32_t(P_A) * 4u, &tmAl, fb, kb * BK, arow);
                    tma_load_2d_pair(st + uint32_t(2 * P_A) * 4u, half ? &tmBh2 : &tmBh, fb, kb * BK,
                                   brow);
                    tma_load_2d_pair(st + uint32_t(2 * P_A + P_B) * 4u, half ? &tmBl2 : &tmBl, fb,
                                   kb * BK, brow);
                    ++issued;
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            *issued_slot = issued;
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer (CTA 0)
        if (lane == 0 && rank == 0) {
            const uint32_t ring_s = smem_addr(ring);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                const int a = j & 1;
                // both CTAs' epilogues have handed this accumulator back (first use: free)
                if (!mbar_wait_cluster(&acc_empty[a], (uint32_t(j >> 1) & 1u) ^ 1u, p.timeout_ns)) {
                    atomicOr(&g_error_word, ERR_EMPTY_WAIT);
                    set_abort();
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = taddr + uint32_t(a) * ACC_COLS;
                int tm_unused, col_unused, ncols;
                plan.item(p, j, tm_unused, col_unused, ncols);
                const uint32_t idesc = ncols == P_BN ? P_IDESC : P_IDESC_HALF;
                for (int kb = 0; kb < k_tiles; ++kb) {
                    if (*abort_flag || !mbar_wait_cluster(&full[stage], phase, p.timeout_ns)) {
                        if (!*abort_flag) atomicOr(&g_error_word, ERR_FULL_WAIT);
                        set_abort();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ah = ring_s + uint32_t(stage * P_STAGE_FLOATS) * 4u;
                    const uint32_t al = ah + uint32_t(P_A) * 4u;
                    const uint32_t bh = ah + uint32_t(2 * P_A) * 4u;
                    const uint32_t bl = bh + uint32_t(P_B) * 4u;
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint32_t off = uint32_t(kk) * 32u;   // 8 tf32 = 32 bytes along K
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        mma_tf32_pair(d, smem_desc_sw(al + off), smem_desc_sw(bh + off), idesc, acc);
                        mma_tf32_pair(d, smem_desc_sw(ah + off), smem_desc_sw(bl + off), idesc, 1u);
                        mma_tf32_pair(d, smem_desc_sw(ah + off), smem_desc_sw(bh + off), idesc, 1u);
                    }
                    mma_commit_pair(&empty[stage]);   // both CTAs' stage free once read
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit_pair(&acc_full[a]);   // the tile's accumulators are complete
            }
            if (!ok) {
                // no MMA may still run when either CTA frees its TMEM or exits
                mma_commit_pair(drain);
                if (!mbar_wait(drain, 0u, drain_limit_ns(p.timeout_ns)))
                    atomicOr(&g_error_word, ERR_DRAIN_WAIT);
            }
        }
    } else if (warp >= 4) {
        // ================================================================ epilogue (both CTAs)
        const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
        float *buf = epi + quarter * (32 * 33);
        const float alpha = p.alpha, beta = p.beta;
        for (int j = 0; j < my_tiles; ++j) {
            const int a = j & 1;
            if (__any_sync(0xffffffffu, *abort_flag)) break;
            bool ready = mbar_wait(&acc_full[a], uint32_t(j >> 1) & 1u, p.timeout_ns);
            ready = __all_sync(0xffffffffu, ready);
            if (!ready) {
                if (lane == 0) {
                    atomicOr(&g_error_word, ERR_FULL_WAIT);
                    set_abort();
                }
                break;
            }
            tc_fence_after();
            int tm, col0, ncols;
            plan.item(p, j, tm, col0, ncols);
            const int row0 = tm * P_BM + int(rank) * P_ROWS + quarter * 32;
            const uint32_t src = taddr + uint32_t(a) * ACC_COLS + (uint32_t(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < ncols / 32; ++c) {
                float v[32];
                __syncwarp();   // tcgen05.ld is warp-collective; buf reuse
                // range-checked build: the 32 columns lie in this accumulator
                if (!SG_IN_RANGE(a * ACC_COLS + c * 32 + 32 <= TMEM_COLS && c * 32 + 32 <= ACC_COLS))
                    break;
                tmem_load32(src + uint32_t(c * 32), v);
                if (c == ncols / 32 - 1) {
                    // all of this accumulator is in registers: hand it back to CTA 0
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(dsmem_map(smem_addr(&acc_empty[a]), 0u));
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) buf[lane * 33 + i] = v[i];
                __syncwarp();
                const int col = col0 + c * 32 + lane;
                const bool col_ok = col < p.N;
                float cin[32];
#pragma unroll
                for (int r = 0; r < 32; ++r)
                    cin[r] = (beta != 0.0f && col_ok && row0 + r < p.M)
                                 ? __ldcs(p.C + (long long)(row0 + r) * p.ldc + col)
                                 : 0.0f;
                if (col_ok) {
#pragma unroll
                    for (int r = 0; r < 32; ++r) {
                        if (row0 + r < p.M &&
                            SG_IN_RANGE(row0 + r >= tm * P_BM && row0 + r < (tm + 1) * P_BM &&
                                        col >= col0 && col < col0 + ncols)) {
                            const float x = buf[r * 33 + lane];
                            p.C[(long long)(row0 + r) * p.ldc + col] =
                                (beta != 0.0f) ? fmaf(alpha, x, beta * cin[r]) : alpha * x;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_barrier();   // CTA 0's MMAs and both CTAs' remote arrivals are done
    // After an abort, copies of either producer may still be writing its CTA's
    // ring, and they count on CTA 0's full barriers, which only CTA 0 can wait
    // on.  Every abort was set in both CTAs before the barrier above, so both
    // take this branch or neither.  CTA 0 completes the arrivals of stages
    // that only one producer filled (the other, which never arrived, expects
    // no bytes there), waits until the last P_STAGES fillings have landed, and
    // the second cluster barrier keeps CTA 1 resident until then.
    if (*abort_flag) {
        if (rank == 0 && threadIdx.x == 0) {
            const int mine = *issued_slot;
            const int peer = ld_cluster_u32(dsmem_map(smem_addr((const void *)issued_slot), 1u));
            const int lo = mine < peer ? mine : peer, hi = mine < peer ? peer : mine;
            // a producer runs at most P_STAGES fillings ahead of the MMAs, which
            // consume only stages both filled, so hi - lo <= P_STAGES
            for (int q = lo; q < hi; ++q) mbar_arrive(&full[q % P_STAGES]);
            for (int q = hi > P_STAGES ? hi - P_STAGES : 0; q < hi; ++q)
                if (!mbar_wait_cluster(&full[q % P_STAGES], uint32_t((q / P_STAGES) & 1),
                                       drain_limit_ns(p.timeout_ns))) {
                    atomicOr(&g_error_word, ERR_DRAIN_WAIT);
                    break;
                }
        }
        cluster_barrier();
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(taddr, TMEM_COLS);
}

}  // namespace t3
}  // namespace sg

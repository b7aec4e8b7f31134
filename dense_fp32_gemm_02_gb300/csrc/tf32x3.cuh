// tf32x3.cuh -- FP32 GEMM on the 5th-generation tensor cores by the 3xTF32
// split: every fp32 operand x is written as x = hi + lo with hi = tf32(x) and
// lo = tf32(x - hi); the product A*B is taken as
//     A_hi*B_hi + A_hi*B_lo + A_lo*B_hi
// (the dropped A_lo*B_lo term is below 2^-22 of |A||B|), each a TF32 MMA with
// fp32 accumulation in tensor memory.  Per product the relative error is about
// 3 * 2^-22, inside the FP32 tolerance 1e-6*K*|alpha|*sum|A||B| for every K.
//
// Kernel layout (persistent: one CTA per SM walks 128 x 256 output tiles
// b, b + gridDim.x, ...; a last wave of at most half the SMs is cut into
// 128 x 128 tiles, one per SM; 256 threads):
//   warp 0    thread 0 issues TMA copies of A_hi, A_lo (128 x 16) and B_hi,
//             B_lo (256 x 16, B transposed so both operands are K-major) into
//             a 4-stage ring, 64-byte swizzled;
//   warp 1    allocates all 512 TMEM columns (two 128 x 256 fp32
//             accumulators); thread 32 issues tcgen05.mma (M 128, N 256, K 8)
//             three times per 8-wide k step into the tile's accumulator and
//             commits each stage back to the producer through its empty barrier;
//   warps 4-7 read a finished accumulator from TMEM (32 lanes each), hand it
//             back, and apply alpha/beta on the way to C, staged through
//             shared memory for coalesced rows -- while the MMAs of the next
//             tile already run in the other accumulator.
// Every barrier wait is bounded; after an expiry the CTA stops issuing,
// waits (bounded) for its copies and MMAs in flight, and always frees TMEM.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace sg {
namespace t3 {

constexpr int BM = 128, BN = 256, BK = 16, STAGES = 4;
// K-major operand rows of BK floats: 64 bytes, so the TMA box and the MMA
// descriptor both use the 64-byte swizzle; 8-row groups are 8 x 64 bytes apart.
constexpr int ROW_BYTES = BK * 4;
static_assert(ROW_BYTES == 64 || ROW_BYTES == 128, "64- or 128-byte swizzle rows");
constexpr uint32_t SWIZZLE_CODE = ROW_BYTES == 128 ? 2u : 4u;   // descriptor layout field
constexpr int A_TILE = BM * BK;                       // floats, 8 KB
constexpr int B_TILE = BN * BK;                       // floats, 16 KB
constexpr int STAGE_FLOATS = 2 * A_TILE + 2 * B_TILE; // A_hi, A_lo, B_hi, B_lo
constexpr uint32_t STAGE_BYTES = STAGE_FLOATS * 4u;   // 48 KB
constexpr uint32_t STAGE_BYTES_HALF = STAGE_BYTES - uint32_t(B_TILE) * 4u;   // B boxes of BN/2 rows
constexpr int THREADS = 256;
constexpr int EPI_WARPS = 4;                          // warps 4..7
constexpr uint32_t ACC_COLS = 256;                    // 128 lanes x 256 fp32 columns
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;          // two accumulators: all of TMEM
constexpr int EPI_FLOATS = EPI_WARPS * 32 * 33;       // per-warp 32 x 33 staging blocks
// ring + staging + 1 KB alignment slack + barriers; more than half the SM's
// shared memory, so one CTA per SM and the whole TMEM is this CTA's
constexpr size_t SMEM_BYTES = size_t(STAGES) * STAGE_BYTES + size_t(EPI_FLOATS) * 4 + 1024 + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM");

// Instruction descriptor of tcgen05.mma.kind::tf32: D f32, A and B tf32, both
// K-major, N = 256, M = 128.
constexpr uint32_t IDESC = (1u << 4)                    // D format: f32
                           | (2u << 7)                  // A format: tf32
                           | (2u << 10)                 // B format: tf32
                           | (uint32_t(BN >> 3) << 17)  // N / 8
                           | (uint32_t(BM >> 4) << 24); // M / 16
// The same with N = 128, for the half-width tiles of the last wave.
constexpr uint32_t IDESC_HALF = (IDESC & ~(0x3Fu << 17)) | (uint32_t((BN / 2) >> 3) << 17);

// Shared-memory matrix descriptor: K-major operand, rows of ROW_BYTES with the
// matching swizzle (the layout the TMA writes), 8-row groups 8 rows apart.
__device__ __forceinline__ uint64_t smem_desc_sw(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);           // start address, 16-byte units
    d |= uint64_t(1) << 16;                           // leading offset (unused: K fits one row)
    d |= uint64_t((8 * ROW_BYTES) >> 4) << 32;        // stride between 8-row groups
    d |= uint64_t(1) << 46;                           // descriptor version
    d |= uint64_t(SWIZZLE_CODE) << 61;                // 64- or 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D (tmem) = A * B (+ D when accumulate != 0)
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tf32 rounding (round to nearest, ties away from zero) of an fp32 value.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t t;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(x));
    return __uint_as_float(t);
}

__device__ __forceinline__ void split(float x, float &hi, float &lo) {
    hi = to_tf32(x);
    // x - hi is exact in fp32; a non-finite x keeps everything in hi
    lo = isfinite(x) ? to_tf32(x - hi) : 0.0f;
}

struct Params {
    float *C;
    long long ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n, group_m;
    unsigned long long timeout_ns;
};

// Work of CTA b: its whole tiles t = b, b + G, ... below `full`, then, when
// the last partial wave holds at most G/2 tiles, that wave cut into
// half-width tiles (BM x BN/2) h = b, b + G, ... below 2 * (tiles - full), so
// the last wave takes half as long.  Item j of the CTA: tile coordinates, the
// first output column and the width (BN or BN/2).
struct WorkPlan {
    int full;      // whole tiles
    int halves;    // half-width tiles after them
    int mine_full, mine;

    __device__ void init(const Params &p) {
        const int G = gridDim.x, b = blockIdx.x;
        const int tiles = p.tiles_m * p.tiles_n;
        const int tail = tiles % G;
        full = (tail != 0 && 2 * tail <= G) ? tiles - tail : tiles;
        halves = 2 * (tiles - full);
        mine_full = b < full ? (full - 1 - b) / G + 1 : 0;
        const int mine_half = b < halves ? (halves - 1 - b) / G + 1 : 0;
        mine = mine_full + mine_half;
    }

    __device__ void item(const Params &p, int j, int &tm, int &col0, int &ncols) const {
        int tn;
        if (j < mine_full) {
            tile_coords(blockIdx.x + j * gridDim.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            col0 = tn * BN;
            ncols = BN;
        } else {
            const int h = blockIdx.x + (j - mine_full) * gridDim.x;
            tile_coords(full + h / 2, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            col0 = tn * BN + (h & 1) * (BN / 2);
            ncols = BN / 2;
        }
    }
};

__global__ void __launch_bounds__(THREADS, 1)
    sgemm_3xtf32_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                        const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                        const __grid_constant__ CUtensorMap tmBh2,
                        const __grid_constant__ CUtensorMap tmBl2,
                        const Params p) {
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    float *ring = reinterpret_cast<float *>(base);
    float *epi = ring + STAGES * STAGE_FLOATS;
    uint64_t *full = reinterpret_cast<uint64_t *>(epi + EPI_FLOATS);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;     // [2] MMA -> epilogue
    uint64_t *acc_empty = acc_full + 2;      // [2] epilogue -> MMA
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *tmem_base;

    WorkPlan plan;
    plan.init(p);
    const int my_tiles = plan.mine;
    const int k_tiles = (p.K + BK - 1) / BK;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmAh);
            tma_prefetch_desc(&tmAl);
            tma_prefetch_desc(&tmBh);
            tma_prefetch_desc(&tmBl);
            tma_prefetch_desc(&tmBh2);
            tma_prefetch_desc(&tmBl2);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
                int tm, col0, ncols;
                plan.item(p, j, tm, col0, ncols);
                for (int kb = 0; kb < k_tiles; ++kb) {
                    if (*abort_flag) break;
                    // first use of a stage: parity 1 counts as complete
                    if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns)) {
                        atomicOr(&g_error_word, ERR_EMPTY_WAIT);
                        *abort_flag = 1;
                        break;
                    }
                    float *st = ring + stage * STAGE_FLOATS;
                    mbar_arrive_expect_tx(&full[stage], ncols == BN ? STAGE_BYTES : STAGE_BYTES_HALF);
                    tma_load_2d(st, &tmAh, &full[stage], kb * BK, tm * BM);
                    tma_load_2d(st + A_TILE, &tmAl, &full[stage], kb * BK, tm * BM);
                    // a half-width tile copies BN/2-row boxes of B (tmBh2, tmBl2) into
                    // the first half of each B region
                    const bool half = ncols != BN;
                    tma_load_2d(st + 2 * A_TILE, half ? &tmBh2 : &tmBh, &full[stage], kb * BK, col0);
                    tma_load_2d(st + 2 * A_TILE + B_TILE, half ? &tmBl2 : &tmBl, &full[stage],
                                kb * BK, col0);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // after an abort: let the copies already issued land before exit
            if (*abort_flag) {
                for (long long q = (issued > STAGES ? issued - STAGES : 0); q < issued; ++q)
                    if (!mbar_wait(&full[q % STAGES], uint32_t((q / STAGES) & 1),
                                   drain_limit_ns(p.timeout_ns))) {
                        atomicOr(&g_error_word, ERR_DRAIN_WAIT);
                        break;
                    }
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t ring_s = smem_addr(ring);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                const int a = j & 1;
                // the epilogue has handed this accumulator back (first use: free)
                if (!mbar_wait(&acc_empty[a], (uint32_t(j >> 1) & 1u) ^ 1u, p.timeout_ns)) {
                    atomicOr(&g_error_word, ERR_EMPTY_WAIT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = taddr + uint32_t(a) * ACC_COLS;
                int tm_unused, col_unused, ncols;
                plan.item(p, j, tm_unused, col_unused, ncols);
                const uint32_t idesc = ncols == BN ? IDESC : IDESC_HALF;
                for (int kb = 0; kb < k_tiles; ++kb) {
                    if (*abort_flag || !mbar_wait(&full[stage], phase, p.timeout_ns)) {
                        if (!*abort_flag) atomicOr(&g_error_word, ERR_FULL_WAIT);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ah = ring_s + uint32_t(stage * STAGE_FLOATS) * 4u;
                    const uint32_t al = ah + A_TILE * 4u;
                    const uint32_t bh = ah + 2u * A_TILE * 4u;
                    const uint32_t bl = bh + B_TILE * 4u;
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint32_t off = uint32_t(kk) * 32u;   // 8 tf32 = 32 bytes along K
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        mma_tf32(d, smem_desc_sw(al + off), smem_desc_sw(bh + off), idesc, acc);
                        mma_tf32(d, smem_desc_sw(ah + off), smem_desc_sw(bl + off), idesc, 1u);
                        mma_tf32(d, smem_desc_sw(ah + off), smem_desc_sw(bh + off), idesc, 1u);
                    }
                    mma_commit(&empty[stage]);     // stage free once these MMAs have read it
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit(&acc_full[a]);  // this tile's accumulator is complete
            }
            if (!ok) {
                // no MMA may still run when TMEM is freed
                mma_commit(drain);
                if (!mbar_wait(drain, 0u, drain_limit_ns(p.timeout_ns)))
                    atomicOr(&g_error_word, ERR_DRAIN_WAIT);
            }
        }
    } else if (warp >= 4) {
        // ================================================================ epilogue
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
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
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            int tm, col0, ncols;
            plan.item(p, j, tm, col0, ncols);
            const int row0 = tm * BM + quarter * 32;
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
                    // all of this accumulator is in registers: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[a]);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) buf[lane * 33 + i] = v[i];
                __syncwarp();
                // row r of the block: lane = column; C rows read and written
                // 128 contiguous bytes at a time, all 32 loads in flight first
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
                            SG_IN_RANGE(row0 + r >= tm * BM && row0 + r < (tm + 1) * BM &&
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
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(taddr, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ split pre-pass
// A (M x K, row pitch lda) -> Ah, Al (M x K, row pitch ldk): same layout, K-major.
// Each thread keeps 16 floats in flight: 4 float4 when `vec4` (A 16-byte
// aligned, lda and K multiples of 4), else 16 scalars; a block covers 4096
// consecutive floats of a row per step.
__global__ void __launch_bounds__(256)
    split_a_kernel(const float *__restrict__ A, long long lda, int M, int K, float *__restrict__ Ah,
                   float *__restrict__ Al, long long ldk, int vec4) {
    for (long long m = blockIdx.y; m < M; m += gridDim.y) {
        const float *src = A + m * lda;
        float *dh = Ah + m * ldk, *dl = Al + m * ldk;
        for (long long c0 = (long long)blockIdx.x * 4096; c0 < K; c0 += (long long)gridDim.x * 4096) {
            if (vec4) {
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long c = c0 + (j * 256 + threadIdx.x) * 4;
                    v[j] = c < K ? __ldcs(reinterpret_cast<const float4 *>(src + c))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long c = c0 + (j * 256 + threadIdx.x) * 4;
                    if (c < K) {
                        float4 h, l;
                        split(v[j].x, h.x, l.x);
                        split(v[j].y, h.y, l.y);
                        split(v[j].z, h.z, l.z);
                        split(v[j].w, h.w, l.w);
                        *reinterpret_cast<float4 *>(dh + c) = h;
                        *reinterpret_cast<float4 *>(dl + c) = l;
                    }
                }
            } else {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const long long c = c0 + j * 256 + threadIdx.x;
                    v[j] = c < K ? __ldcs(src + c) : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const long long c = c0 + j * 256 + threadIdx.x;
                    if (c < K) {
                        float h, l;
                        split(v[j], h, l);
                        dh[c] = h;
                        dl[c] = l;
                    }
                }
            }
        }
    }
}

// B (K x N, row pitch ldb) -> Bh, Bl (N x K, row pitch ldk): transposed so B is
// K-major too.  64x64 tiles through shared memory, 16 loads in flight per thread.
__global__ void __launch_bounds__(256)
    split_bt_kernel(const float *__restrict__ B, long long ldb, int K, int N, float *__restrict__ Bh,
                    float *__restrict__ Bl, long long ldk) {
    __shared__ float tile[64][65];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (long long k0 = (long long)blockIdx.y * 64; k0 < K; k0 += (long long)gridDim.y * 64) {
        for (long long n0 = (long long)blockIdx.x * 64; n0 < N; n0 += (long long)gridDim.x * 64) {
            float v[16];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const long long k = k0 + w * 8 + r;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long n = n0 + lane + 32 * h;
                    v[2 * r + h] = (k < K && n < N) ? __ldcs(B + k * ldb + n) : 0.0f;
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) tile[w * 8 + r][lane + 32 * h] = v[2 * r + h];
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const long long n = n0 + w * 8 + r;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long k = k0 + lane + 32 * h;
                    if (n < N && k < K) {
                        float hi, lo;
                        split(tile[lane + 32 * h][w * 8 + r], hi, lo);
                        Bh[n * ldk + k] = hi;
                        Bl[n * ldk + k] = lo;
                    }
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace t3
}  // namespace sg

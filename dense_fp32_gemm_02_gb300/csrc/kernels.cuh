// kernels.cuh -- device code of the FP32 SGEMM: the A-transpose pre-pass, the
// B re-pitch copy, the persistent TMA-fed FFMA main kernel, the alpha==0 / K==0
// scaling kernel and the bounded-wait self test.
//
// Design, in terms of the techniques the SGEMM pages describe:
//  * block tiling with a K slab staged in shared memory per step and an
//    outer-product register micro-tile per thread ("How to implement matrix
//    multiplication efficiently?", sections "Tiling" and "Thread-level
//    optimisation");
//  * A stored transposed in shared memory so one thread reads its column of A
//    with 128-bit loads (same article, "Bank conflicts" section; "SGEMM CUDA
//    kernel (Second Half)", Part 8 "Transposed As").  Here the transpose is a
//    pre-pass into global memory so that the tensor-memory accelerator (TMA)
//    can copy A tiles exactly like B tiles;
//  * double buffering, generalised to an S-stage ring of TMA copies guarded by
//    full/empty shared-memory barriers;
//  * the zig-zag lane map of "SGEMM CUDA kernel (Second Half)" (section
//    "LDS.128 Shared Memory Transactions"): for A reads lane i and lane i^1
//    fetch the same address, for B reads lane i and lane i^2 do.  The page
//    expects such pairs to merge quarter-warp transactions; on sm_103 every
//    128-bit shared load was measured at four wavefronts regardless, so the
//    map here only keeps each quarter-warp free of bank conflicts, and the
//    thread tile is sized by shared-memory bytes per FMA instead;
//  * zero-filled edge tiles (the TMA fills out-of-range box elements with 0)
//    and guarded stores, as in exercise 1 of "3.3 Shared memory and tiling".
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace sg {

// device error word bits
enum : unsigned {
    ERR_FULL_WAIT = 1u,    // consumer gave up waiting for a TMA copy
    ERR_EMPTY_WAIT = 2u,   // producer gave up waiting for a free stage
    ERR_DRAIN_WAIT = 4u,   // copies still in flight after an abort
    ERR_SELFTEST = 8u,     // the bounded-wait self test expired (expected)
};

// One word per device; every kernel of this library reports expiries here.
__device__ unsigned int g_error_word = 0;

// ------------------------------------------------------------------ configuration
// Micro-kernel of the consumer warps.
enum Micro : int {
    MICRO_FFMA = 0,    // one scalar fused multiply-add per output per k
    MICRO_FFMA2 = 1,   // packed FP32x2 FMA on two vertically adjacent outputs:
                       //   (c[i][j], c[i+1][j]) += (a[i], a[i+1]) * (b[j], b[j])
};

// Lanes of a warp form a LANES_M x LANES_N = 4 x 8 grid.  A thread owns a
// TM x TN tile made of (TM/4) x (TN/4) sub-tiles of 4x4 spaced 16 rows and 32
// columns apart, so a warp covers (4*TM) x (8*TN) outputs and every fragment
// load is one 128-bit shared load of four consecutive floats.
template <int BM_, int BN_, int BK_, int STAGES_, int WARPS_M_, int WARPS_N_, int TM_, int TN_,
          int MICRO_>
struct TileConfig {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int TM = TM_, TN = TN_;
    static constexpr int MICRO = MICRO_;
    static constexpr int LANES_M = 4, LANES_N = 8;
    static constexpr int WM = TM * LANES_M, WN = TN * LANES_N;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    static constexpr int THREADS = CONSUMER_WARPS * 32;
    static constexpr int A_STAGE = BK * BM;   // floats: K-rows of the transposed A tile
    static constexpr int B_STAGE = BK * BN;   // floats: K-rows of the B tile
    static constexpr uint32_t STAGE_BYTES = uint32_t(A_STAGE + B_STAGE) * 4u;
    static constexpr size_t SMEM_BYTES =
        size_t(STAGES) * STAGE_BYTES + 2 * STAGES * sizeof(uint64_t) + 16 + 1024;

    static_assert(WM * WARPS_M == BM && WN * WARPS_N == BN, "warp grid must cover the tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tile is made of 4x4 sub-tiles");
    static_assert(BM <= 256 && BN <= 256 && BK <= 256, "TMA box edge is at most 256");
    static_assert((A_STAGE * 4) % 1024 == 0 && (B_STAGE * 4) % 1024 == 0, "stage alignment");
    static_assert(SMEM_BYTES <= 232448, "at most 227 KB of shared memory per CTA");
};

struct MainParams {
    float *C;
    long long ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n, group_m;
    int c_vec4;              // C base 16-byte aligned and ldc % 4 == 0
    unsigned long long timeout_ns;
};

// Grouped raster: tiles are visited in groups of `group_m` tile-rows, column
// by column inside a group, so CTAs running at the same time share rows of A
// and columns of B in L2 (the wave / L2 hit-rate argument of the Hands-on-GEMM
// article, "Block-level optimisation").
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn) {
    const int per_group = group_m * tiles_n;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int gm = min(tiles_m - first_m, group_m);
    const int local = tile - g * per_group;
    tm = first_m + local % gm;
    tn = local / gm;
}

// Fragment loads for one k: TM values of A (a K-row of the transposed tile)
// and TN values of B, 128 bits at a time.
template <class Cfg>
__device__ __forceinline__ void load_fragments(const float *a_row, const float *b_row,
                                               float (&fa)[Cfg::TM], float (&fb)[Cfg::TN]) {
#pragma unroll
    for (int s = 0; s < Cfg::TM / 4; ++s) {
        const float4 v = *reinterpret_cast<const float4 *>(a_row + s * 16);
        fa[4 * s + 0] = v.x;
        fa[4 * s + 1] = v.y;
        fa[4 * s + 2] = v.z;
        fa[4 * s + 3] = v.w;
    }
#pragma unroll
    for (int t = 0; t < Cfg::TN / 4; ++t) {
        const float4 v = *reinterpret_cast<const float4 *>(b_row + t * 32);
        fb[4 * t + 0] = v.x;
        fb[4 * t + 1] = v.y;
        fb[4 * t + 2] = v.z;
        fb[4 * t + 3] = v.w;
    }
}

// acc += fa (outer product) fb
template <class Cfg>
__device__ __forceinline__ void outer_product(float (&acc)[Cfg::TM][Cfg::TN],
                                              const float (&fa)[Cfg::TM],
                                              const float (&fb)[Cfg::TN]) {
    if constexpr (Cfg::MICRO == MICRO_FFMA2) {
        // Row pair outer, column inner: the (a[i], a[i+1]) operand stays the same
        // over TN consecutive instructions.  Measured on sm_103 (16x8 tile, two
        // warps per sub-partition, fragments from registers): 127 FMA/clk/SM in
        // this order against 118 with the column loop outside.
#pragma unroll
        for (int i = 0; i < Cfg::TM; i += 2) {
            const float2 aa = make_float2(fa[i], fa[i + 1]);
#pragma unroll
            for (int j = 0; j < Cfg::TN; ++j) {
                const float2 r = ffma2(aa, make_float2(fb[j], fb[j]),
                                       make_float2(acc[i][j], acc[i + 1][j]));
                acc[i][j] = r.x;
                acc[i + 1][j] = r.y;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
            for (int j = 0; j < Cfg::TN; ++j) acc[i][j] = fmaf(fa[i], fb[j], acc[i][j]);
    }
}

// ------------------------------------------------------------------ main kernel
// Persistent kernel: CTA b computes tiles b, b + gridDim.x, ...  The k-slabs of
// all its tiles form one sequence q = 0, 1, 2, ...; slab q lives in ring stage
// q % STAGES.  Thread 0 issues the TMA copies of slab q + STAGES - 1 when the
// CTA starts consuming slab q, after every warp has released that stage's
// previous contents (empty barrier), so STAGES - 1 slabs are in flight.  Warps wait on the full barrier of a stage
// (TMA byte count) before reading it and arrive on its empty barrier after.
// There is no separate producer warp: with 8 warps per CTA each SM sub-
// partition holds two warps and a thread can keep up to 255 registers.
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    sgemm_tma_ffma_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const MainParams p) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TM = Cfg::TM, TN = Cfg::TN;

    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    float *sA = reinterpret_cast<float *>(base);
    float *sB = sA + STAGES * Cfg::A_STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * Cfg::B_STAGE);
    uint64_t *empty = full + STAGES;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int num_tiles = p.tiles_m * p.tiles_n;
    const int k_tiles = (p.K + BK - 1) / BK;
    const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const long long total_slabs = (long long)my_tiles * k_tiles;

    // Issue state, used by thread 0 only: the next slab to copy is k-slab
    // `pkt` of this CTA's tile number `pj`, into stage `pstage` whose empty
    // barrier is in phase parity `pphase`.
    long long issued = 0;
    int pj = 0, pkt = 0, pstage = 0, ptm = 0, ptn = 0;
    uint32_t pphase = 0;
    bool aborted = false;
    if (threadIdx.x == 0 && my_tiles > 0) tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, ptm, ptn);

    // Thread 0: issue the copies of the next slab.  Returns false if the wait
    // for its stage to be released expired.
    auto issue_next = [&]() -> bool {
        // first use of a stage: parity 1 refers to the phase before the
        // barrier's first one and counts as complete
        if (!mbar_wait(&empty[pstage], pphase ^ 1u, p.timeout_ns)) {
            atomicOr(&g_error_word, ERR_EMPTY_WAIT);
            return false;
        }
        mbar_arrive_expect_tx(&full[pstage], Cfg::STAGE_BYTES);
        tma_load_2d(sA + pstage * Cfg::A_STAGE, &tmA, &full[pstage], ptm * BM, pkt * BK);
        tma_load_2d(sB + pstage * Cfg::B_STAGE, &tmB, &full[pstage], ptn * BN, pkt * BK);
        ++issued;
        if (++pstage == STAGES) {
            pstage = 0;
            pphase ^= 1u;
        }
        if (++pkt == k_tiles) {
            pkt = 0;
            ++pj;
            if (pj < my_tiles)
                tile_coords(blockIdx.x + pj * gridDim.x, p.tiles_m, p.tiles_n, p.group_m, ptm, ptn);
        }
        return true;
    };

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        while (issued < STAGES - 1 && issued < total_slabs)
            if (!issue_next()) {
                aborted = true;
                break;
            }
    }

    const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
    const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
    // zig-zag lane map: lane bits {1,4} -> row group, bits {0,2,3} -> column group
    const int lm = ((lane >> 1) & 1) | ((lane >> 3) & 2);
    const int ln = (lane & 1) | ((lane >> 1) & 6);
    const int a_off = wm0 + lm * 4;
    const int b_off = wn0 + ln * 4;

    int stage = 0;          // stage of the next slab to consume
    uint32_t phase = 0;     // parity of that stage's full barrier
    for (int j = 0; j < my_tiles; ++j) {
        int tm, tn;
        tile_coords(blockIdx.x + j * gridDim.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);

        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int jj = 0; jj < TN; ++jj) acc[i][jj] = 0.0f;

        for (int kt = 0; kt < k_tiles; ++kt) {
            if (threadIdx.x == 0 && !aborted && issued < total_slabs) aborted = !issue_next();
            const int s = stage;
            bool ok = !aborted && mbar_wait(&full[s], phase, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) atomicOr(&g_error_word, ERR_FULL_WAIT);
                aborted = true;
                goto done;
            }
            const float *a_s = sA + s * Cfg::A_STAGE + a_off;
            const float *b_s = sB + s * Cfg::B_STAGE + b_off;
            // register double buffering of the fragments: the loads for k+1
            // are issued before the FMAs of k
            float fa[2][TM], fb[2][TN];
            load_fragments<Cfg>(a_s, b_s, fa[0], fb[0]);
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                if (kk + 1 < BK)
                    load_fragments<Cfg>(a_s + (kk + 1) * BM, b_s + (kk + 1) * BN,
                                        fa[(kk + 1) & 1], fb[(kk + 1) & 1]);
                outer_product<Cfg>(acc, fa[kk & 1], fb[kk & 1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // -------------------------------------------------------------- epilogue
        {
            const int row0 = tm * BM + a_off;
            const int col0 = tn * BN + b_off;
            const float alpha = p.alpha, beta = p.beta;
#pragma unroll
            for (int s4 = 0; s4 < TM / 4; ++s4) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int row = row0 + s4 * 16 + r;
                    if (row >= p.M) continue;
                    float *crow = p.C + (long long)row * p.ldc;
#pragma unroll
                    for (int t = 0; t < TN / 4; ++t) {
                        const int col = col0 + t * 32;
                        const float *v = &acc[4 * s4 + r][4 * t];
                        if (p.c_vec4 && col + 3 < p.N) {
                            float4 o;
                            if (beta != 0.0f) {
                                const float4 c = __ldcs(reinterpret_cast<const float4 *>(crow + col));
                                o.x = fmaf(alpha, v[0], beta * c.x);
                                o.y = fmaf(alpha, v[1], beta * c.y);
                                o.z = fmaf(alpha, v[2], beta * c.z);
                                o.w = fmaf(alpha, v[3], beta * c.w);
                            } else {
                                o.x = alpha * v[0];
                                o.y = alpha * v[1];
                                o.z = alpha * v[2];
                                o.w = alpha * v[3];
                            }
                            __stcs(reinterpret_cast<float4 *>(crow + col), o);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (col + e < p.N) {
                                    const float c = (beta != 0.0f) ? beta * crow[col + e] : 0.0f;
                                    crow[col + e] = (beta != 0.0f) ? fmaf(alpha, v[e], c)
                                                                   : alpha * v[e];
                                }
                            }
                        }
                    }
                }
            }
        }
    }
done:
    // After an abort, thread 0 waits (bounded) for the copies it issued and no
    // warp consumed, so no copy is still writing when the CTA exits.
    if (threadIdx.x == 0 && aborted) {
        const long long first = issued > STAGES ? issued - STAGES : 0;
        for (long long qq = first; qq < issued; ++qq) {
            const int s = int(qq % STAGES);
            if (!mbar_wait(&full[s], uint32_t((qq / STAGES) & 1), p.timeout_ns)) {
                atomicOr(&g_error_word, ERR_DRAIN_WAIT);
                break;
            }
        }
    }
}

// ------------------------------------------------------------------ pre-pass
// At[k][m] = A[m][k].  32x32 tiles through shared memory: coalesced reads along
// k, coalesced writes along m.
__global__ void __launch_bounds__(256)
    pack_a_transpose_kernel(const float *__restrict__ A, long long lda, int M, int K,
                            float *__restrict__ At, long long ldat) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    for (long long m0 = (long long)blockIdx.y * 32; m0 < M; m0 += (long long)gridDim.y * 32) {
        for (long long k0 = (long long)blockIdx.x * 32; k0 < K; k0 += (long long)gridDim.x * 32) {
#pragma unroll
            for (int r = ty; r < 32; r += 8) {
                const long long m = m0 + r, k = k0 + tx;
                tile[r][tx] = (m < M && k < K) ? __ldcs(A + m * lda + k) : 0.0f;
            }
            __syncthreads();
#pragma unroll
            for (int r = ty; r < 32; r += 8) {
                const long long k = k0 + r, m = m0 + tx;
                if (k < K && m < M) At[k * ldat + m] = tile[tx][r];
            }
            __syncthreads();
        }
    }
}

// Bp[k][n] = B[k][n] with a 16-byte row pitch (ldbp % 4 == 0) for the TMA.
__global__ void __launch_bounds__(256)
    pack_b_copy_kernel(const float *__restrict__ B, long long ldb, int K, int N,
                       float *__restrict__ Bp, long long ldbp) {
    const long long total = (long long)K * N;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long k = idx / N, n = idx - k * N;
        Bp[k * ldbp + n] = B[k * ldb + n];
    }
}

// C = beta * C on the M x N block (C not read when beta == 0): the alpha == 0 /
// K == 0 case, where A and B are not read.
__global__ void __launch_bounds__(256)
    scale_c_kernel(float *C, long long ldc, int M, int N, float beta) {
    const long long total = (long long)M * N;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / N, j = idx - i * N;
        float *c = C + i * ldc + j;
        *c = (beta == 0.0f) ? 0.0f : beta * *c;
    }
}

// One thread waits on a barrier that nothing completes; the bounded wait must
// expire, record ERR_SELFTEST and return.
__global__ void wait_timeout_selftest_kernel(unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(&bar, 0u, timeout_ns)) atomicOr(&g_error_word, ERR_SELFTEST);
    }
}

}  // namespace sg

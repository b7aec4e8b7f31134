// kernels.cuh -- device code of the FP32 SGEMM's persistent TMA-fed FFMA main
// kernel (tile configurations, work split, epilogue, the kernel template).
// The pre-pass, scaling, small-problem and self-test kernels are in
// aux_kernels.cuh.
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
//    fetch the same address, for B reads lane i and lane i^2 do, so the
//    quarter-warp transactions of a 128-bit shared load merge in pairs.  On
//    sm_103 this measures at 2.0 wavefronts per 128-bit load (a layout in
//    which neighbouring lanes read different addresses measured 4.0);
//  * zero-filled edge tiles (the TMA fills out-of-range box elements with 0)
//    and guarded stores, as in exercise 1 of "3.3 Shared memory and tiling".
#pragma once

#include <cstdint>
#include <type_traits>
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
    ERR_BOUNDS = 16u,      // range-checked build: an index was out of range
};

// One word per device; every kernel of this library reports expiries here.
// Internal linkage: each translation unit that includes this file has its own
// copy, and the host reads and clears all of them (variant.cuh).
static __device__ unsigned int g_error_word = 0;

// Range checks of the range-checked build (compiled with -DSGEMM_DEBUG_BOUNDS,
// the stand-in for a memory checker): SG_IN_RANGE(cond) is true when cond
// holds; otherwise it records ERR_BOUNDS in the device error word and is
// false, and the caller skips the access.  In the normal build it is `true`
// and the checks cost nothing.
#ifdef SGEMM_DEBUG_BOUNDS
__device__ __forceinline__ bool sg_in_range(bool ok) {
    if (!ok) atomicOr(&g_error_word, ERR_BOUNDS);
    return ok;
}
#define SG_IN_RANGE(cond) ::sg::sg_in_range(bool(cond))
#else
#define SG_IN_RANGE(cond) true
#endif

// Limit of the waits that, after an abort, let this CTA's own copies (and
// tensor-core operations) in flight complete before it exits.  Those always
// complete, so the wait only has to outlast them: it takes its own generous
// limit rather than the caller's, which may be short and has just expired.
constexpr unsigned long long kDrainLimitNs = 1000000000ull;   // 1 s
__device__ __forceinline__ unsigned long long drain_limit_ns(unsigned long long timeout_ns) {
    return timeout_ns > kDrainLimitNs ? timeout_ns : kDrainLimitNs;
}

// ------------------------------------------------------------------ configuration
// Micro-kernel of the consumer warps.
enum Micro : int {
    MICRO_FFMA = 0,    // one scalar fused multiply-add per output per k
    MICRO_FFMA2 = 1,   // packed FP32x2 FMA on two vertically adjacent outputs:
                       //   (c[i][j], c[i+1][j]) += (a[i], a[i+1]) * (b[j], b[j])
};

// Who issues the TMA copies of the k-slabs.
enum Issue : int {
    ISSUE_THREAD0 = 0,       // consumer thread 0, at the start of each of its slabs
    ISSUE_PRODUCER_WG = 1,   // a producer warpgroup in front of the consumer warps
    ISSUE_LAST_WARP = 2,     // the consumer warp that releases a stage last refills it
};

// Lanes of a warp form a LANES_M x LANES_N = 4 x 8 grid.  A thread owns a
// TM x TN tile made of (TM/4) x (TN/4) sub-tiles of 4x4 spaced 16 rows and 32
// columns apart, so a warp covers (4*TM) x (8*TN) outputs and every fragment
// load is one 128-bit shared load of four consecutive floats.
template <int BM_, int BN_, int BK_, int STAGES_, int WARPS_M_, int WARPS_N_, int TM_, int TN_,
          int MICRO_, int ISSUE_>
struct TileConfig {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int TM = TM_, TN = TN_;
    static constexpr int MICRO = MICRO_;
    static constexpr int LANES_M = 4, LANES_N = 8;
    static constexpr int WM = TM * LANES_M, WN = TN * LANES_N;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    static constexpr int CONSUMER_THREADS = CONSUMER_WARPS * 32;
    static constexpr int ISSUE = ISSUE_;
    static constexpr bool WS = ISSUE_ == ISSUE_PRODUCER_WG;
    static constexpr int PRODUCER_THREADS = WS ? 128 : 0;
    static constexpr int THREADS = PRODUCER_THREADS + CONSUMER_THREADS;
    // Register split (setmaxnreg, WS only): the launch gives every thread
    // LAUNCH_REGS; the producer warpgroup drops to PRODUCER_REGS and the
    // consumers rise to CONSUMER_REGS.  The split must fit the launch's total.
    static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8;
    static constexpr int PRODUCER_REGS = 40;
    static constexpr int CONSUMER_REGS_FIT =
        ((LAUNCH_REGS * THREADS - PRODUCER_REGS * PRODUCER_THREADS) / CONSUMER_THREADS) / 8 * 8;
    static constexpr int CONSUMER_REGS = CONSUMER_REGS_FIT > 248 ? 248 : CONSUMER_REGS_FIT;
    static constexpr int A_STAGE = BK * BM;   // floats: K-rows of the transposed A tile
    static constexpr int B_STAGE = BK * BN;   // floats: K-rows of the B tile
    static constexpr uint32_t STAGE_BYTES = uint32_t(A_STAGE + B_STAGE) * 4u;
    static constexpr size_t RING_SMEM_BYTES =
        size_t(STAGES) * STAGE_BYTES + 2 * STAGES * sizeof(uint64_t) + 16 + 1024;
    // Epilogue of C rows (StagedEpilogueConfig): direct 128-bit accesses from
    // the registers (false), or every row through a staging area in shared
    // memory, per consumer warp the four rows of WN columns it writes in one
    // epilogue round (true).
    static constexpr bool STAGED_EPI = false;
    // A staged row is WN floats plus 16 of padding: the eight lanes of a
    // quarter-warp write two rows in one 128-bit store, and the padding puts
    // the second row 16 banks after the first, so they do not conflict.
    static constexpr int EPI_ROW = WN + 16;
    static constexpr int EPI_STAGE_FLOATS = LANES_M * EPI_ROW;
    static constexpr size_t EPI_BYTES = size_t(CONSUMER_WARPS) * EPI_STAGE_FLOATS * 4;
    static constexpr size_t SMEM_BYTES = RING_SMEM_BYTES;
    // Epilogue rounds whose C_in loads are issued together (staged epilogue).
    static constexpr int EPI_BATCH = 1;
    static constexpr int TILE_FLOATS = BM * BN;
    // EX: the kernel serves batched calls and the fused bias/activation
    // epilogue (see ExConfig); the plain kernel leaves that code out, which
    // keeps its main loop under the register cap.
    static constexpr bool EX = false;
    static constexpr bool BATCH = false;
    // TallBatchConfig: a batch run as one tall GEMM (B's rows offset per batch)
    static constexpr bool TALL = false;
    // Failure-detection test instantiation only (AbortTestConfig): the CTA
    // slab at which consumer warp 0 of CTA 0 leaves out its release; -1 here.
    static constexpr int DROP_RELEASE_SLAB = -1;
    // CTAs resident per SM (TwoPerSMConfig: 2, each with half the registers
    // and at most half the shared memory)
    static constexpr int CTAS_PER_SM = 1;

    static_assert(WM * WARPS_M == BM && WN * WARPS_N == BN, "warp grid must cover the tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tile is made of 4x4 sub-tiles");
    static_assert(BM <= 256 && BN <= 256 && BK <= 256, "TMA box edge is at most 256");
    static_assert((A_STAGE * 4) % 1024 == 0 && (B_STAGE * 4) % 1024 == 0, "stage alignment");
    static_assert(SMEM_BYTES <= 232448, "at most 227 KB of shared memory per CTA");
    static_assert(CONSUMER_WARPS % 4 == 0, "whole consumer warpgroups");
    static_assert(!WS || PRODUCER_REGS * PRODUCER_THREADS + CONSUMER_REGS * CONSUMER_THREADS <=
                             LAUNCH_REGS * THREADS,
                  "register split exceeds the launch allocation");
};

// Activation of the fused epilogue.
enum Act : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2 };

// The same tile configuration for the batched / fused-epilogue kernel.
template <class Base>
struct ExConfig : Base {
    static constexpr bool EX = true;
    static constexpr bool BATCH = true;
};

// The same tile configuration with the fused epilogue but one GEMM (2-D
// tensor maps, no batch coordinate): a bias or an activation on an unbatched
// call.
template <class Base>
struct FusedConfig : Base {
    static constexpr bool EX = true;
    static constexpr bool BATCH = false;
};

// The same tile configuration for a batch of GEMMs run as one tall GEMM: the
// batches' transposed A side by side (K x batch*M), their C one under the
// other (batch*M x N, batch b at row b*M), their B one under the other (batch
// b's rows at b*K).  Every batch holds whole tiles (M a multiple of BM, K of
// BK) and the raster groups are one batch's tile rows (group_m = M/BM), so a
// tile's raster group is its batch, and only the copies of B depend on it:
// their k coordinate starts at that batch's first row of B.  The rest is the
// plain kernel, with its epilogue and its 123 registers (the batched kernel,
// ExConfig, needs 128 and runs its main loop 2 % slower).
template <class Base>
struct TallBatchConfig : Base {
    static constexpr bool TALL = true;
};

// The same tile configuration with one release left out on purpose: consumer
// warp 0 of CTA 0 does not arrive on the empty barrier of the CTA's slab 2.
// The issuer's wait for that stage then expires with no copy into it in
// flight, and the kernel's abort path runs: error word, abort flag, no C
// written for the CTA's tiles, copies drained.  Launched only by the library's
// failure-detection test switch (sgemm_debug_drop_release); never by default.
template <class Base>
struct AbortTestConfig : Base {
    static constexpr int DROP_RELEASE_SLAB = 2;
};

// The same tile configuration with the staged epilogue (store_tile_staged),
// for C whose rows do not all start 16-byte aligned.
template <class Base>
struct StagedEpilogueConfig : Base {
    static constexpr bool STAGED_EPI = true;
    static constexpr size_t SMEM_BYTES = Base::RING_SMEM_BYTES + Base::EPI_BYTES;
    static_assert(SMEM_BYTES <= 232448, "staging areas fit beside the ring");
};

// The same tile configuration with two CTAs resident per SM: the two run
// their tiles independently, so one CTA's epilogue overlaps the other's main
// loop.  The configuration must fit twice in an SM (registers: THREADS x 128
// at most half the register file; shared memory: at most half of 227 KB).
template <class Base>
struct TwoPerSMConfig : Base {
    static constexpr int CTAS_PER_SM = 2;
    static_assert(Base::SMEM_BYTES <= 232448 / 2 - 1024, "two CTAs fit an SM's shared memory");
    static_assert(Base::THREADS <= 256, "two CTAs fit an SM's register file at 128 registers");
};

struct MainParams {
    float *C;
    long long ldc;
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n, group_m;
    int c_vec4;              // C base 16-byte aligned (rows then checked one by one)
    unsigned long long timeout_ns;
    // Work split.  Tiles [0, dp_tiles) are whole-tile work, CTA b taking tiles
    // b, b + gridDim.x, ...  The k-slabs of the remaining tiles, in tile-major
    // order, form one range of sk_slabs slabs cut into gridDim.x contiguous,
    // nearly equal pieces, one per CTA (stream-K).
    int dp_tiles;
    long long sk_slabs;
    float *partials;         // 2 * gridDim.x slots of BM*BN floats (sk_slabs > 0)
    int *counters;           // one per stream-K tile, zero at launch (sk_slabs > 0)
};

// Parameters only the batched / fused-epilogue kernel (EX) reads; a separate
// kernel argument, so the plain kernel's parameters stay as they are.
struct ExParams {
    // Batches: tile t belongs to batch t / (tiles_m * tiles_n).  Batch b's C
    // starts at C + b * stride_c; its A and B are plane b of the 3-D tensor
    // maps (plane 0 for every batch when a_planes / b_planes is 1).
    int batch;
    // TallBatchConfig: rows of B per batch (0 when every batch shares one B)
    int tall_b_rows;
    long long stride_c;
    int a_planes, b_planes;
    // Fused epilogue: C = act(alpha*acc + beta*C + bias[col]); bias may be null
    // (batch b's bias at bias + b * stride_bias).
    const float *bias;
    long long stride_bias;
    int bias_vec4;           // bias base 16-byte aligned and stride_bias % 4 == 0
    int act;
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

// Batch and tile coordinates of tile number `tile`.
__device__ __forceinline__ void decode_tile(const struct MainParams &p, int tile, int &tb, int &tm,
                                            int &tn) {
    const int per_batch = p.tiles_m * p.tiles_n;
    tb = tile / per_batch;
    tile_coords(tile - tb * per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
}

// 128-bit shared-memory load from a 32-bit shared-window address.  Explicit
// shared addressing keeps fragment addresses in one 32-bit register each; with
// generic 64-bit pointers the consumer loop needed 255 registers instead of 222
// and ran 7% slower on sm_103.  The memory clobber keeps the loads between the
// barrier wait and release that guard the stage they read.
__device__ __forceinline__ float4 lds128(uint32_t addr) {
    float4 v;
    asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "r"(addr)
        : "memory");
    return v;
}

// Fragment loads for one k: TM values of A (a K-row of the transposed tile)
// and TN values of B, 128 bits at a time.  a_row, b_row: shared addresses.
template <class Cfg>
__device__ __forceinline__ void load_fragments(uint32_t a_row, uint32_t b_row,
                                               float (&fa)[Cfg::TM], float (&fb)[Cfg::TN]) {
#pragma unroll
    for (int s = 0; s < Cfg::TM / 4; ++s) {
        const float4 v = lds128(a_row + s * 16 * 4);
        fa[4 * s + 0] = v.x;
        fa[4 * s + 1] = v.y;
        fa[4 * s + 2] = v.z;
        fa[4 * s + 3] = v.w;
    }
#pragma unroll
    for (int t = 0; t < Cfg::TN / 4; ++t) {
        const float4 v = lds128(b_row + t * 32 * 4);
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

// ------------------------------------------------------------------ warp specialisation
template <int N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
// Named CTA barrier `id` over `count` threads (whole, converged warps).
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ work split
// One contiguous run of k-slabs of one tile that a CTA computes.
struct Segment {
    int tile;     // tile index in raster order
    int kb, ke;   // slab range [kb, ke)
    int slot;     // partial-sum slot, or -1 when the segment is the whole tile
};

// First stream-K slab of CTA b (relative to the stream-K region).
__device__ __forceinline__ long long sk_start(int b, long long sk_slabs, int grid) {
    return ((long long)b * sk_slabs) / grid;
}

// The CTA whose stream-K range holds slab x: the largest b with sk_start(b) <= x.
__device__ __forceinline__ int sk_owner(long long x, long long sk_slabs, int grid) {
    int b = int(((x + 1) * grid - 1) / sk_slabs);
    if (b > grid - 1) b = grid - 1;
    while (b > 0 && sk_start(b, sk_slabs, grid) > x) --b;
    while (b + 1 < grid && sk_start(b + 1, sk_slabs, grid) <= x) ++b;
    return b;
}

// Segments of one CTA, in the order it computes them: its whole tiles, then
// the pieces of its stream-K range (at most one partial piece at each end).
// A partial piece at the start of the range uses slot 2b, one at the end 2b+1.
struct SegmentIter {
    int next_dp;
    long long x, end;
    bool at_first_sk;

    __device__ void init(const MainParams &p) {
        next_dp = blockIdx.x;
        x = sk_start(blockIdx.x, p.sk_slabs, gridDim.x);
        end = sk_start(blockIdx.x + 1, p.sk_slabs, gridDim.x);
        at_first_sk = true;
    }

    __device__ bool next(const MainParams &p, int k_tiles, Segment &seg) {
        if (next_dp < p.dp_tiles) {
            seg.tile = next_dp;
            seg.kb = 0;
            seg.ke = k_tiles;
            seg.slot = -1;
            next_dp += gridDim.x;
            return true;
        }
        if (x >= end) return false;
        const long long rel = x / k_tiles;
        seg.tile = p.dp_tiles + int(rel);
        seg.kb = int(x - rel * k_tiles);
        seg.ke = int(min((long long)k_tiles, (long long)seg.kb + (end - x)));
        const bool whole = (seg.kb == 0 && seg.ke == k_tiles);
        seg.slot = whole ? -1 : 2 * int(blockIdx.x) + (at_first_sk ? 0 : 1);
        at_first_sk = false;
        x += seg.ke - seg.kb;
        return true;
    }
};

// Segment number `si` of this CTA (the same sequence SegmentIter yields),
// computed from scratch so a caller keeps only the counter between segments.
__device__ __forceinline__ bool segment_at(const MainParams &p, int k_tiles, int si, Segment &seg) {
    const int b = blockIdx.x, G = gridDim.x;
    const int n_dp = p.dp_tiles > b ? (p.dp_tiles - 1 - b) / G + 1 : 0;
    if (si < n_dp) {
        seg.tile = b + si * G;
        seg.kb = 0;
        seg.ke = k_tiles;
        seg.slot = -1;
        return true;
    }
    const int j = si - n_dp;
    const long long x0 = sk_start(b, p.sk_slabs, G), x1 = sk_start(b + 1, p.sk_slabs, G);
    const long long x = j == 0 ? x0 : (x0 / k_tiles + j) * (long long)k_tiles;
    if (x >= x1) return false;
    const long long rel = x / k_tiles;
    seg.tile = p.dp_tiles + int(rel);
    seg.kb = int(x - rel * k_tiles);
    seg.ke = int(min((long long)k_tiles, (long long)seg.kb + (x1 - x)));
    const bool whole = (seg.kb == 0 && seg.ke == k_tiles);
    seg.slot = whole ? -1 : 2 * b + (j == 0 ? 0 : 1);
    return true;
}

// ------------------------------------------------------------------ epilogue
// Activation of the fused epilogue (ACT_GELU: the erf form v * Phi(v)).
__device__ __forceinline__ float activate(float v, int act) {
    if (act == ACT_RELU) return fmaxf(v, 0.0f);
    if (act == ACT_GELU) return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
    return v;
}

// C = alpha * acc + beta * C for this thread's outputs of tile (tm, tn);
// C is not read when beta == 0.  Rows >= M and columns >= N are not written.
template <class Cfg>
__device__ __forceinline__ void store_tile(const float (&acc)[Cfg::TM][Cfg::TN], const MainParams &p,
                                           int tm, int tn, int a_off, int b_off) {
    const int row0 = tm * Cfg::BM + a_off;
    const int col0 = tn * Cfg::BN + b_off;
    const float alpha = p.alpha, beta = p.beta;
    // The rows of C are read one after another below (a store to one row may
    // alias the next row's load, so the loads cannot be hoisted); start all
    // their lines towards L2 first, so only the first row waits for DRAM.
    // Measured: ragged 4097x3001x1023 (beta 1) 2.5 % faster, 8192^3 (beta 0.5)
    // 0.14 % faster.
    if (beta != 0.0f) {
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i) {
            const int row = row0 + (i >> 2) * 16 + (i & 3);
            if (row < p.M) {
                const float *crow = p.C + (long long)row * p.ldc + col0;
#pragma unroll
                for (int t = 0; t < Cfg::TN / 4; ++t)
                    if (col0 + t * 32 < p.N) prefetch_l2(crow + t * 32);
            }
        }
    }
#pragma unroll
    for (int s4 = 0; s4 < Cfg::TM / 4; ++s4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + s4 * 16 + r;
            if (row >= p.M) continue;
            float *crow = p.C + (long long)row * p.ldc;
            // 128-bit accesses where this row starts 16-byte aligned (every row
            // when ldc % 4 == 0; one row in four for an odd ldc)
            const bool c_row_vec = p.c_vec4 && (reinterpret_cast<uintptr_t>(crow) & 15u) == 0;
#pragma unroll
            for (int t = 0; t < Cfg::TN / 4; ++t) {
                const int col = col0 + t * 32;
                const float *v = &acc[4 * s4 + r][4 * t];
                // range-checked build: the four outputs lie in this tile
                if (!SG_IN_RANGE(row >= tm * Cfg::BM && row < (tm + 1) * Cfg::BM &&
                                 col >= tn * Cfg::BN && col + 3 < (tn + 1) * Cfg::BN))
                    continue;
                if (c_row_vec && col + 3 < p.N) {
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
                            crow[col + e] = (beta != 0.0f) ? fmaf(alpha, v[e], c) : alpha * v[e];
                        }
                    }
                }
            }
        }
    }
}

// The lines of C_in that the staged epilogue reads for this thread's warp
// (rows roww .. roww + 4 * TM - 1 of its WN columns) started towards L2: lane
// l takes row roww + l (and roww + l + 32, ...).  Issued when the warp starts
// a tile, so the epilogue's first round finds them in L2 too.
template <class Cfg>
__device__ __forceinline__ void prefetch_c_tile_rows(const MainParams &p, int tm, int tn, int a_off,
                                                     int b_off) {
    constexpr int TM = Cfg::TM, WN = Cfg::WN, RH = WN / 32;
    const int lane = threadIdx.x & 31;
    const int rg = (a_off % Cfg::WM) >> 2, j = (b_off % WN) >> 2;
    const int roww = tm * Cfg::BM + a_off - 4 * rg;
    const int colw = tn * Cfg::BN + b_off - 4 * j;
#pragma unroll
    for (int i = 0; i < (4 * TM + 31) / 32; ++i) {
        const int row = roww + lane + 32 * i;
        if (lane + 32 * i < 4 * TM && row < p.M) {
            const float *crow = p.C + (long long)row * p.ldc;
#pragma unroll
            for (int h = 0; h <= RH; ++h) {
                const int col = min(colw + 32 * h, colw + WN - 1);
                if (col < p.N) prefetch_l2(crow + col);
            }
        }
    }
}

// The epilogue for C whose rows do not all start 16-byte aligned (ldc % 4 !=
// 0, or C itself not 16-byte aligned): C = alpha * acc + beta * C for this
// thread's outputs of tile (tm, tn); C is not read when beta == 0; rows >= M
// and columns >= N are not written.
//
// A thread's own outputs are four consecutive columns, 32 apart, of rows 16
// apart, so 32-bit accesses straight from the registers would touch, per warp
// access, four rows 16 bytes apart: four times the sectors they use.  Instead
// the warp's outputs go through its staging area in shared memory (the
// coalesced write-back through shared memory of "SGEMM CUDA kernel (Second
// Half)", Part 9).  In round (s4, r) the warp holds four rows of C (one per
// row group of lanes, 4 rows apart) of WN columns; the lanes write them to the
// area, read them back row by row, and every warp access to C then covers 128
// contiguous bytes of one row.  C_in is read the same way, EPI_BATCH rounds
// at a time; every line of the warp's part of C_in was started towards L2
// when the warp began the tile (prefetch_c_tile_rows).
template <class Cfg>
__device__ __forceinline__ void store_tile_staged(const float (&acc)[Cfg::TM][Cfg::TN],
                                                  const MainParams &p, int tm, int tn, int a_off,
                                                  int b_off, uint32_t epi) {
    constexpr int TM = Cfg::TM, TN = Cfg::TN, WN = Cfg::WN;
    constexpr int RH = WN / 32;          // 32-column parts of a warp row
    constexpr int RB = Cfg::EPI_BATCH;   // rounds whose C_in is loaded together
    static_assert(4 * RH == TN, "a round holds TN values per lane");
    static_assert(TM <= 32 && 4 % RB == 0, "rounds of a row group");
    const int lane = threadIdx.x & 31;
    const int rg = (a_off % Cfg::WM) >> 2, j = (b_off % WN) >> 2;   // lane row group, column group
    const int roww = tm * Cfg::BM + a_off - 4 * rg;                  // the warp's first row
    const int colw = tn * Cfg::BN + b_off - 4 * j;                   // and first column
    const float alpha = p.alpha, beta = p.beta;
    // (C_in's lines were started towards L2 when the warp began the tile:
    // prefetch_c_tile_rows)
#pragma unroll
    for (int g = 0; g < TM / RB; ++g) {
        const int s4 = (g * RB) / 4, r0 = (g * RB) % 4;
        float cin[RB][TN];
        if (beta != 0.0f) {
#pragma unroll
            for (int rr = 0; rr < RB; ++rr)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int rq = roww + 4 * q + 16 * s4 + r0 + rr;
                    const float *crow = p.C + (long long)rq * p.ldc;
#pragma unroll
                    for (int h = 0; h < RH; ++h) {
                        const int col = colw + lane + 32 * h;
                        cin[rr][RH * q + h] = (rq < p.M && col < p.N) ? __ldcs(crow + col) : 0.0f;
                    }
                }
        }
#pragma unroll
        for (int rr = 0; rr < RB; ++rr) {
            __syncwarp();   // the previous round's reads of the area are done
#pragma unroll
            for (int t = 0; t < TN / 4; ++t) {
                const float *v = &acc[4 * s4 + r0 + rr][4 * t];
                if (SG_IN_RANGE(rg * Cfg::EPI_ROW + 4 * j + 32 * t + 3 < Cfg::EPI_STAGE_FLOATS))
                    sts128(epi + uint32_t(rg * Cfg::EPI_ROW + 4 * j + 32 * t) * 4u,
                           make_float4(v[0], v[1], v[2], v[3]));
            }
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rq = roww + 4 * q + 16 * s4 + r0 + rr;
                float *crow = p.C + (long long)rq * p.ldc;
#pragma unroll
                for (int h = 0; h < RH; ++h) {
                    const int col = colw + lane + 32 * h;
                    if (!SG_IN_RANGE(q * Cfg::EPI_ROW + lane + 32 * h < Cfg::EPI_STAGE_FLOATS &&
                                     rq >= tm * Cfg::BM && rq < (tm + 1) * Cfg::BM &&
                                     col >= tn * Cfg::BN && col < (tn + 1) * Cfg::BN))
                        continue;
                    const float x = lds32(epi + uint32_t(q * Cfg::EPI_ROW + lane + 32 * h) * 4u);
                    if (rq < p.M && col < p.N)
                        __stcs(crow + col, (beta != 0.0f) ? fmaf(alpha, x, beta * cin[rr][RH * q + h])
                                                          : alpha * x);
                }
            }
        }
    }
}

// The epilogue of the batched / fused kernel: C = act(alpha * acc + beta * C +
// bias) for this thread's outputs of tile (tm, tn) of batch tb; C is not read
// when beta == 0, and without a bias or an activation the plain alpha/beta
// update is all that runs.  Rows >= M and columns >= N are not written.
template <class Cfg>
__device__ __forceinline__ void store_tile_ex(const float (&acc)[Cfg::TM][Cfg::TN],
                                              const MainParams &p, const ExParams &x, int tb,
                                              int tm, int tn, int a_off, int b_off) {
    const int row0 = tm * Cfg::BM + a_off;
    const int col0 = tn * Cfg::BN + b_off;
    const float alpha = p.alpha, beta = p.beta;
    float *const Cb = p.C + (long long)tb * x.stride_c;
    const float *const bias = x.bias ? x.bias + (long long)tb * x.stride_bias : nullptr;
    const bool fused = bias != nullptr || x.act != ACT_NONE;
    // C's lines towards L2 before the row-by-row reads (as in store_tile)
    if (beta != 0.0f) {
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i) {
            const int row = row0 + (i >> 2) * 16 + (i & 3);
            if (row < p.M) {
                const float *crow = Cb + (long long)row * p.ldc + col0;
#pragma unroll
                for (int t = 0; t < Cfg::TN / 4; ++t)
                    if (col0 + t * 32 < p.N) prefetch_l2(crow + t * 32);
            }
        }
    }
    // the bias of four columns (read where it is used: an L1 hit after the
    // first row, and four live registers instead of TN)
    auto bias4 = [&](int col) {
        if (bias && x.bias_vec4 && col + 3 < p.N)
            return __ldg(reinterpret_cast<const float4 *>(bias + col));
        float4 q;
        q.x = (bias && col < p.N) ? bias[col] : 0.0f;
        q.y = (bias && col + 1 < p.N) ? bias[col + 1] : 0.0f;
        q.z = (bias && col + 2 < p.N) ? bias[col + 2] : 0.0f;
        q.w = (bias && col + 3 < p.N) ? bias[col + 3] : 0.0f;
        return q;
    };
#pragma unroll
    for (int s4 = 0; s4 < Cfg::TM / 4; ++s4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + s4 * 16 + r;
            if (row >= p.M) continue;
            float *crow = Cb + (long long)row * p.ldc;
            const bool c_row_vec = p.c_vec4 && (reinterpret_cast<uintptr_t>(crow) & 15u) == 0;
#pragma unroll
            for (int t = 0; t < Cfg::TN / 4; ++t) {
                const int col = col0 + t * 32;
                const float *v = &acc[4 * s4 + r][4 * t];
                // range-checked build: the four outputs lie in this tile
                if (!SG_IN_RANGE(row >= tm * Cfg::BM && row < (tm + 1) * Cfg::BM &&
                                 col >= tn * Cfg::BN && col + 3 < (tn + 1) * Cfg::BN))
                    continue;
                if (c_row_vec && col + 3 < p.N) {
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
                    if (fused) {
                        const float4 bq = bias4(col);
                        o.x = activate(bias ? o.x + bq.x : o.x, x.act);
                        o.y = activate(bias ? o.y + bq.y : o.y, x.act);
                        o.z = activate(bias ? o.z + bq.z : o.z, x.act);
                        o.w = activate(bias ? o.w + bq.w : o.w, x.act);
                    }
                    __stcs(reinterpret_cast<float4 *>(crow + col), o);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (col + e < p.N) {
                            const float c = (beta != 0.0f) ? beta * crow[col + e] : 0.0f;
                            float o = (beta != 0.0f) ? fmaf(alpha, v[e], c) : alpha * v[e];
                            if (fused) o = activate(bias ? o + bias[col + e] : o, x.act);
                            crow[col + e] = o;
                        }
                    }
                }
            }
        }
    }
}

// Partial-sum slot layout: float4 number v of consumer thread t sits at
// (v * CONSUMER_THREADS + t),
// so each warp store or load of one float4 per lane covers 512 contiguous bytes.
template <class Cfg>
__device__ __forceinline__ void write_partial(const float (&acc)[Cfg::TM][Cfg::TN], float *slot,
                                              int ctid) {
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
        for (int j4 = 0; j4 < Cfg::TN / 4; ++j4) {
            const int v = i * (Cfg::TN / 4) + j4;
            __stcg(reinterpret_cast<float4 *>(slot) + (size_t)v * Cfg::CONSUMER_THREADS + ctid,
                   make_float4(acc[i][4 * j4], acc[i][4 * j4 + 1], acc[i][4 * j4 + 2],
                               acc[i][4 * j4 + 3]));
        }
}

// Row i of the thread tile, summed over the tile's pieces in k order: pieces
// are the non-empty stream-K ranges of CTAs b_lo..b_hi; sk_start advances by
// sk_q plus a carry from sk_r (no division).  The piece of CTA b sits in slot
// 2b when the tile is b's first one, else in slot 2b+1.
template <class Cfg>
__device__ __forceinline__ void sum_pieces_row(float (&row)[Cfg::TN], const float *partials, int i,
                                               int ctid, int b_lo, int b_hi, long long q0, int r0,
                                               long long sk_q, int sk_r, long long tile_start) {
    float4 sum[Cfg::TN / 4];
    bool first = true;
    long long b0 = q0;
    int r = r0;
    for (int b = b_lo; b <= b_hi; ++b) {
        long long b1 = b0 + sk_q;
        r += sk_r;
        if (r >= int(gridDim.x)) {
            r -= gridDim.x;
            ++b1;
        }
        if (b0 < b1) {
            int slot = 2 * b + (b0 >= tile_start ? 0 : 1);
            if (!SG_IN_RANGE(slot >= 0 && slot < 2 * int(gridDim.x))) slot = 0;
            const float4 *src = reinterpret_cast<const float4 *>(partials + (size_t)slot * Cfg::TILE_FLOATS);
#pragma unroll
            for (int j4 = 0; j4 < Cfg::TN / 4; ++j4) {
                const float4 q =
                    __ldcg(src + (size_t)(i * (Cfg::TN / 4) + j4) * Cfg::CONSUMER_THREADS + ctid);
                if (first) {
                    sum[j4] = q;
                } else {
                    sum[j4].x += q.x;
                    sum[j4].y += q.y;
                    sum[j4].z += q.z;
                    sum[j4].w += q.w;
                }
            }
            first = false;
        }
        b0 = b1;
    }
#pragma unroll
    for (int j4 = 0; j4 < Cfg::TN / 4; ++j4) {
        row[4 * j4] = sum[j4].x;
        row[4 * j4 + 1] = sum[j4].y;
        row[4 * j4 + 2] = sum[j4].z;
        row[4 * j4 + 3] = sum[j4].w;
    }
}

// After an abort: this CTA's partial sums may be wrong, so every stream-K
// tile it holds a piece of is made impossible to complete: its counter is
// raised far past any piece count, and no CTA ever sums the tile's pieces
// into C.  Called by each thread that records an expiry, before it reaches the
// consumer barrier at which thread 0 counts the CTA's piece, so it comes first
// in the counter's order.  Several calls only add more.
__device__ __forceinline__ void block_stream_k_tiles(const MainParams &p, int k_tiles) {
    const long long x0 = sk_start(blockIdx.x, p.sk_slabs, gridDim.x);
    const long long x1 = sk_start(blockIdx.x + 1, p.sk_slabs, gridDim.x);
    for (long long t = x0 / k_tiles; x0 < x1 && t <= (x1 - 1) / k_tiles; ++t)
        if (SG_IN_RANGE(t < p.sk_slabs / k_tiles)) atomicAdd(&p.counters[t], 1 << 24);
}

// ------------------------------------------------------------------ main kernel
// Shared-memory ring and flags of one CTA, addressed by 32-bit shared-window
// addresses that all derive from one base register:
//   [ A stages | B stages | full barriers | empty barriers | abort flag ].
template <class Cfg>
struct Ring {
    uint32_t base;
    static constexpr uint32_t B_OFF = uint32_t(Cfg::STAGES * Cfg::A_STAGE) * 4u;
    static constexpr uint32_t BAR_OFF = B_OFF + uint32_t(Cfg::STAGES * Cfg::B_STAGE) * 4u;
    static constexpr uint32_t EPI_OFF = BAR_OFF + 16u * Cfg::STAGES + 16u;
    static constexpr uint32_t BYTES = EPI_OFF + (Cfg::STAGED_EPI ? uint32_t(Cfg::EPI_BYTES) : 0u);
    static_assert(EPI_OFF % 16 == 0, "staging areas take 128-bit accesses");

    __device__ uint32_t a(int s) const { return base + uint32_t(s * Cfg::A_STAGE) * 4u; }
    __device__ uint32_t b(int s) const { return base + B_OFF + uint32_t(s * Cfg::B_STAGE) * 4u; }
    __device__ uint32_t full(int s) const { return base + BAR_OFF + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + BAR_OFF + 8u * (Cfg::STAGES + s); }
    __device__ uint32_t abort_flag() const { return base + BAR_OFF + 16u * Cfg::STAGES; }
    __device__ bool aborted() const { return ld_shared_flag(abort_flag()) != 0; }
    __device__ void set_abort() const { st_shared_flag(abort_flag(), 1); }
    // epilogue staging area of consumer warp cw (StagedEpilogueConfig)
    __device__ uint32_t epi(int cw) const {
        return base + EPI_OFF + uint32_t(cw * Cfg::EPI_STAGE_FLOATS) * 4u;
    }
};

// State of the TMA issuer: the next slab to copy is slab `slab` of segment
// `seg` (tile coordinates tm, tn) into ring stage `stage`, whose empty barrier
// is in phase parity `phase`.
struct IssueState {
    SegmentIter iter;
    Segment seg;
    long long issued;
    int have, slab, tm, tn, stage;
    uint32_t phase;

    __device__ void init(const MainParams &p) {
        iter.init(p);
        issued = 0;
        have = 0;
        slab = tm = tn = stage = 0;
        phase = 0;
    }
};

// The issuer state of the batched kernel: also the batch of the current tile.
struct IssueStateEx : IssueState {
    int tb;
};

// The issuer state of the tall-batch kernel: also the first row of B of the
// current tile's batch.
struct IssueStateTall : IssueState {
    int b_row0;
};

template <class Cfg>
using IssueStateOf = typename std::conditional<
    Cfg::BATCH, IssueStateEx,
    typename std::conditional<Cfg::TALL, IssueStateTall, IssueState>::type>::type;

// Issue the copies of the next slab.  Returns false when there is none left or
// the wait for the stage to be released expired (abort).
template <class Cfg, class State>
__device__ __forceinline__ bool issue_one(State &st, const Ring<Cfg> &ring,
                                          const CUtensorMap *tmA, const CUtensorMap *tmB,
                                          const MainParams &p, const ExParams &x, int k_tiles) {
    if (ring.aborted()) return false;
    if (!st.have) {
        Segment sg;
        if (!st.iter.next(p, k_tiles, sg)) return false;
        st.seg = sg;
        st.have = 1;
        st.slab = sg.kb;
        int tm, tn;
        if constexpr (Cfg::BATCH) {
            int tb;
            decode_tile(p, sg.tile, tb, tm, tn);
            st.tb = tb;
        } else {
            tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            // the raster group (tile_coords) is the batch
            if constexpr (Cfg::TALL) st.b_row0 = (sg.tile / (p.group_m * p.tiles_n)) * x.tall_b_rows;
        }
        st.tm = tm;
        st.tn = tn;
    }
    const int s = st.stage;
    // range-checked build: the copy's box starts on a 16-byte boundary (x a
    // multiple of 4 floats), inside the k range, into a stage of the ring;
    // otherwise nothing is copied and the CTA aborts as after an expiry
    if (!SG_IN_RANGE(s >= 0 && s < Cfg::STAGES && st.slab >= 0 && st.slab < k_tiles &&
                     (st.tm * Cfg::BM) % 4 == 0 && (st.tn * Cfg::BN) % 4 == 0 &&
                     st.tm < p.tiles_m && st.tn < p.tiles_n)) {
        ring.set_abort();
        return false;
    }
    // first use of a stage: parity 1 refers to the phase before the barrier's
    // first one and counts as complete
    if (!mbar_wait_at(ring.empty(s), st.phase ^ 1u, p.timeout_ns)) {
        atomicOr(&g_error_word, ERR_EMPTY_WAIT);
        block_stream_k_tiles(p, k_tiles);
        ring.set_abort();
        return false;
    }
    mbar_arrive_expect_tx_at(ring.full(s), Cfg::STAGE_BYTES);
    if constexpr (Cfg::BATCH) {
        tma_load_3d_at(ring.a(s), tmA, ring.full(s), st.tm * Cfg::BM, st.slab * Cfg::BK,
                       x.a_planes > 1 ? st.tb : 0);
        tma_load_3d_at(ring.b(s), tmB, ring.full(s), st.tn * Cfg::BN, st.slab * Cfg::BK,
                       x.b_planes > 1 ? st.tb : 0);
    } else if constexpr (Cfg::TALL) {
        tma_load_2d_at(ring.a(s), tmA, ring.full(s), st.tm * Cfg::BM, st.slab * Cfg::BK);
        tma_load_2d_at(ring.b(s), tmB, ring.full(s), st.tn * Cfg::BN,
                       st.b_row0 + st.slab * Cfg::BK);
    } else {
        tma_load_2d_at(ring.a(s), tmA, ring.full(s), st.tm * Cfg::BM, st.slab * Cfg::BK);
        tma_load_2d_at(ring.b(s), tmB, ring.full(s), st.tn * Cfg::BN, st.slab * Cfg::BK);
    }
    st.issued = st.issued + 1;
    if (s + 1 == Cfg::STAGES) {
        st.stage = 0;
        st.phase ^= 1u;
    } else {
        st.stage = s + 1;
    }
    if (++st.slab == st.seg.ke) st.have = 0;
    return true;
}

// After an abort: wait for the last copies issued, so none is still writing
// shared memory when the CTA exits.  The wait is bounded by drain_limit_ns, not
// by the caller's limit that has just expired.
template <class Cfg>
__device__ __forceinline__ void drain_copies(const Ring<Cfg> &ring, long long issued,
                                             const MainParams &p) {
    const long long first = issued > Cfg::STAGES ? issued - Cfg::STAGES : 0;
    for (long long q = first; q < issued; ++q) {
        const int s = int(q % Cfg::STAGES);
        if (!mbar_wait_at(ring.full(s), uint32_t((q / Cfg::STAGES) & 1),
                          drain_limit_ns(p.timeout_ns))) {
            atomicOr(&g_error_word, ERR_DRAIN_WAIT);
            break;
        }
    }
}

// Stream-K fixup data of the current segment, written by consumer thread 0
// at the segment's start (where the integer divisions cost no accumulator
// registers) and read by all consumers after the segment's main loop.
struct FixInfo {
    long long tile_start;   // first slab of the tile in the stream-K range
    long long q0;           // sk_start(b_lo)
    int r0;                 // (b_lo * sk_slabs) mod gridDim.x
    int b_lo, b_hi;         // CTAs holding pieces of the tile
    int pieces;             // CTAs among them with a non-empty range
    int last;               // this CTA's piece completed the tile
};

// The consumer warps: FFMA micro-tiles over the ring, stream-K fixup and the
// epilogue.  `before_slab` runs before the wait for every slab (the issuer
// hook of ISSUE_THREAD0); `after_release(s)` runs on lane 0 of every warp
// right after the warp released stage s (the issuer hook of ISSUE_LAST_WARP).
//
// Register budget: the accumulators and two fragment buffers take TM*TN +
// 2*(TM+TN) registers for the whole main loop, so little else stays live
// across it: the ring is one base address, and the segment's tile, slot and
// stream-K constants are fetched again after the loop instead of being kept.
template <class Cfg, class Hook, class Release>
__device__ __forceinline__ void consumer_loop(const Ring<Cfg> &ring, const MainParams &p,
                                              const ExParams &x, int k_tiles, int cw, int ctid,
                                              FixInfo &fix,
                                              Hook &&before_slab, Release &&after_release) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TM = Cfg::TM, TN = Cfg::TN;
    constexpr int BAR_CONSUMERS = 1;
    const int lane = threadIdx.x & 31;
    // zig-zag lane map: lane bits {1,4} -> row group, bits {0,2,3} -> column group
    auto a_off = [&] {
        return (cw % Cfg::WARPS_M) * Cfg::WM + (((lane >> 1) & 1) | ((lane >> 3) & 2)) * 4;
    };
    auto b_off = [&] {
        return (cw / Cfg::WARPS_M) * Cfg::WN + ((lane & 1) | ((lane >> 1) & 6)) * 4;
    };
    // this thread's fragment addresses in stage 0; stage s adds s times the stage size
    const uint32_t a_base = ring.a(0) + uint32_t(a_off()) * 4u;
    const uint32_t b_base = ring.b(0) + uint32_t(b_off()) * 4u;

    int stage = 0;          // stage of the next slab to consume
    uint32_t phase = 0;     // parity of that stage's full barrier
    int q = 0;              // slabs consumed so far (AbortTestConfig only)
    for (int si = 0;; ++si) {
        int nslabs, slot;
        {
            Segment seg;
            if (!segment_at(p, k_tiles, si, seg)) break;
            nslabs = seg.ke - seg.kb;
            slot = seg.slot;
            if (slot >= 0 && ctid == 0) {
                const long long rel = seg.tile - p.dp_tiles;
                fix.tile_start = rel * k_tiles;
                fix.b_lo = sk_owner(fix.tile_start, p.sk_slabs, gridDim.x);
                fix.b_hi = sk_owner(fix.tile_start + k_tiles - 1, p.sk_slabs, gridDim.x);
                fix.q0 = sk_start(fix.b_lo, p.sk_slabs, gridDim.x);
                fix.r0 = int(((long long)fix.b_lo * p.sk_slabs) % gridDim.x);
                int pieces = 0;
                for (int b = fix.b_lo; b <= fix.b_hi; ++b)
                    pieces +=
                        sk_start(b, p.sk_slabs, gridDim.x) < sk_start(b + 1, p.sk_slabs, gridDim.x);
                fix.pieces = pieces;
            }
        }

        if constexpr (Cfg::STAGED_EPI) {
            if (p.beta != 0.0f) {
                Segment seg;
                segment_at(p, k_tiles, si, seg);
                int tm, tn;
                tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                prefetch_c_tile_rows<Cfg>(p, tm, tn, a_off(), b_off());
            }
        }

        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int jj = 0; jj < TN; ++jj) acc[i][jj] = 0.0f;

        for (int n = nslabs; n > 0; --n) {
            before_slab();
            const int s = stage;
            // Fast path: one try_wait that finds the slab already copied.  Only
            // if some lane misses it does the warp take a warp-uniform look at
            // the abort flag and enter the bounded wait.
            if (!__all_sync(0xffffffffu, mbar_try_wait_at(ring.full(s), phase)) &&
                !__any_sync(0xffffffffu, ring.aborted())) {
                bool ok = mbar_wait_at(ring.full(s), phase, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) {
                        atomicOr(&g_error_word, ERR_FULL_WAIT);
                        block_stream_k_tiles(p, k_tiles);
                    }
                    ring.set_abort();
                }
            }
            uint32_t a_s = a_base + uint32_t(s * Cfg::A_STAGE) * 4u;
            uint32_t b_s = b_base + uint32_t(s * Cfg::B_STAGE) * 4u;
            // range-checked build: every fragment this thread reads in the slab
            // lies in stage s (otherwise read the stage's start instead)
            if (!SG_IN_RANGE(
                    (a_s & 15u) == 0 && (b_s & 15u) == 0 && a_s >= ring.a(s) && b_s >= ring.b(s) &&
                    a_s + uint32_t((BK - 1) * BM + (TM / 4 - 1) * 16 + 4) * 4u <=
                        ring.a(s) + uint32_t(Cfg::A_STAGE) * 4u &&
                    b_s + uint32_t((BK - 1) * BN + (TN / 4 - 1) * 32 + 4) * 4u <=
                        ring.b(s) + uint32_t(Cfg::B_STAGE) * 4u)) {
                a_s = ring.a(s);
                b_s = ring.b(s);
            }
            // register double buffering of the fragments: the loads for k+1
            // are issued before the FMAs of k
            float fa[2][TM], fb[2][TN];
            load_fragments<Cfg>(a_s, b_s, fa[0], fb[0]);
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                if (kk + 1 < BK)
                    load_fragments<Cfg>(a_s + (kk + 1) * BM * 4, b_s + (kk + 1) * BN * 4,
                                        fa[(kk + 1) & 1], fb[(kk + 1) & 1]);
                outer_product<Cfg>(acc, fa[kk & 1], fb[kk & 1]);
            }
            __syncwarp();
            if (lane == 0) {
                if constexpr (Cfg::DROP_RELEASE_SLAB >= 0) {
                    if (!(blockIdx.x == 0 && cw == 0 && q == Cfg::DROP_RELEASE_SLAB))
                        mbar_arrive_at(ring.empty(s));
                } else {
                    mbar_arrive_at(ring.empty(s));
                }
                after_release(s);
            }
            ++q;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }

        bool finish = true;
        if (slot >= 0) {
            // ---- stream-K piece: publish the partial sums; the piece that
            // completes the tile's count adds all pieces in k order
            if (SG_IN_RANGE(slot >= 0 && slot < 2 * int(gridDim.x)))
                write_partial<Cfg>(acc, p.partials + (size_t)slot * (BM * BN), ctid);
            __threadfence();
            named_barrier(BAR_CONSUMERS, Cfg::CONSUMER_THREADS);
            if (ctid == 0) {
                const int rel_tile = int(fix.tile_start / k_tiles);
                if (SG_IN_RANGE(rel_tile >= 0 && rel_tile < p.sk_slabs / k_tiles)) {
                    const int before = atomicAdd(&p.counters[rel_tile], 1);
                    fix.last = (before == fix.pieces - 1);
                } else {
                    fix.last = 0;
                }
            }
            named_barrier(BAR_CONSUMERS, Cfg::CONSUMER_THREADS);
            finish = fix.last;
            const long long tile_start = fix.tile_start, q0 = fix.q0;
            const int r0 = fix.r0, b_lo = fix.b_lo, b_hi = fix.b_hi;
            // everyone has read `fix` before thread 0 can write it again
            named_barrier(BAR_CONSUMERS, Cfg::CONSUMER_THREADS);
            if (finish) {
                __threadfence();
                // sk_start(b + 1) = sk_start(b) + sk_q + carry, carry from sk_r:
                // additions only
                const long long sk_q = p.sk_slabs / gridDim.x;
                const int sk_r = int(p.sk_slabs % gridDim.x);
                // this CTA's own piece is read back too, so the sum order is the
                // k order whichever piece arrived last
#pragma unroll
                for (int i = 0; i < TM; ++i)
                    sum_pieces_row<Cfg>(acc[i], p.partials, i, ctid, b_lo, b_hi, q0, r0, sk_q, sk_r,
                                        tile_start);
            }
        }
        if (finish && !ring.aborted()) {
            Segment seg;
            segment_at(p, k_tiles, si, seg);
            int tm, tn;
            if constexpr (Cfg::BATCH) {
                int tb;
                decode_tile(p, seg.tile, tb, tm, tn);
                store_tile_ex<Cfg>(acc, p, x, tb, tm, tn, a_off(), b_off());
            } else if constexpr (Cfg::EX) {
                tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                store_tile_ex<Cfg>(acc, p, x, 0, tm, tn, a_off(), b_off());
            } else if constexpr (Cfg::STAGED_EPI) {
                tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                store_tile_staged<Cfg>(acc, p, tm, tn, a_off(), b_off(), ring.epi(cw));
            } else {
                tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                store_tile<Cfg>(acc, p, tm, tn, a_off(), b_off());
            }
        }
    }
}

// Persistent kernel.  Each CTA walks its segments (SegmentIter); the k-slabs of
// all its segments form one sequence q = 0, 1, 2, ...; slab q lives in ring
// stage q % STAGES.  The issuer copies a slab into a stage once every consumer
// warp has released the stage's previous contents (empty barrier); consumer
// warps wait on the full barrier of a stage (TMA byte count) before reading it.
//
// ISSUE_PRODUCER_WG: warpgroup 0 is the producer; it gives back registers
// (setmaxnreg.dec) and one of its threads issues all copies, STAGES ahead.  The
// consumer warps take the registers (setmaxnreg.inc).  Otherwise the CTA is
// the consumer warps alone: with ISSUE_THREAD0 consumer thread 0 issues slab
// q + STAGES - 1 when starting slab q; with ISSUE_LAST_WARP the warp that
// releases slab q last issues slab q + STAGES.
//
// A stream-K piece that is not a whole tile writes its partial sums to its
// slot and increments the tile's counter; the piece that brings the counter to
// the tile's piece count adds all pieces' slots in k order (so the result does
// not depend on which piece finishes last) and runs the epilogue.  No CTA ever
// waits for another.
//
// Expiry of a bounded wait sets a CTA-wide abort flag: from then on no thread
// waits again and nothing more is written to C; the stream-K tiles the CTA
// holds pieces of are made impossible to complete (block_stream_k_tiles), so
// they stay unwritten too; every
// consumer still passes the consumer barriers, and at the end the issuing
// thread waits for the copies it issued (drain_limit_ns).
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::CTAS_PER_SM)
    sgemm_tma_ffma_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const MainParams p,
                          const ExParams x) {
    constexpr int STAGES = Cfg::STAGES;
    constexpr int BAR_END = 2;

    static_assert(Ring<Cfg>::BYTES + 1024 <= Cfg::SMEM_BYTES, "ring fits the dynamic shared memory");
    extern __shared__ unsigned char smem_raw[];
    // stages 1024-byte aligned
    const Ring<Cfg> ring{(smem_addr(smem_raw) + 1023u) & ~1023u};
    __shared__ FixInfo fix;
    // issuer state in shared memory (ISSUE_THREAD0, ISSUE_LAST_WARP): keeping
    // it out of registers leaves them to the accumulators
    __shared__ IssueStateOf<Cfg> ist;
    __shared__ int released[STAGES];   // ISSUE_LAST_WARP: warps done with a stage

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(
            smem_raw + (ring.full(0) - smem_addr(smem_raw)));
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars[s], 1);
            mbar_init(&bars[STAGES + s], Cfg::CONSUMER_WARPS);
            released[s] = 0;
        }
        st_shared_flag(ring.abort_flag(), 0);
        ist.init(p);
        fence_barrier_init();
    }
    __syncthreads();

    const int k_tiles = (p.K + Cfg::BK - 1) / Cfg::BK;

    if constexpr (Cfg::WS) {
        if (warp < Cfg::PRODUCER_THREADS / 32) {
            // ======================================================== producer
            regs_decrease<Cfg::PRODUCER_REGS>();
            if (warp != 0) return;
            IssueStateOf<Cfg> st;
            st.init(p);
            if (lane == 0) {
                tma_prefetch_desc(&tmA);
                tma_prefetch_desc(&tmB);
                while (issue_one<Cfg>(st, ring, &tmA, &tmB, p, x, k_tiles)) {
                }
            }
            __syncwarp();
            // wait until every consumer is done, then (after an abort) make
            // sure no copy is still writing shared memory when the CTA exits
            named_barrier(BAR_END, 32 + Cfg::CONSUMER_THREADS);
            if (lane == 0 && ring.aborted()) drain_copies<Cfg>(ring, st.issued, p);
            return;
        }
        // ============================================================ consumers
        regs_increase<Cfg::CONSUMER_REGS>();
        consumer_loop<Cfg>(ring, p, x, k_tiles, warp - Cfg::PRODUCER_THREADS / 32,
                           threadIdx.x - Cfg::PRODUCER_THREADS, fix, [] {}, [](int) {});
        named_barrier(BAR_END, 32 + Cfg::CONSUMER_THREADS);
    } else if constexpr (Cfg::ISSUE == ISSUE_THREAD0) {
        if (threadIdx.x == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            for (int i = 0; i < STAGES - 1; ++i) issue_one<Cfg>(ist, ring, &tmA, &tmB, p, x, k_tiles);
        }
        consumer_loop<Cfg>(
            ring, p, x, k_tiles, warp, threadIdx.x, fix,
            [&] {
                if (threadIdx.x == 0) issue_one<Cfg>(ist, ring, &tmA, &tmB, p, x, k_tiles);
            },
            [](int) {});
        if (threadIdx.x == 0 && ring.aborted()) drain_copies<Cfg>(ring, ist.issued, p);
    } else {
        // ISSUE_LAST_WARP: thread 0 fills every stage once; afterwards the warp
        // whose release completes a stage's count copies the next slab into it
        // at once, so no warp waits for the others.  Slab q + STAGES goes into
        // the stage of slab q, and the releases of slab q all precede those of
        // q + 1, so the elected warps use `ist` one at a time, in slab order.
        if (threadIdx.x == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            for (int i = 0; i < STAGES; ++i) issue_one<Cfg>(ist, ring, &tmA, &tmB, p, x, k_tiles);
        }
        consumer_loop<Cfg>(ring, p, x, k_tiles, warp, threadIdx.x, fix, [] {}, [&](int s) {
            __threadfence_block();
            if (atomicAdd(&released[s], 1) == Cfg::CONSUMER_WARPS - 1) {
                released[s] = 0;
                __threadfence_block();
                issue_one<Cfg>(ist, ring, &tmA, &tmB, p, x, k_tiles);
            }
        });
        // every warp is past its last issue before the copies are counted
        __syncthreads();
        if (threadIdx.x == 0 && ring.aborted()) drain_copies<Cfg>(ring, ist.issued, p);
    }
}

}  // namespace sg

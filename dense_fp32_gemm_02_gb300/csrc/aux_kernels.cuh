// aux_kernels.cuh -- the kernels around the FP32 SGEMM's main kernel: the
// A-transpose pre-pass (single and batched), the B re-pitch copy, the
// alpha == 0 / K == 0 scaling kernel, the deferred beta * C_in addition of the
// host-buffer pipeline, the direct kernel for small problems and the
// bounded-wait self test.  Non-template kernels: included by sgemm.cu only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.cuh"

namespace sg {

// ------------------------------------------------------------------ pre-pass
// At[k][m] = A[m][k] for the 64x64 tile at (m0, k0), through shared memory,
// 256 threads: each thread has 16 independent loads in flight (coalesced
// along k) and then 16 stores (coalesced along m).
__device__ __forceinline__ void transpose_tile(const float *__restrict__ A, long long lda, int M,
                                               int K, float *__restrict__ At, long long ldat,
                                               long long m0, long long k0,
                                               float (&tile)[64][65]) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;   // 8 warps
    float v[16];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const long long m = m0 + w * 8 + r;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long k = k0 + lane + 32 * h;
            v[2 * r + h] = (m < M && k < K) ? __ldcs(A + m * lda + k) : 0.0f;
        }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) tile[w * 8 + r][lane + 32 * h] = v[2 * r + h];
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const long long k = k0 + w * 8 + r;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long m = m0 + lane + 32 * h;
            if (k < K && m < M && SG_IN_RANGE(m < ldat))
                At[k * ldat + m] = tile[lane + 32 * h][w * 8 + r];
        }
    }
    __syncthreads();
}

// At[k][m] = A[m][k] for one plane: the block grid (x along k, y along m)
// walks its 64x64 tiles.
__device__ __forceinline__ void transpose_plane(const float *__restrict__ A, long long lda, int M,
                                                int K, float *__restrict__ At, long long ldat) {
    __shared__ float tile[64][65];
    for (long long m0 = (long long)blockIdx.y * 64; m0 < M; m0 += (long long)gridDim.y * 64)
        for (long long k0 = (long long)blockIdx.x * 64; k0 < K; k0 += (long long)gridDim.x * 64)
            transpose_tile(A, lda, M, K, At, ldat, m0, k0, tile);
}

// The pre-pass of a single GEMM.  Block (0,0) also zeroes `zero_count` ints at
// `zero` (the stream-K tile counters of the GEMM that follows on the stream).
__global__ void __launch_bounds__(256)
    pack_a_transpose_kernel(const float *__restrict__ A, long long lda, int M, int K,
                            float *__restrict__ At, long long ldat, int *zero, int zero_count) {
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero[i] = 0;
    transpose_plane(A, lda, M, K, At, ldat);
}

// The batched pre-pass: plane z = blockIdx.z transposes A + z * stride_a into
// At + z * at_plane (the host launches at most 65535 planes per call).  Held to
// 64 registers (four blocks per SM).
__global__ void __launch_bounds__(256, 4)
    pack_a_transpose_batched_kernel(const float *__restrict__ A, long long lda, long long stride_a,
                                    int M, int K, float *__restrict__ At, long long ldat,
                                    long long at_plane, int *zero, int zero_count) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero[i] = 0;
    transpose_plane(A + (long long)blockIdx.z * stride_a, lda, M, K,
                    At + (long long)blockIdx.z * at_plane, ldat);
}

// Bp[k][n] = B[k][n] with a 16-byte row pitch (ldbp % 4 == 0) and a 16-byte
// plane pitch for the TMA, plane by plane (batch z of B at B + z * stride_b).
// One block row per k (grid-stride), threads along n.
__global__ void __launch_bounds__(256)
    pack_b_copy_kernel(const float *__restrict__ B, long long ldb, long long stride_b, int K,
                       int N, float *__restrict__ Bp, long long ldbp, long long bp_plane,
                       int planes) {
    for (int z = blockIdx.z; z < planes; z += gridDim.z) {
        for (long long k = blockIdx.y; k < K; k += gridDim.y) {
            const float *src = B + (long long)z * stride_b + k * ldb;
            float *dst = Bp + (long long)z * bp_plane + k * ldbp;
            for (long long n = (long long)blockIdx.x * blockDim.x + threadIdx.x; n < N;
                 n += (long long)gridDim.x * blockDim.x)
                if (SG_IN_RANGE(n < ldbp)) dst[n] = __ldcs(src + n);
        }
    }
}

// The pre-pass of one GEMM whose B must be re-pitched, in one launch: blocks
// [0, a_blocks) walk the 64x64 tiles of the A transpose, the others walk
// strips of 16 rows x 256 columns of the B copy (a thread copies one column
// of a strip: 16 loads in flight, coalesced along n; the rows of B need not
// be 16-byte aligned, those of Bp are).  Block 0 also zeroes `zero_count`
// ints at `zero` (the stream-K tile counters of the GEMM that follows).
__global__ void __launch_bounds__(256)
    pack_ab_kernel(const float *__restrict__ A, long long lda, int M, int K,
                   float *__restrict__ At, long long ldat, const float *__restrict__ B,
                   long long ldb, int N, float *__restrict__ Bp, long long ldbp, int a_blocks,
                   int *zero, int zero_count) {
    __shared__ float tile[64][65];
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero[i] = 0;
    if (int(blockIdx.x) < a_blocks) {
        const long long kt = (K + 63) / 64, tiles = kt * ((M + 63) / 64);
        for (long long t = blockIdx.x; t < tiles; t += a_blocks)
            transpose_tile(A, lda, M, K, At, ldat, (t / kt) * 64, (t % kt) * 64, tile);
        return;
    }
    const long long nt = (N + 255) / 256, strips = nt * ((K + 15) / 16);
    const long long b_blocks = gridDim.x - a_blocks;
    for (long long t = blockIdx.x - a_blocks; t < strips; t += b_blocks) {
        const long long k0 = (t / nt) * 16, n = (t % nt) * 256 + threadIdx.x;
        if (n >= N) continue;
        float v[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = (k0 + r < K) ? __ldcs(B + (k0 + r) * ldb + n) : 0.0f;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (k0 + r < K && SG_IN_RANGE(n < ldbp)) Bp[(k0 + r) * ldbp + n] = v[r];
    }
}

// C = act(beta * C + bias) on each batch's M x N block (C not read when
// beta == 0): the alpha == 0 / K == 0 case, where A and B are not read.
__global__ void __launch_bounds__(256)
    scale_c_kernel(float *C, long long ldc, long long stride_c, int M, int N, int batch,
                   float beta, const float *bias, long long stride_bias, int act) {
    const long long per = (long long)M * N, total = per * batch;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long b = idx / per, rem = idx - b * per;
        const long long i = rem / N, j = rem - i * N;
        float *c = C + b * stride_c + i * ldc + j;
        float v = (beta == 0.0f) ? 0.0f : beta * *c;
        if (bias) v += bias[b * stride_bias + j];
        *c = activate(v, act);
    }
}

// C += beta * X over an M x N block (row pitches ldc and ldx): the deferred
// beta * C_in term of the host-buffer pipeline's first row block.
__global__ void __launch_bounds__(256)
    add_scaled_kernel(float *C, long long ldc, const float *__restrict__ X, long long ldx, int M,
                      int N, float beta) {
    const long long total = (long long)M * N;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / N, j = idx - i * N;
        float *c = C + i * ldc + j;
        *c = fmaf(beta, X[i * ldx + j], *c);
    }
}

// ------------------------------------------------------------------ small problems
// C = alpha*A*B + beta*C for problems too small to fill the GPU with the
// persistent kernel's 256x128 tiles: one CTA per TS x TS output tile (TS 64,
// or 32 when 64x64 tiles would leave most SMs idle), reading A and B directly
// (any leading dimension or alignment), no pre-pass, no workspace, one launch.
// 256 threads in a 16x16 grid, (TS/16) x (TS/16) outputs each; k in steps of
// 32 through shared memory (A stored transposed, as in the pages' tiled
// kernel), the next step's operands loaded into registers meanwhile.  Every
// output sums its k terms in ascending order with fused multiply-adds, so the
// result is deterministic.
constexpr int SMALL_BK = 32;

// This thread's TS/16 x TS/16 outputs of the tile at blockIdx.(y, x), summed
// over k in [kb, ke) (acc starts at zero).
template <int TS>
__device__ __forceinline__ void small_tile_sum(float (&acc)[TS / 16][TS / 16], int M, int N,
                                               const float *__restrict__ A, long long lda,
                                               const float *__restrict__ B, long long ldb,
                                               int kb, int ke) {
    constexpr int T = TS / 16;                       // outputs per thread along each side
    constexpr int LOADS = TS * SMALL_BK / 256;       // elements of A (and of B) per thread
    __shared__ float As[SMALL_BK][TS + 4];           // As[k][m]
    __shared__ float Bs[SMALL_BK][TS + 4];           // Bs[k][n]
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const long long row0 = (long long)blockIdx.y * TS, col0 = (long long)blockIdx.x * TS;
#pragma unroll
    for (int i = 0; i < T; ++i)
#pragma unroll
        for (int j = 0; j < T; ++j) acc[i][j] = 0.0f;
    // TS x BK of A and BK x TS of B per step: consecutive threads along k for A
    // and along n for B (coalesced); the next step's values are loaded into
    // registers while the current step's FMAs run
    float ra[LOADS], rb[LOADS];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int q = 0; q < LOADS; ++q) {
            const int e = threadIdx.x + q * 256;
            const long long gr = row0 + e / SMALL_BK;
            const int gk = k0 + e % SMALL_BK;
            ra[q] = (gr < M && gk < ke) ? A[gr * lda + gk] : 0.0f;
            const long long gc = col0 + e % TS;
            const int gkb = k0 + e / TS;
            rb[q] = (gkb < ke && gc < N) ? B[(long long)gkb * ldb + gc] : 0.0f;
        }
    };
    fetch(kb);
    for (int k0 = kb; k0 < ke; k0 += SMALL_BK) {
#pragma unroll
        for (int q = 0; q < LOADS; ++q) {
            const int e = threadIdx.x + q * 256;
            As[e % SMALL_BK][e / SMALL_BK] = ra[q];
            Bs[e / TS][e % TS] = rb[q];
        }
        __syncthreads();
        if (k0 + SMALL_BK < ke) fetch(k0 + SMALL_BK);
#pragma unroll
        for (int kk = 0; kk < SMALL_BK; ++kk) {
            float a[T], b[T];
#pragma unroll
            for (int i = 0; i < T; ++i) a[i] = As[kk][ty * T + i];
#pragma unroll
            for (int j = 0; j < T; ++j) b[j] = Bs[kk][tx * T + j];
#pragma unroll
            for (int i = 0; i < T; ++i)
#pragma unroll
                for (int j = 0; j < T; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
}

// alpha/beta update of this thread's outputs of the tile at blockIdx.(y, x)
template <int TS>
__device__ __forceinline__ void small_tile_store(const float (&acc)[TS / 16][TS / 16], int M, int N,
                                                 float alpha, float beta, float *__restrict__ C,
                                                 long long ldc) {
    constexpr int T = TS / 16;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const long long row0 = (long long)blockIdx.y * TS, col0 = (long long)blockIdx.x * TS;
#pragma unroll
    for (int i = 0; i < T; ++i) {
        const long long r = row0 + ty * T + i;
        if (r >= M) continue;
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const long long c = col0 + tx * T + j;
            if (c >= N) continue;
            float *out = C + r * ldc + c;
            *out = (beta != 0.0f) ? fmaf(alpha, acc[i][j], beta * *out) : alpha * acc[i][j];
        }
    }
}

template <int TS>
__global__ void __launch_bounds__(256)
    sgemm_small_kernel(int M, int N, int K, float alpha, const float *__restrict__ A,
                       long long lda, const float *__restrict__ B, long long ldb, float beta,
                       float *__restrict__ C, long long ldc) {
    float acc[TS / 16][TS / 16];
    small_tile_sum<TS>(acc, M, N, A, lda, B, ldb, 0, K);
    small_tile_store<TS>(acc, M, N, alpha, beta, C, ldc);
}

// The small-problem kernel with the k range split over the CTAs of a
// thread-block cluster of 1 x 1 x S (S = gridDim.z, at most 8): a tile's S
// CTAs sum k in [z * kchunk, (z + 1) * kchunk) each, so a problem of few
// tiles keeps S times as many SMs busy and each CTA walks 1/S of the k
// steps.  CTAs 1 .. S-1 leave their partial sums in their shared memory; CTA
// 0 adds them to its own in the order z = 1, 2, ... through distributed
// shared memory and runs the alpha/beta update, so the result does not depend
// on which CTA finishes first.  A second cluster barrier keeps every CTA's
// shared memory until CTA 0 has read it.
template <int TS>
__global__ void __launch_bounds__(256)
    sgemm_small_splitk_kernel(int M, int N, int K, int kchunk, float alpha,
                              const float *__restrict__ A, long long lda,
                              const float *__restrict__ B, long long ldb, float beta,
                              float *__restrict__ C, long long ldc) {
    constexpr int T = TS / 16;
    __shared__ float part[T * T][256];   // [output][thread]: a warp's accesses are contiguous
    const int z = int(cluster_ctarank());
    const int kb = z * kchunk;
    const int ke = int(min((long long)K, (long long)kb + kchunk));
    float acc[T][T];
    small_tile_sum<TS>(acc, M, N, A, lda, B, ldb, kb, ke);
    if (z != 0) {
#pragma unroll
        for (int i = 0; i < T; ++i)
#pragma unroll
            for (int j = 0; j < T; ++j) part[i * T + j][threadIdx.x] = acc[i][j];
    }
    cluster_barrier();   // the partial sums are visible to CTA 0
    if (z == 0) {
        const uint32_t mine = smem_addr(&part[0][threadIdx.x]);
        for (int r = 1; r < int(gridDim.z); ++r) {
            if (!SG_IN_RANGE(r < 8)) break;
            const uint32_t peer = dsmem_map(mine, uint32_t(r));
#pragma unroll
            for (int i = 0; i < T; ++i)
#pragma unroll
                for (int j = 0; j < T; ++j)
                    acc[i][j] += dsmem_ld_f32(peer + uint32_t((i * T + j) * 256) * 4u);
        }
        small_tile_store<TS>(acc, M, N, alpha, beta, C, ldc);
    }
    cluster_barrier();   // no CTA leaves while CTA 0 may still read its shared memory
}

// ------------------------------------------------------------------ skinny M
// GEMMs with at most SKINNY_ROWS rows of A and C.  Every element of B is used
// by M <= 32 FMAs only, so the work is bound by reading B once from HBM (at
// M = 1 it is a vector-matrix product), not by the FMA units the tiled
// kernels are built for.  Block (x, y) owns columns x * 256 * COLS + t + 256 q
// (q < COLS) for thread t, so every warp load of B covers 128 contiguous
// bytes of one row without any alignment rule, and the k range
// [y * kchunk, min(K, (y + 1) * kchunk)): the grid's y dimension splits K so
// that a few column blocks still fill every SM.  A's rows of each 128-deep
// sub-range sit in shared memory, k-major, read by all threads at once (four
// rows per 128-bit read).  MINB: blocks per SM the register allocation leaves
// room for; UNR: k steps unrolled.  Each element sums its k terms in ascending order by fp32 FMAs;
// with one k range the block applies alpha / beta and writes C, otherwise it
// writes its partial sums to P (range y at P + y * M * N, row-major M x N)
// and skinny_reduce_kernel adds the ranges in y order.
constexpr int SKINNY_ROWS = 32;
constexpr int SKINNY_THREADS = 256;
constexpr int SKINNY_KSUB = 128;     // k values of A staged in shared memory at a time

template <int MR, int COLS, int MINB, int UNR>
__global__ void __launch_bounds__(SKINNY_THREADS, MINB)
    sgemm_skinny_kernel(int M, int N, int K, int kchunk, float alpha, const float *__restrict__ A,
                        long long lda, const float *__restrict__ B, long long ldb, float beta,
                        float *__restrict__ C, long long ldc, float *__restrict__ P) {
    // A's sub-range k-major: the MR values of one k are contiguous (128-bit reads)
    __shared__ __align__(16) float As[SKINNY_KSUB][MR];
    const int t = threadIdx.x;
    const long long col0 = (long long)blockIdx.x * (SKINNY_THREADS * COLS) + t;
    // (the end in 64 bits: kb + kchunk may pass 2^31 when K is close to it)
    const int kb = int(blockIdx.y) * kchunk;
    const int ke = int(min((long long)K, (long long)kb + kchunk));
    float acc[MR][COLS];
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int q = 0; q < COLS; ++q) acc[i][q] = 0.0f;
    for (int k0 = kb; k0 < ke; k0 += SKINNY_KSUB) {
        const int kn = min(SKINNY_KSUB, ke - k0);
        __syncthreads();   // the previous sub-range's reads of As are done
        for (int e = t; e < MR * SKINNY_KSUB; e += SKINNY_THREADS) {
            const int i = e % MR, kk = e / MR;
            As[kk][i] = (i < M && kk < kn) ? A[(long long)i * lda + k0 + kk] : 0.0f;
        }
        __syncthreads();
        // UNR k steps in flight: UNR x COLS loads of B per thread
#pragma unroll UNR
        for (int kk = 0; kk < kn; ++kk) {
            const float *brow = B + (long long)(k0 + kk) * ldb;
            float b[COLS];
#pragma unroll
            for (int q = 0; q < COLS; ++q) {
                const long long col = col0 + q * SKINNY_THREADS;
                b[q] = col < N ? __ldcs(brow + col) : 0.0f;
            }
            if constexpr (MR % 4 == 0) {
#pragma unroll
                for (int i = 0; i < MR; i += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(&As[kk][i]);
#pragma unroll
                    for (int q = 0; q < COLS; ++q) {
                        acc[i][q] = fmaf(a4.x, b[q], acc[i][q]);
                        acc[i + 1][q] = fmaf(a4.y, b[q], acc[i + 1][q]);
                        acc[i + 2][q] = fmaf(a4.z, b[q], acc[i + 2][q]);
                        acc[i + 3][q] = fmaf(a4.w, b[q], acc[i + 3][q]);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < MR; ++i) {
                    const float a = As[kk][i];
#pragma unroll
                    for (int q = 0; q < COLS; ++q) acc[i][q] = fmaf(a, b[q], acc[i][q]);
                }
            }
        }
    }
    const bool split = gridDim.y > 1;
#pragma unroll
    for (int i = 0; i < MR; ++i) {
        if (i >= M) break;
#pragma unroll
        for (int q = 0; q < COLS; ++q) {
            const long long col = col0 + q * SKINNY_THREADS;
            if (col >= N) continue;
            if (split) {
                // range-checked build: the partial sum lies in P's S x M x N floats
                const long long pi = ((long long)blockIdx.y * M + i) * N + col;
                if (SG_IN_RANGE(pi < (long long)gridDim.y * M * N)) P[pi] = acc[i][q];
            } else {
                float *out = C + (long long)i * ldc + col;
                *out = (beta != 0.0f) ? fmaf(alpha, acc[i][q], beta * *out) : alpha * acc[i][q];
            }
        }
    }
}

// ------------------------------------------------------------------ skinny N
// GEMMs with at most SKINNY_COLS_MAX columns of B and C (at N = 1 a
// matrix-vector product): A, M x K, is the operand read once from HBM, and a
// tiled kernel would pad N up to its 128-column tile and transpose all of A
// first.  Block (x, y) owns rows x * 128 .. x * 128 + 127, one per thread, and
// the k range [y * kchunk, min(K, (y + 1) * kchunk)).  Its 32-deep steps of A
// (each warp copies one row's 128 contiguous bytes at a time; no alignment
// rule) and of B (k-major) go into shared memory by asynchronous copies, two
// steps in flight: the next step is being copied while the threads add this
// step's 32 terms of their row to their NR accumulators in k order, B read
// four columns at a time (the same address for every thread).  Output as in
// sgemm_skinny_kernel: alpha / beta into C with one k range, partial sums to
// P (range y at P + y * M * N) otherwise.
constexpr int SKINNY_COLS_MAX = 32;
constexpr int SKINNY_N_ROWS = 128;   // rows per block, one per thread
constexpr int SKINNY_N_KC = 32;      // k values per staged step

template <int NR>
__global__ void __launch_bounds__(SKINNY_N_ROWS)
    sgemm_skinny_n_kernel(int M, int N, int K, int kchunk, float alpha, const float *__restrict__ A,
                          long long lda, const float *__restrict__ B, long long ldb, float beta,
                          float *__restrict__ C, long long ldc, float *__restrict__ P) {
    static_assert(NR % 4 == 0, "B is read four columns at a time");
    constexpr int KC = SKINNY_N_KC, ROWS = SKINNY_N_ROWS;
    __shared__ float As[2][ROWS][KC + 1];                 // +1: rows in distinct banks
    __shared__ __align__(16) float Bs[2][KC][NR];
    const int t = threadIdx.x, lane = t % 32, warp = t / 32;
    const long long row0 = (long long)blockIdx.x * ROWS;
    // (the end in 64 bits: kb + kchunk may pass 2^31 when K is close to it)
    const int kb = int(blockIdx.y) * kchunk;
    const int ke = int(min((long long)K, (long long)kb + kchunk));
    const int steps = (ke - kb + KC - 1) / KC;
    // copies of step s into buffer s % 2: warp w takes rows w, w + 4, ...,
    // lane l column k0 + l; past M or the k range the copy reads nothing and
    // zero-fills (its source address stays A's or B's first element)
    auto issue = [&](int s) {
        const int k0 = kb + s * KC, buf = s & 1;
        const int kn = min(KC, ke - k0);
#pragma unroll
        for (int r = warp; r < ROWS; r += ROWS / 32) {
            const long long row = row0 + r;
            const bool ok = row < M && lane < kn;
            cp_async4(smem_addr(&As[buf][r][lane]), ok ? A + row * lda + k0 + lane : A,
                      ok ? 4u : 0u);
        }
        for (int e = t; e < KC * NR; e += ROWS) {
            const int kk = e / NR, j = e % NR;
            const bool ok = kk < kn && j < N;
            cp_async4(smem_addr(&Bs[buf][kk][j]), ok ? B + (long long)(k0 + kk) * ldb + j : B,
                      ok ? 4u : 0u);
        }
    };
    float acc[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) acc[j] = 0.0f;
    if (steps > 0) issue(0);
    cp_async_commit();
    for (int s = 0; s < steps; ++s) {
        if (s + 1 < steps) issue(s + 1);
        cp_async_commit();
        cp_async_wait<1>();   // step s has landed (this thread's copies)
        __syncthreads();      // and every other thread's
        const int buf = s & 1;
#pragma unroll 8
        for (int kk = 0; kk < KC; ++kk) {
            const float a = As[buf][t][kk];
#pragma unroll
            for (int j = 0; j < NR; j += 4) {
                const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][j]);
                acc[j] = fmaf(a, b4.x, acc[j]);
                acc[j + 1] = fmaf(a, b4.y, acc[j + 1]);
                acc[j + 2] = fmaf(a, b4.z, acc[j + 2]);
                acc[j + 3] = fmaf(a, b4.w, acc[j + 3]);
            }
        }
        __syncthreads();      // buffer s % 2 is free for step s + 2
    }
    cp_async_wait<0>();
    const long long row = row0 + t;
    if (row >= M) return;
    const bool split = gridDim.y > 1;
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        if (j >= N) break;
        if (split) {
            // range-checked build: the partial sum lies in P's S x M x N floats
            const long long pi = ((long long)blockIdx.y * M + row) * N + j;
            if (SG_IN_RANGE(pi < (long long)gridDim.y * M * N)) P[pi] = acc[j];
        } else {
            float *out = C + row * ldc + j;
            *out = (beta != 0.0f) ? fmaf(alpha, acc[j], beta * *out) : alpha * acc[j];
        }
    }
}

// C[i][j] = alpha * (P_0 + P_1 + ... + P_{S-1})[i][j] + beta * C[i][j], the
// ranges added in order (C not read when beta == 0).
__global__ void __launch_bounds__(256)
    skinny_reduce_kernel(int M, int N, int S, const float *__restrict__ P, float alpha, float beta,
                         float *__restrict__ C, long long ldc) {
    const long long total = (long long)M * N;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long i = e / N, j = e - i * N;
        if (!SG_IN_RANGE(i < M && j < N)) continue;
        float sum = P[e];
        for (int y = 1; y < S; ++y) sum += P[(long long)y * total + e];
        float *out = C + i * ldc + j;
        *out = (beta != 0.0f) ? fmaf(alpha, sum, beta * *out) : alpha * sum;
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

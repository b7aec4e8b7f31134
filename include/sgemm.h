/*
 * sgemm.h -- C ABI of the GB300 (sm_103a) FP32 SGEMM library, libsgemm.so.
 *
 * Operation (all entry points that compute):
 *
 *     C[i*ldc + j] = alpha * sum_{k<K} A[i*lda + k] * B[k*ldb + j]  +  beta * C[i*ldc + j]
 *
 * for 0 <= i < M, 0 <= j < N: row-major FP32, A is M x K, B is K x N, C is M x N.
 * This is the computation stated with the naive kernel of "How to implement
 * matrix multiplication efficiently? An introduction from a CUDA beginner's
 * view" (makelele.cn repost of the Hands-on-GEMM article, section "Naive GEMM
 * and prerequisites": row-major A (M rows, K columns), B (K rows, N columns),
 * C (M rows, N columns), c = alpha*A*B + beta*C with alpha applied after the
 * k sum), with BLAS-style leading dimensions added.
 *
 * Conventions shared by every entry point:
 *  - Sizes are elements.  lda >= max(1,K), ldb >= max(1,N), ldc >= max(1,N).
 *  - M, N and K are at most 2^31 - 65536 (SGEMM_ERR_TOO_LARGE above that).
 *  - beta == 0: C is not read on input (NaN/Inf in it do not propagate).
 *  - alpha == 0 or K == 0: A and B are not read; C = beta*C (0 when beta == 0).
 *  - M == 0 or N == 0: nothing is read or written; returns SGEMM_OK.
 *  - Elements of C outside the M x N block (columns N..ldc-1) are never written.
 *  - Pointers must be 4-byte aligned; no other alignment is required.
 *  - C must not overlap A or B (not checked).
 *  - Summation order is fixed per build, shape and GPU model: results are bitwise
 *    reproducible run to run.  On the FFMA path each element's k terms are
 *    accumulated by fp32 fused multiply-adds over k ascending; where the work
 *    split cuts a tile along k (stream-K), the pieces' partial sums are added in
 *    k order.  alpha and beta are applied once, after the sum.
 *  - Nothing here exits or aborts the process: every failure is a status code.
 */
#ifndef DENSE_FP32_GEMM_02_GB300_SGEMM_H
#define DENSE_FP32_GEMM_02_GB300_SGEMM_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so that this header needs
 * no CUDA headers.  NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *sgemm_stream_t;

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1,        /* a size, leading dimension or pointer is invalid */
    SGEMM_ERR_UNSUPPORTED_DEVICE = 2, /* the current CUDA device is not sm_103 */
    SGEMM_ERR_CUDA = 3,               /* a CUDA runtime/driver call failed; see sgemm_last_cuda_error() */
    SGEMM_ERR_TIMEOUT = 4,            /* a bounded in-kernel wait expired (reported by sgemm_device_status) */
    SGEMM_ERR_ALLOC = 5,              /* device or pinned workspace allocation failed */
    SGEMM_ERR_TOO_LARGE = 6,          /* a size past 2^31 - 65536, or (sgemm_noalloc) the problem
                                         does not fit its fixed scratch */
    SGEMM_ERR_BOUNDS = 7              /* range-checked build only: an index was out of range
                                         (reported by sgemm_device_status) */
} sgemm_status;

/*
 * sgemm -- the GEMM on device memory, asynchronous on `stream`.
 *
 * A, B, C: device pointers owned by the caller; the library keeps no reference
 * after the call returns.  The work is enqueued on `stream` and the call returns
 * without synchronising.  A, B and C must stay valid until that work completes.
 * The library may use a device workspace for a transposed copy of A (K rows of
 * M floats, M rounded up to a multiple of 4) and, when B's row
 * pitch or address does not meet the 16-byte rule of the tensor-memory
 * accelerator, a padded copy of B.  The workspace comes from a stream-ordered
 * memory pool owned by the library (one per device) and is returned to it on
 * `stream` after the last kernel that reads it.
 *
 * Returns SGEMM_OK once the work is enqueued; errors raised by the device while
 * the kernels run surface on the caller's next synchronisation of `stream`, and
 * a bounded-wait expiry inside the kernel through sgemm_device_status().
 */
int sgemm(int M, int N, int K, float alpha,
          const float *A, int lda,
          const float *B, int ldb,
          float beta, float *C, int ldc,
          sgemm_stream_t stream);

/* Activation of the fused epilogue of sgemm_ex. */
typedef enum {
    SGEMM_ACT_NONE = 0, /* identity */
    SGEMM_ACT_RELU = 1, /* max(z, 0) */
    SGEMM_ACT_GELU = 2  /* z * Phi(z) = 0.5 z (1 + erf(z / sqrt 2)) */
} sgemm_act;

/*
 * sgemm_ex -- strided batched GEMM with a fused bias and activation, on device
 * memory, asynchronous on `stream`.
 *
 * For b = 0 .. batch-1, with X_b = X + b * stride_x (strides in elements):
 *
 *   C_b[i][j] = act( alpha * sum_k A_b[i][k] * B_b[k][j] + beta * C_b[i][j] + bias_b[j] )
 *
 * Row-major like sgemm, with the same leading-dimension rules.  The article
 * "How to implement matrix multiplication efficiently? An introduction from a
 * CUDA beginner's view" (introduction) motivates the GEMM by neural-network
 * layers and names operator fusion with it as the next step; it fixes neither
 * a bias nor an activation, so this entry point takes the layer form: a bias
 * per output column (broadcast over the rows; bias == NULL for none) and an
 * element-wise activation `act` (sgemm_act).  batch == 1, bias == NULL and
 * SGEMM_ACT_NONE is exactly sgemm().
 *
 * stride_a or stride_b 0 means every batch uses the same A or B.  Batches of C
 * must not overlap: batch > 1 requires stride_c >= (M - 1) * ldc + N.  C is not
 * read when beta == 0; when K == 0 or alpha == 0, A and B are not read and
 * C_b = act(beta * C_b + bias_b).  Ownership, workspace and asynchrony are as
 * for sgemm(); the workspace holds one transposed A per batch (one when
 * stride_a == 0).
 *
 * A batch with no bias and no activation, its own A per batch, M a multiple of
 * 256 up to 4096, K a multiple of 64 and stride_c == M * ldc (batches of C one
 * under the other) runs as one (batch*M) x N GEMM on the plain kernel; B is
 * then read in place when shared or when stride_b == K * ldb, and re-pitched
 * that way when its rows break the 16-byte rule.  Other batches run the
 * batched kernel.  Either way the result meets sgemm()'s tolerance and is
 * bitwise the same from call to call.
 *
 * Errors: SGEMM_ERR_INVALID_ARG for a negative size, batch or stride, an
 * unknown `act`, a bias pointer not 4-byte aligned, overlapping batches of C,
 * or any condition sgemm() rejects; batch == 0 (like M == 0 or N == 0) is a
 * successful no-op.  The other codes are those of sgemm().
 */
int sgemm_ex(int M, int N, int K, float alpha,
             const float *A, int lda, long long stride_a,
             const float *B, int ldb, long long stride_b,
             float beta, float *C, int ldc, long long stride_c,
             int batch, const float *bias, long long stride_bias, int act,
             sgemm_stream_t stream);

/*
 * sgemm_host -- the same GEMM on HOST buffers; synchronous.
 *
 * A, B, C are host pointers (page-locked memory gives the fastest copies, but
 * pageable memory is accepted).  The call works through row blocks of A and C
 * (M >= 2048: a first block of 1024 rows, a last one of 512, blocks of about
 * 2048 rows between them; one block otherwise): block i is copied in on a
 * host-to-device copy stream, multiplied on `stream` while block i+1 is
 * copied in, and copied back into C (respecting ldc) on a device-to-host copy
 * stream while block i+1 is multiplied.  When K >= 4096, block 0 and B are
 * copied in k-chunks (columns of A, rows of B: the first K/8 deep, each next
 * one half again as deep) and block 0 is multiplied chunk by chunk as they
 * land, the first chunk with beta = 0 and the others accumulating into its C
 * rows; beta * C_in is added to block 0 after its C_in has been copied in
 * behind the chunks.  So the first GEMM waits for an eighth of B and of A's
 * first block only.  Device buffers come from the library pool; the two copy
 * streams are the library's own (one pair per device).  `stream` is
 * synchronised before returning, so C holds the result on return.  Results
 * meet the same tolerance as sgemm(); they need not be bitwise equal to one
 * sgemm() call on the whole matrix (row blocks change the k split of leftover
 * tiles, and the k-chunks of block 0 round its partial sums in C).
 */
int sgemm_host(int M, int N, int K, float alpha,
               const float *A, int lda,
               const float *B, int ldb,
               float beta, float *C, int ldc,
               sgemm_stream_t stream);

/*
 * sgemm_3xtf32 -- the same GEMM on the tensor cores (tcgen05, TF32 inputs,
 * fp32 accumulation in tensor memory) by the 3xTF32 split: each operand is
 * x = hi + lo with hi = tf32(x), lo = tf32(x - hi), and A*B is taken as
 * A_hi*B_hi + A_hi*B_lo + A_lo*B_hi.  The result meets the same FP32
 * tolerance as sgemm() (about 3 * 2^-22 relative error per product, fp32
 * accumulation) but is not bitwise equal to it.  Arguments, ownership, stream
 * behaviour and errors as for sgemm().  Workspace: the hi and lo parts of A
 * (2 x M x roundup(K,4) floats) and of B transposed (2 x N x roundup(K,4)),
 * from the library's stream-ordered pool.  Non-finite inputs give NaN or Inf
 * results as IEEE arithmetic on the parts does; an input of magnitude near
 * FLT_MAX may overflow in its tf32 part.
 */
int sgemm_3xtf32(int M, int N, int K, float alpha,
                 const float *A, int lda,
                 const float *B, int ldb,
                 float beta, float *C, int ldc,
                 sgemm_stream_t stream);

/*
 * sgemm_host_3xtf32 -- sgemm_host() through the 3xTF32 tensor-core path: B is
 * split once on the device, each row block of A is split and multiplied as
 * in sgemm_3xtf32().  Same arguments and synchronisation as sgemm_host(); the
 * pipeline differs in two points (this path is bound by the host link, not
 * by its first multiply): equal row blocks of at least 1024 rows (at most 8),
 * and block 0's C_in is copied in front of its first chunk.  Same tolerance as
 * sgemm_3xtf32().
 */
int sgemm_host_3xtf32(int M, int N, int K, float alpha,
                      const float *A, int lda,
                      const float *B, int ldb,
                      float beta, float *C, int ldc,
                      sgemm_stream_t stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *sgemm_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int sgemm_version(void);

/* The cudaError_t value behind the most recent SGEMM_ERR_CUDA / SGEMM_ERR_ALLOC
 * on the calling thread (0 if none). */
int sgemm_last_cuda_error(void);

/*
 * sgemm_last_kernel -- the configuration of the last main kernel that a call
 * from the calling thread launched (any entry point), as static text that stays
 * valid for the life of the process: a kernel variant's name (as
 * sgemm_variant_name gives it; the batched, fused, tall-batch and
 * staged-epilogue kernels have their own), the direct small-problem kernel,
 * one of the two 3xTF32 kernels, or the scale-only kernel of alpha == 0 or
 * K == 0.  "" before the thread's first launch.  Set when the launch is
 * enqueued, not when it completes.  No GPU work.
 */
const char *sgemm_last_kernel(void);

/*
 * sgemm_device_status -- synchronises `stream`, then reads and clears the
 * library's device-side error word for the current device.  Returns SGEMM_OK,
 * or SGEMM_ERR_TIMEOUT if a kernel gave up a bounded wait (it then wrote no
 * result for the affected tiles), or SGEMM_ERR_BOUNDS (range-checked build
 * only, sgemm_debug_bounds_checks) if a kernel found an index out of range, or
 * SGEMM_ERR_CUDA if the synchronisation itself failed.
 */
int sgemm_device_status(sgemm_stream_t stream);

/*
 * sgemm_set_wait_timeout_ns -- limit (nanoseconds) for every in-kernel wait on
 * a shared-memory barrier, for launches made after the call.  Default 2e9.
 * A wait that exceeds it sets the device error word and the kernel returns.
 * Values below 1000 are rejected with SGEMM_ERR_INVALID_ARG.
 */
int sgemm_set_wait_timeout_ns(unsigned long long ns);

/*
 * sgemm_selftest_wait_timeout -- failure-detection self test.  Launches one
 * block whose thread waits on a shared-memory barrier that nothing ever
 * completes, with the given limit (nanoseconds, >= 1000, <= 1e10).  The wait
 * expires, the kernel records the expiry in the device error word and returns.
 * The call then behaves like sgemm_device_status(stream): it returns
 * SGEMM_ERR_TIMEOUT when the expiry was detected and reported (the expected
 * outcome), and the error word is left cleared.
 */
int sgemm_selftest_wait_timeout(unsigned long long ns, sgemm_stream_t stream);

/*
 * sgemm_debug_bounds_checks -- 1 when this library is the range-checked build
 * (compiled with -DSGEMM_DEBUG_BOUNDS: libsgemm_debug_bounds.so), 0 otherwise.
 * In that build every kernel checks the indices of its shared-memory,
 * global-memory, tensor-memory and TMA accesses against the ranges they must
 * lie in (the fragments of a slab inside its ring stage, the outputs of a tile
 * inside the tile, stream-K slots and counters inside their arrays, pre-pass
 * writes inside the row pitch, ...).  An index out of range is not used: the
 * access is skipped and sgemm_device_status() reports SGEMM_ERR_BOUNDS.  It is
 * the library's own stand-in for a memory checker, for tests; it runs slower
 * and is never the library the package loads by default.
 */
int sgemm_debug_bounds_checks(void);

/*
 * sgemm_debug_drop_release -- failure-detection test switch, off (0) by
 * default.  With 1, later plain sgemm() calls (not sgemm_ex, sgemm_host,
 * sgemm_noalloc or the 3xTF32 entry points) run a test build of the default
 * persistent kernel, also for problems small enough for the direct kernel.  In
 * it, consumer warp 0 of CTA 0 leaves out its release of the CTA's third
 * k-slab, so the wait for that stage to be freed expires after the limit of
 * sgemm_set_wait_timeout_ns (set a short one first: the call then takes about
 * two limits) while no copy into it is in flight.  The kernel's own abort path
 * runs: the expiry is recorded (sgemm_device_status returns SGEMM_ERR_TIMEOUT),
 * CTA 0 writes nothing more to C, the output tiles it was computing (whole, or
 * shared with other CTAs through stream-K pieces) stay unwritten, its copies
 * in flight land before it exits, and every other tile is written as usual.
 * CTA 0 must have at least five k-slabs of work for the expiry to happen.  No
 * fault, trap or hang is involved; the context stays usable.  0 restores
 * normal calls; anything but 0 or 1 gives SGEMM_ERR_INVALID_ARG.
 */
int sgemm_debug_drop_release(int on);

/*
 * Kernel timing for benchmarks.  sgemm_profile_enable(1) makes later sgemm()
 * calls record CUDA events on their stream around their main GEMM kernel and
 * around their packing kernels.  sgemm_profile_collect() synchronises those
 * events, writes the summed milliseconds and the number of launches of each
 * kind (any pointer may be NULL), and clears the record.  Disabled by default.
 */
int sgemm_profile_enable(int on);
int sgemm_profile_collect(double *main_ms, long long *main_launches,
                          double *pack_ms, long long *pack_launches);

/* Number of kernels this library has launched in this process. */
long long sgemm_kernel_launch_count(void);

/*
 * sgemm_config_string -- the kernel configuration sgemm() would pick for the
 * given shape (tile sizes, stages, micro-kernel, work split), as text that
 * stays valid until the calling thread's next call.  With a CUDA device
 * current, the choice is the one sgemm() makes on that device: the direct
 * small-problem kernel for problems of fewer 256x128 tile slabs than SMs, the
 * skinny-M kernel for at most 32 rows, the skinny-N kernel for at most 32
 * columns, else a tiled variant (the 128x128 tile when the default tile makes
 * fewer tiles than a quarter of the SMs; C whose rows are not all 16-byte
 * aligned, read with beta != 0, takes the same tile with its staged epilogue,
 * which the shape alone does not show); the text also says when the work
 * split leaves out the stream-K tail (whole tiles alone would leave under 1 %
 * of the SMs' slots idle).  Without a device: the tiled variant for the
 * shape.  No GPU work.
 */
const char *sgemm_config_string(int M, int N, int K);

/*
 * Kernel variants, for tile-configuration sweeps.  Every variant computes the
 * same result within the tolerance above; they differ in tile sizes, pipeline
 * depth and micro-kernel.  sgemm_variant_count() gives their number,
 * sgemm_variant_name(i) a static description ("" for an invalid index), and
 * sgemm_set_variant(i) forces variant i for later sgemm() calls in this
 * process, also on shapes that would otherwise take the direct small-problem
 * or skinny kernels (-1 restores the automatic choice; anything else out of
 * range gives SGEMM_ERR_INVALID_ARG).
 */
int sgemm_variant_count(void);
const char *sgemm_variant_name(int id);
int sgemm_set_variant(int id);

/*
 * Main kernel of the 3xTF32 entry points: -1 (the default) chooses per shape,
 * 0 forces the single-CTA kernel (128 x 256 tiles), 1 the CTA-pair kernel (each
 * 256 x 256 tile on a pair of SMs, a 2-CTA cluster sharing the MMA, tcgen05
 * cta_group::2).  The automatic choice compares the two kernels' waves over the
 * SMs and takes the pair on a tie (its main loop is faster).  Both meet the
 * same tolerance; results may differ in the last bits.  Applies to later calls
 * in this process; anything outside -1..1 gives SGEMM_ERR_INVALID_ARG.  The
 * pair kernel is launched as 2-CTA clusters of one CTA per SM: where the
 * device cannot hold them (a partitioned GPU), its launch fails with
 * SGEMM_ERR_CUDA and 0 selects the single-CTA kernel.
 */
int sgemm_set_3xtf32_kernel(int pair);

/*
 * sgemm_noalloc -- the same GEMM as sgemm(), for callers that cannot allocate
 * device memory.  The pages this library follows have no counterpart to it.
 *
 * Who needs it: code that runs where allocating is not allowed or not safe,
 * for instance inside a host framework that has already handed all device
 * memory to its own allocator, or on a latency-critical path where a
 * cudaMalloc (which can synchronise the device or fail under memory pressure)
 * must not happen.  sgemm() takes its workspace from a memory pool, which is
 * an allocation; this entry point never allocates: no cudaMalloc, cudaFree,
 * pool or library allocation.
 *
 * How: the workspace (the transposed copy of A, plus a re-pitched copy of B
 * when B's address or row pitch is not a multiple of 16 bytes) lives in one
 * fixed array in device memory of 8,388,608 floats (32 MiB), which every
 * device that loads this library keeps until the process exits.
 * A, B and C are the caller's device pointers, as for sgemm().
 *
 * Limit: K * roundup(M, 4), rounded up to a multiple of 64, plus
 * K * roundup(N, 4) when B needs the re-pitched copy, must not exceed that
 * number of floats; otherwise the call returns SGEMM_ERR_TOO_LARGE and does
 * nothing.  Problems with alpha == 0 or K == 0 need no scratch.
 *
 * Set-up: the first call on each device (made with that device current) looks
 * up the array's device address and configures the kernels; make that first
 * call before any stream capture.
 *
 * Sharing: every call on a device uses the same array, and it keeps whatever
 * the previous call left there; each call overwrites the part it reads before
 * reading it.  Calls whose work overlaps on the GPU (on different streams, or
 * from several host threads) race on the array: order them on one stream or
 * synchronise between them.  Results and errors are otherwise as for sgemm().
 */
int sgemm_noalloc(int M, int N, int K, float alpha,
                  const float *A, int lda,
                  const float *B, int ldb,
                  float beta, float *C, int ldc,
                  sgemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_FP32_GEMM_02_GB300_SGEMM_H */

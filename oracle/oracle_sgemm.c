/*
 * oracle_sgemm.c -- CPU oracle for the row-major FP32 GEMM  C = alpha*A*B + beta*C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (plain definition, no blocking, fusion or reordering):
 *
 *   C_out[i][j] = (float)( alpha * sum_{k=0..K-1} A[i][k]*B[k][j]  +  beta * C_in[i][j] )
 *
 * with every product and partial sum carried in IEEE double, k ascending, and one
 * final rounding to float.  alpha is applied once, after the sum, as in the naive
 * kernel of "How to implement matrix multiplication efficiently? An introduction
 * from a CUDA beginner's view" (makelele.cn repost of the Hands-on-GEMM article,
 * section "Naive GEMM and prerequisites": c = alpha*A*B + beta*C, the alpha
 * multiply placed after the k loop to save multiplies).  The row-major layout
 * (A is M rows by K columns, B is K by N, C is M by N) is the one that section
 * states.  Leading dimensions lda/ldb/ldc (elements between consecutive rows)
 * follow the BLAS convention.
 *
 * Readings taken where the pages are silent (also listed in the design notes):
 *  - beta == 0: C_in is not read, so NaN/Inf in C_in do not propagate.
 *  - alpha == 0: the product term is exactly zero and A, B are not read.
 *  - K == 0: the sum is empty (zero), so C_out = beta*C_in.
 *
 * Tolerance bound returned beside each element (the acceptance rule for the
 * GPU result; the exercise page "3.3 Shared memory and tiling - exercises",
 * exercise 2, asks for a tolerance rather than equality because summation order
 * changes the float rounding):
 *
 *   bound[i][j] = 1e-6 * K * |alpha| * sum_k |A[i][k]|*|B[k][j]|  +  1e-6 * |beta * C_in[i][j]|
 *
 * Build: plain C99, no vendor intrinsics, -O2 -ffp-contract=off (no fused
 * multiply-add contraction, no fast-math) so x86-64 and aarch64 give the same
 * bits.  Single-threaded; callers split rows across threads.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_ALLOC 2

/* Final combination of one element: one rounding to float after the double math. */
static float combine(double alpha, double sum, double beta, const float *c_in_elem,
                     double abs_sum, long long K, double *bound_elem)
{
    double prod = (alpha == 0.0) ? 0.0 : alpha * sum;
    double cterm = 0.0;
    if (beta != 0.0)
        cterm = beta * (double)(*c_in_elem);
    if (bound_elem) {
        double b = 1e-6 * (double)K * fabs(alpha) * abs_sum;
        if (beta != 0.0)
            b += 1e-6 * fabs(cterm);
        *bound_elem = b;
    }
    return (float)(prod + cterm);
}

/*
 * Full rows of C.  For each requested row index rows[r] (0 <= rows[r] < M) this
 * writes out[r*N + j] and, if bound != NULL, bound[r*N + j] for 0 <= j < N.
 * Loop order i, k, j with a double accumulator row (the i-k-j form keeps B
 * rows contiguous; the k order of every individual sum is still ascending).
 */
int oracle_sgemm_rows(long long M, long long N, long long K, float alpha,
                      const float *A, long long lda, const float *B, long long ldb,
                      float beta, const float *C_in, long long ldc,
                      const long long *rows, long long nrows,
                      float *out, double *bound)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || !rows || (!out && nrows * N > 0))
        return ORACLE_ERR_ARG;
    if (beta != 0.0f && !C_in && nrows * N > 0)
        return ORACLE_ERR_ARG;
    if (N == 0 || nrows == 0)
        return ORACLE_OK;

    double *acc = (double *)malloc(sizeof(double) * (size_t)N);
    double *abs_acc = (double *)malloc(sizeof(double) * (size_t)N);
    if (!acc || !abs_acc) {
        free(acc);
        free(abs_acc);
        return ORACLE_ERR_ALLOC;
    }

    const int use_products = (alpha != 0.0f);
    for (long long r = 0; r < nrows; ++r) {
        long long i = rows[r];
        if (i < 0 || i >= M) {
            free(acc);
            free(abs_acc);
            return ORACLE_ERR_ARG;
        }
        memset(acc, 0, sizeof(double) * (size_t)N);
        memset(abs_acc, 0, sizeof(double) * (size_t)N);
        if (use_products) {
            for (long long k = 0; k < K; ++k) {
                double a = (double)A[i * lda + k];
                double abs_a = fabs(a);
                const float *brow = B + k * ldb;
                for (long long j = 0; j < N; ++j) {
                    double b = (double)brow[j];
                    acc[j] += a * b;
                    abs_acc[j] += abs_a * fabs(b);
                }
            }
        }
        for (long long j = 0; j < N; ++j) {
            const float *c_elem = (beta != 0.0f) ? &C_in[i * ldc + j] : NULL;
            out[r * N + j] = combine((double)alpha, acc[j], (double)beta, c_elem,
                                     abs_acc[j], K, bound ? &bound[r * N + j] : NULL);
        }
    }
    free(acc);
    free(abs_acc);
    return ORACLE_OK;
}

/*
 * Selected full columns of C, for rows row_begin <= i < row_end.
 * Writes out[(i-row_begin)*ncols + c] for the column index cols[c].
 * The requested columns of B are first gathered into a K x ncols copy (a plain
 * copy, no arithmetic) so the k loop walks contiguous memory; every sum is
 * still taken in ascending k.
 */
int oracle_sgemm_cols(long long M, long long N, long long K, float alpha,
                      const float *A, long long lda, const float *B, long long ldb,
                      float beta, const float *C_in, long long ldc,
                      const long long *cols, long long ncols,
                      long long row_begin, long long row_end,
                      float *out, double *bound)
{
    if (M < 0 || N < 0 || K < 0 || ncols < 0 || !cols)
        return ORACLE_ERR_ARG;
    if (row_begin < 0 || row_end > M || row_begin > row_end)
        return ORACLE_ERR_ARG;
    long long nr = row_end - row_begin;
    if (nr == 0 || ncols == 0)
        return ORACLE_OK;
    if (!out || (beta != 0.0f && !C_in))
        return ORACLE_ERR_ARG;
    for (long long c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N)
            return ORACLE_ERR_ARG;

    const int use_products = (alpha != 0.0f);
    float *bcols = NULL;
    if (use_products && K > 0) {
        bcols = (float *)malloc(sizeof(float) * (size_t)(K * ncols));
        if (!bcols)
            return ORACLE_ERR_ALLOC;
        for (long long k = 0; k < K; ++k)
            for (long long c = 0; c < ncols; ++c)
                bcols[k * ncols + c] = B[k * ldb + cols[c]];
    }
    double *acc = (double *)malloc(sizeof(double) * (size_t)ncols);
    double *abs_acc = (double *)malloc(sizeof(double) * (size_t)ncols);
    if (!acc || !abs_acc) {
        free(bcols);
        free(acc);
        free(abs_acc);
        return ORACLE_ERR_ALLOC;
    }

    for (long long i = row_begin; i < row_end; ++i) {
        memset(acc, 0, sizeof(double) * (size_t)ncols);
        memset(abs_acc, 0, sizeof(double) * (size_t)ncols);
        if (use_products) {
            for (long long k = 0; k < K; ++k) {
                double a = (double)A[i * lda + k];
                double abs_a = fabs(a);
                const float *brow = bcols + k * ncols;
                for (long long c = 0; c < ncols; ++c) {
                    double b = (double)brow[c];
                    acc[c] += a * b;
                    abs_acc[c] += abs_a * fabs(b);
                }
            }
        }
        long long o = (i - row_begin) * ncols;
        for (long long c = 0; c < ncols; ++c) {
            const float *c_elem = (beta != 0.0f) ? &C_in[i * ldc + cols[c]] : NULL;
            out[o + c] = combine((double)alpha, acc[c], (double)beta, c_elem,
                                 abs_acc[c], K, bound ? &bound[o + c] : NULL);
        }
    }
    free(bcols);
    free(acc);
    free(abs_acc);
    return ORACLE_OK;
}

/*
 * Fused epilogue: the GEMM of one batch followed by a bias and an activation,
 * the layer form in which neural networks use matrix multiplication (the
 * article "How to implement matrix multiplication efficiently? An introduction
 * from a CUDA beginner's view" motivates GEMM optimisation by neural-network
 * workloads and names operator fusion with the GEMM as the next step; it fixes
 * no bias or activation, so the forms below are this oracle's reading):
 *
 *   Z[i][j]     = alpha * sum_k A[i][k]*B[k][j]  +  beta * C_in[i][j]  +  bias[j]
 *   C_out[i][j] = (float) act(Z[i][j])
 *
 * in double with one final rounding; bias == NULL means no bias (the bias is
 * per output column, broadcast over the rows); act 0 = identity, 1 = ReLU
 * max(Z, 0), 2 = GELU in its erf form Z * Phi(Z) = 0.5 * Z * (1 + erf(Z / sqrt 2)).
 * A batched GEMM is one call per batch on that batch's own matrices.
 *
 * Bound: the plain bound plus 1e-6 * |bias[j]| for Z; identity and ReLU
 * (1-Lipschitz) keep it; GELU takes 1.129 * bound_Z + 1e-6 * |Z|, where 1.129
 * is the largest slope of Z * Phi(Z) (at Z = sqrt 2: Phi(sqrt 2) + sqrt 2 *
 * phi(sqrt 2)) and the second term covers a single-precision erf.
 */
#define ORACLE_ACT_NONE 0
#define ORACLE_ACT_RELU 1
#define ORACLE_ACT_GELU 2

static double activation(int act, double z)
{
    if (act == ORACLE_ACT_RELU)
        return z > 0.0 ? z : 0.0;
    if (act == ORACLE_ACT_GELU)
        return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
    return z;
}

int oracle_sgemm_ex_rows(long long M, long long N, long long K, float alpha,
                         const float *A, long long lda, const float *B, long long ldb,
                         float beta, const float *C_in, long long ldc,
                         const float *bias, int act,
                         const long long *rows, long long nrows,
                         float *out, double *bound)
{
    if (act < ORACLE_ACT_NONE || act > ORACLE_ACT_GELU)
        return ORACLE_ERR_ARG;
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || !rows || (!out && nrows * N > 0))
        return ORACLE_ERR_ARG;
    if (beta != 0.0f && !C_in && nrows * N > 0)
        return ORACLE_ERR_ARG;
    if (N == 0 || nrows == 0)
        return ORACLE_OK;

    double *acc = (double *)malloc(sizeof(double) * (size_t)N);
    double *abs_acc = (double *)malloc(sizeof(double) * (size_t)N);
    if (!acc || !abs_acc) {
        free(acc);
        free(abs_acc);
        return ORACLE_ERR_ALLOC;
    }
    for (long long r = 0; r < nrows; ++r) {
        long long i = rows[r];
        if (i < 0 || i >= M) {
            free(acc);
            free(abs_acc);
            return ORACLE_ERR_ARG;
        }
        memset(acc, 0, sizeof(double) * (size_t)N);
        memset(abs_acc, 0, sizeof(double) * (size_t)N);
        if (alpha != 0.0f) {
            for (long long k = 0; k < K; ++k) {
                double a = (double)A[i * lda + k];
                const float *brow = B + k * ldb;
                for (long long j = 0; j < N; ++j) {
                    acc[j] += a * (double)brow[j];
                    abs_acc[j] += fabs(a) * fabs((double)brow[j]);
                }
            }
        }
        for (long long j = 0; j < N; ++j) {
            double z = (alpha == 0.0f) ? 0.0 : (double)alpha * acc[j];
            double bz = 1e-6 * (double)K * fabs((double)alpha) * abs_acc[j];
            if (beta != 0.0f) {
                double cterm = (double)beta * (double)C_in[i * ldc + j];
                z += cterm;
                bz += 1e-6 * fabs(cterm);
            }
            if (bias) {
                z += (double)bias[j];
                bz += 1e-6 * fabs((double)bias[j]);
            }
            out[r * N + j] = (float)activation(act, z);
            if (bound)
                bound[r * N + j] = (act == ORACLE_ACT_GELU) ? 1.129 * bz + 1e-6 * fabs(z) : bz;
        }
    }
    free(acc);
    free(abs_acc);
    return ORACLE_OK;
}

/* Version tag so the loader can refuse a stale build. */
int oracle_abi_version(void) { return 2; }

/*
 * ref_gemm.c -- CPU oracle for row-major single-precision matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  The product
 * path (the CUDA library) never calls it and shares no code with it.
 *
 * Definition followed ("Lecture 12: final project", runguoli.com ECE408
 * notes l12, section 3 "CPU golden reference", goldenReference):
 *
 *     C[i][j] = (float)( sum_{k = 0 .. K-1} (double)A[i*K + k] * (double)B[k*N + j] )
 *
 * with the sum taken in double, k ascending, starting from 0.0, and one final
 * round-to-nearest-even conversion to float.  Indexing is 64-bit.  A is M x K,
 * B is K x N and C is M x N, all packed row-major.  K == 0 gives C == 0.
 *
 * The loop is the textbook i-j-k triple loop.  The only concurrency is an
 * OpenMP split of the independent output rows; every element is still summed
 * by one thread in ascending k, so the thread count cannot change a bit.
 *
 * A product of two floats has at most 48 significant bits and is exact in
 * double, so fused or unfused multiply-add in the compiled loop gives the same
 * value; no -ffast-math is used.
 */
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static float ref_dot(const float* A, const float* B, int64_t N, int64_t K,
                     int64_t i, int64_t j)
{
    double sum = 0.0;
    for (int64_t k = 0; k < K; ++k)
        sum += (double)A[i * K + k] * (double)B[k * N + j];
    return (float)sum;
}

/* Full product.  nthreads <= 0 uses the OpenMP default. */
void ref_gemm(const float* A, const float* B, float* C,
              int64_t M, int64_t N, int64_t K, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            C[i * N + j] = ref_dot(A, B, N, K, i, j);
    (void)nthreads;
}

/* Selected entries: out[t] = C[rows[t]][cols[t]] by the same definition. */
void ref_gemm_entries(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                      const int64_t* rows, const int64_t* cols, int64_t count,
                      float* out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t t = 0; t < count; ++t)
        out[t] = ref_dot(A, B, N, K, rows[t], cols[t]);
    (void)M;
    (void)nthreads;
}

/* Rows [row0, row0 + nrows) of C into out (nrows x N, packed). */
void ref_gemm_rows(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                   int64_t row0, int64_t nrows, float* out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t j = 0; j < N; ++j)
            out[r * N + j] = ref_dot(A, B, N, K, row0 + r, j);
    (void)M;
    (void)nthreads;
}

/*
 * General form, row-major with leading dimensions and transposes:
 *
 *     C[i][j] = (float)( alpha * S + beta * (double)C[i][j] )     (beta != 0)
 *     C[i][j] = (float)( alpha * S )                              (beta == 0)
 *     S       = sum_{k ascending} (double)opA(i, k) * (double)opB(k, j)
 *
 * opA(i, k) = A[i*lda + k] (transa == 0) or A[k*lda + i] (transa == 1);
 * opB(k, j) = B[k*ldb + j] (transb == 0) or B[j*ldb + k] (transb == 1);
 * C[i][j] lives at C[i*ldc + j].  With beta == 0 the old C is never read, so
 * a NaN there cannot leak into the result (the usual BLAS convention).
 * alpha * S and beta * C are formed and added in double; one final rounding.
 */
void ref_gemm_ex(int transa, int transb, int64_t M, int64_t N, int64_t K, double alpha,
                 const float* A, int64_t lda, const float* B, int64_t ldb, double beta,
                 float* C, int64_t ldc, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = transa ? (double)A[k * lda + i] : (double)A[i * lda + k];
                const double b = transb ? (double)B[j * ldb + k] : (double)B[k * ldb + j];
                sum += a * b;
            }
            double r = alpha * sum;
            if (beta != 0.0) r += beta * (double)C[i * ldc + j];
            C[i * ldc + j] = (float)r;
        }
    (void)nthreads;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int ref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

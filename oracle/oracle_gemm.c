/*
 * oracle_gemm.c -- the CPU oracle for C = A.B with f16 operands.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load this
 * library.  It shares no code, header, table or constant with the CUDA
 * library and includes no CUDA header.
 *
 * What it computes is the plain definition of the dot that the pages tile:
 *
 *   C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * ("The PTSS Cliff: A Kernel That Won't Build", section "The Arithmetic of
 * 'Fully Unrolled K'", which writes one output cell as the K-long sum of
 * A[i][k]*B[k][j]; "Intel XPU Backend for Triton", section "Use Tensor
 * Descriptors to load tl.dot arguments and save results", whose loop adds
 * tl.dot of successive K blocks into one accumulator).  The pages accumulate
 * in f32; the oracle accumulates in fp64 so that it is far more accurate than
 * the kernel it judges.  Every f16 input decodes exactly to a double, every
 * product of two f16 values is exact in a double (11 + 11 significant bits),
 * so the only rounding is in the additions, which run in ascending k for
 * every cell.  The result is therefore the same on any IEEE-754 host,
 * whether or not the compiler fuses the multiply into the add.
 *
 * Operands are row-major with strides in elements, the last stride being 1
 * ("Intel XPU Backend for Triton", section "Set last stride to 1").
 * The loops are i, then k, then j: each cell still sums in ascending k, and
 * the inner loop walks a row of B contiguously.  OpenMP splits the rows of C
 * across threads; no thread touches another's rows, so the thread count never
 * changes a result.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   exponent 0      : subnormal, value = fraction * 2^-24
 *   exponent 1..30  : normal,    value = (1024 + fraction) * 2^(exponent - 25)
 *   exponent 31     : infinity (fraction 0) or NaN
 * No flush of subnormals: they decode exactly. */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac | 0x400), expo - 25);
    return sign ? -v : v;
}

/* Decode table for all 65536 binary16 patterns, filled from the function
 * above on first use (a lookup is much faster than the branches). */
static double g_f16_table[65536];
static int g_f16_table_ready = 0;

static void ensure_table(void)
{
    if (g_f16_table_ready)
        return;
#pragma omp critical(oracle_table)
    {
        if (!g_f16_table_ready) {
            for (uint32_t h = 0; h < 65536u; ++h)
                g_f16_table[h] = oracle_f16_to_f64((uint16_t)h);
            g_f16_table_ready = 1;
        }
    }
}

static int pick_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Full product.  A: M x K (row stride lda), B: K x N (row stride ldb),
 * C: M x N doubles (row stride ldc).  Returns 0, or -1 on a bad argument
 * or an allocation failure.  K == 0 gives the empty sum, 0. */
int oracle_gemm_f16_f64(const uint16_t *A, const uint16_t *B, double *C,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc, int nthreads)
{
    if (M < 0 || N < 0 || K < 0)
        return -1;
    if (M == 0 || N == 0)
        return 0;
    if (!C || ldc < N || (K > 0 && (!A || !B || lda < K || ldb < N)))
        return -1;
    ensure_table();
    int bad = 0;
#pragma omp parallel num_threads(pick_threads(nthreads))
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t i = 0; i < M; ++i) {
            if (!acc)
                continue;
            for (int64_t j = 0; j < N; ++j)
                acc[j] = 0.0;
            const uint16_t *arow = A + i * lda;
            for (int64_t k = 0; k < K; ++k) {
                const double a = g_f16_table[arow[k]];
                const uint16_t *brow = B + k * ldb;
                for (int64_t j = 0; j < N; ++j)
                    acc[j] += a * g_f16_table[brow[j]];
            }
            double *crow = C + i * ldc;
            for (int64_t j = 0; j < N; ++j)
                crow[j] = acc[j];
        }
        free(acc);
    }
    return bad ? -1 : 0;
}

/* Selected cells only: out[t] = C[rows[t]][cols[t]] for t < count, each the
 * same ascending-k sum as above.  Used where the full product would take the
 * host too long. */
int oracle_gemm_f16_f64_cells(const uint16_t *A, const uint16_t *B,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb,
                              const int64_t *rows, const int64_t *cols,
                              int64_t count, double *out, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || count < 0)
        return -1;
    if (count == 0)
        return 0;
    if (!rows || !cols || !out || (K > 0 && (!A || !B || lda < K || ldb < N)))
        return -1;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N)
            return -1;
    ensure_table();
#pragma omp parallel for schedule(static) num_threads(pick_threads(nthreads))
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t *arow = A + rows[t] * lda;
        const uint16_t *bcol = B + cols[t];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += g_f16_table[arow[k]] * g_f16_table[bcol[k * ldb]];
        out[t] = acc;
    }
    return 0;
}

/* The thread count the full product would use for a given request. */
int oracle_threads(int nthreads)
{
    return pick_threads(nthreads);
}

/*
 * Plain CPU oracle for the GEMM and the transpose -- TEST INFRASTRUCTURE ONLY.
 *
 * GEMM: the definition C[i][j] = sum_k A[i][k] * B[k][j] with A (M x K) and
 * B (K x N) row-major, as the benchmark of Lei Mao, "CUDA Thread Block
 * Swizzle" (section "CUDA Thread Block Swizzle Benchmark", the GEMM kernel and
 * its torch.matmul check) states the problem.  Everything is carried in IEEE
 * double.  The caller passes A and B already widened to double from the very
 * half-precision values the GPU reads, so every product of two fp16 (or bf16)
 * values is exact here and only the K-term sum rounds (at 2^-53 relative).
 * For each output the terms are added in k order 0, 1, ..., K-1; the loops
 * visit k outside j only so that B is read row by row -- the summation order
 * of every C[i][j] is unchanged.  Rows are split across OpenMP threads.
 *
 * Transpose: out[j][i] = in[i][j] for an M x N matrix of 32-bit words, as the
 * "Matrix Transpose" case study of WHC, "CUDA Swizzle & bank conflict" defines
 * it (the N x M result is row-major).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* C rows [row_begin, row_end) of A*B; C is (row_end-row_begin) x N. */
void oracle_gemm_rows_f64(const double *A, const double *B, double *C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t row_begin, int64_t row_end) {
    (void)M;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = row_begin; i < row_end; ++i) {
        double *c = C + (i - row_begin) * N;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * K + k];
            const double *b = B + k * N;
            for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
        }
    }
}

/* Single entries C[ii[s]][jj[s]] for s = 0 .. count-1 (sampled parity). */
void oracle_gemm_entries_f64(const double *A, const double *B,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t *ii, const int64_t *jj,
                             int64_t count, double *out) {
    (void)M;
    int64_t s;
#pragma omp parallel for schedule(static)
    for (s = 0; s < count; ++s) {
        const int64_t i = ii[s], j = jj[s];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += A[i * K + k] * B[k * N + j];
        out[s] = acc;
    }
}

/* out (N x M) = transpose of in (M x N); 32-bit words copied bit for bit. */
void oracle_transpose_u32(const uint32_t *in, uint32_t *out,
                          int64_t M, int64_t N) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) out[j * M + i] = in[i * N + j];
}

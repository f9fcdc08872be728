/*
 * Test infrastructure -- the CPU oracle for the MoE grouped GEMMs.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * use this file.  It shares no code with the CUDA path and is deliberately
 * plain: one loop nest per operation, FP64 accumulation in the order the
 * definition states, no blocking or reordering.
 *
 * Operations (RapidGEMM README, "Kernels"):
 *
 *   M-grouped GEMM (Mgemm; forward and input gradient).  x is [M,K], w is
 *   [E,N,K], offsets is the cumulative row-offset vector with a leading zero.
 *   Expert e owns rows r in [offsets[e], offsets[e+1]) and
 *       y[r,n] = sum_k x[r,k] * w[e,n,k]          (transpose_B == 0)
 *       y[r,n] = sum_k x[r,k] * w[e,k,n]          (transpose_B != 0, w [E,K,N])
 *
 *   K-grouped FP32 weight gradient (Kgemm).  grad is [M,N], X is [M,K]:
 *       dW[e,n,k] = sum_{r in group e} grad[r,n] * X[r,k]
 *   An expert with no rows has dW[e] = 0.
 *
 *   Nested grouped GEMM (CUTLASS discussion #1452: each subproblem of the
 *   grouped GEMM is itself a grouped GEMM, e.g. an A matrix [M, 3K] grouped
 *   along its columns for the outer problem and along its rows for the inner
 *   one).  x is [M, O*K], w is [O, L, N, K] (or [O, L, K, N]), offsets [L+1]
 *   splits the rows into inner groups shared by every outer group o:
 *       y[r, o*N + n] = sum_k x[r, o*K + k] * w[o, l, n, k]   (r in group l)
 *
 * Inputs are bf16 bit patterns; each value is widened exactly to double.
 * Products of two bf16 values are exact in double, so the result depends only
 * on the summation order, which is ascending k (Mgemm) or ascending r (Kgemm).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no -ffast-math).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* 0 if offsets is a valid cumulative vector for M rows, else -1. */
static int check_offsets(const int32_t *offsets, int E, int64_t M) {
    if (E < 1 || offsets[0] != 0) return -1;
    for (int e = 0; e < E; ++e)
        if (offsets[e + 1] < offsets[e]) return -1;
    if ((int64_t)offsets[E] > M) return -1;
    return 0;
}

/* Expert that owns row r, or -1 if r >= offsets[E].  Linear scan: the first
 * e with offsets[e] <= r < offsets[e+1]. */
static int expert_of_row(const int32_t *offsets, int E, int64_t r) {
    for (int e = 0; e < E; ++e)
        if ((int64_t)offsets[e] <= r && r < (int64_t)offsets[e + 1]) return e;
    return -1;
}

/*
 * Mgemm on a list of rows.  rows[i] must lie in [0, offsets[E]); out is
 * [nrows, N] doubles: out[i,n] = y[rows[i], n].  Returns 0, or -1 on bad
 * arguments.
 */
int oracle_mgemm_rows(const uint16_t *x, const uint16_t *w, const int32_t *offsets,
                      int E, int64_t M, int N, int K, int transpose_B,
                      const int64_t *rows, int64_t nrows, double *out) {
    if (N < 1 || K < 1 || check_offsets(offsets, E, M) != 0) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= (int64_t)offsets[E]) return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t r = rows[i];
        const int e = expert_of_row(offsets, E, r);
        const uint16_t *xr = x + r * (int64_t)K;
        const uint16_t *we = w + (int64_t)e * N * K;
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            if (!transpose_B) {
                const uint16_t *wn = we + (int64_t)n * K; /* w[e,n,:] */
                for (int k = 0; k < K; ++k)
                    acc += bf16_to_double(xr[k]) * bf16_to_double(wn[k]);
            } else {
                for (int k = 0; k < K; ++k) /* w[e,k,n] */
                    acc += bf16_to_double(xr[k]) * bf16_to_double(we[(int64_t)k * N + n]);
            }
            out[i * (int64_t)N + n] = acc;
        }
    }
    return 0;
}

/*
 * Nested grouped GEMM on a list of rows.  out is [nrows, O*N] doubles:
 * out[i, o*N + n] = y[rows[i], o*N + n].  Returns 0, or -1 on bad arguments.
 */
int oracle_mgemm_nested_rows(const uint16_t *x, const uint16_t *w, const int32_t *offsets,
                             int O, int L, int64_t M, int N, int K, int transpose_B,
                             const int64_t *rows, int64_t nrows, double *out) {
    if (O < 1 || N < 1 || K < 1 || check_offsets(offsets, L, M) != 0) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= (int64_t)offsets[L]) return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t r = rows[i];
        const int l = expert_of_row(offsets, L, r);
        for (int o = 0; o < O; ++o) {
            const uint16_t *xr = x + r * (int64_t)O * K + (int64_t)o * K; /* x[r, o*K + :] */
            const uint16_t *wg = w + ((int64_t)o * L + l) * N * K;        /* w[o, l] */
            for (int n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) {
                    const uint16_t b = transpose_B ? wg[(int64_t)k * N + n] : wg[(int64_t)n * K + k];
                    acc += bf16_to_double(xr[k]) * bf16_to_double(b);
                }
                out[i * (int64_t)O * N + (int64_t)o * N + n] = acc;
            }
        }
    }
    return 0;
}

/*
 * Kgemm on a list of (expert, n) pairs.  out is [nsel, K] doubles:
 * out[i,k] = dW[sel_e[i], sel_n[i], k].  Returns 0, or -1 on bad arguments.
 */
int oracle_kgemm_rows(const uint16_t *grad, const uint16_t *X, const int32_t *offsets,
                      int E, int64_t M, int N, int K,
                      const int32_t *sel_e, const int32_t *sel_n, int64_t nsel, double *out) {
    if (N < 1 || K < 1 || check_offsets(offsets, E, M) != 0) return -1;
    for (int64_t i = 0; i < nsel; ++i)
        if (sel_e[i] < 0 || sel_e[i] >= E || sel_n[i] < 0 || sel_n[i] >= N) return -1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nsel; ++i) {
        const int e = sel_e[i];
        const int n = sel_n[i];
        double *o = out + i * (int64_t)K;
        for (int k = 0; k < K; ++k) o[k] = 0.0;
        /* ascending r: o[k] accumulates grad[r,n] * X[r,k] row by row */
        for (int64_t r = offsets[e]; r < (int64_t)offsets[e + 1]; ++r) {
            const double g = bf16_to_double(grad[r * (int64_t)N + n]);
            const uint16_t *xr = X + r * (int64_t)K;
            for (int k = 0; k < K; ++k) o[k] += g * bf16_to_double(xr[k]);
        }
    }
    return 0;
}

/* Number of OpenMP threads a parallel region uses (1 without OpenMP). */
int oracle_num_threads(void) {
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

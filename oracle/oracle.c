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
 *   MXFP8 M-grouped GEMM (the MXFP8 grouped GEMM of the torchao MoE-training
 *   PR and the FP8 block-scaling thread of the DeepGEMM issue; element and
 *   scale encodings after the OCP Microscaling (MX) formats: FP8 E4M3
 *   elements, one E8M0 power-of-two scale per 32 consecutive elements along
 *   the contraction).  xq [M,K] and wq [E,N,K] (or [E,K,N]) are E4M3 codes,
 *   sx [M,K/32] and sw [E,N,K/32] E8M0 codes:
 *       y[r,n] = sum_k (xq[r,k] * 2^(sx[r,k/32]-127)) * (wq[e,n,k] * 2^(sw[e,n,k/32]-127))
 *
 *   MXFP8 K-grouped weight gradient (the wgrad of the same MXFP8 MoE
 *   training: operands quantized along the contraction, which runs over each
 *   expert's rows, so every expert's row range is a whole number of 32-row
 *   scale blocks).  gq [M,N], xq [M,K] E4M3 codes, sg [N,M/32] and
 *   sx [K,M/32] E8M0 codes (one scale per column and 32-row block):
 *       dW[e,n,k] = sum_{r in group e} (gq[r,n] * 2^(sg[n,r/32]-127)) * (xq[r,k] * 2^(sx[k,r/32]-127))
 *
 * Inputs are bf16 bit patterns (E4M3 / E8M0 codes for the MXFP8 GEMMs); each value is widened exactly to double.
 * Products of two bf16 values are exact in double, so the result depends only
 * on the summation order, which is ascending k (Mgemm) or ascending r (Kgemm).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no -ffast-math).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP8 E4M3 (OCP): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
 * 0 is subnormal (m * 2^-9); S.1111.111 is NaN; there is no infinity. */
static double e4m3_to_double(uint8_t b) {
    const int e = (b >> 3) & 0xF, m = b & 0x7;
    if (e == 0xF && m == 0x7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (b & 0x80) ? -v : v;
}

/* E8M0 (OCP MX scale): 2^(s - 127); 0xFF is NaN. */
static double e8m0_to_double(uint8_t s) {
    return s == 0xFF ? NAN : ldexp(1.0, (int)s - 127);
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
 * MXFP8 Mgemm on a list of rows (K a multiple of 32).  out is [nrows, N]
 * doubles.  Each operand element is decoded and multiplied by its block's
 * scale (exact in double), then the products are summed in ascending k.
 */
int oracle_mgemm_mx_rows(const uint8_t *xq, const uint8_t *sx, const uint8_t *wq, const uint8_t *sw,
                         const int32_t *offsets, int E, int64_t M, int N, int K, int transpose_B,
                         const int64_t *rows, int64_t nrows, double *out) {
    if (N < 1 || K < 32 || K % 32 != 0 || check_offsets(offsets, E, M) != 0) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= (int64_t)offsets[E]) return -1;
    const int KS = K / 32;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t r = rows[i];
        const int e = expert_of_row(offsets, E, r);
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                const double a = e4m3_to_double(xq[r * (int64_t)K + k]) *
                                 e8m0_to_double(sx[r * (int64_t)KS + k / 32]);
                const uint8_t bq = transpose_B ? wq[((int64_t)e * K + k) * N + n]   /* w[e,k,n] */
                                               : wq[((int64_t)e * N + n) * K + k];  /* w[e,n,k] */
                const double b = e4m3_to_double(bq) * e8m0_to_double(sw[((int64_t)e * N + n) * KS + k / 32]);
                acc += a * b;
            }
            out[i * (int64_t)N + n] = acc;
        }
    }
    return 0;
}

/*
 * Blocked scale layout for a grouped operand (the scale-to-blocked-format
 * conversion of the torchao MoE-training PR, "128x4" blocks): the rows of
 * src [R, KS] (E8M0 codes, KS scales per row) are grouped by offsets [G+1];
 * each group is cut into blocks of 128 rows starting at its first row, so no
 * block mixes two groups, and the blocks of all groups are numbered in
 * order.  Block b, column chunk c (scale columns 4c..4c+3) occupies bytes
 * (b * ceil(KS/4) + c) * 512 .. +511 of dst, where row i (0..127) of the
 * block and column j (0..3) of the chunk sit at byte 16*(i%32) + 4*(i/32) + j.
 * Positions past a group's last row or past column KS-1 hold 0x7F (scale
 * 1.0).  Bytes of dst past the last block are not written.  dst_bytes must
 * cover every block; returns the number of blocks, or -1.
 */
int64_t oracle_mx_blocked(const uint8_t *src, int64_t R, int KS, const int32_t *offsets, int G,
                          uint8_t *dst, int64_t dst_bytes) {
    if (KS < 1 || check_offsets(offsets, G, R) != 0) return -1;
    const int nc = (KS + 3) / 4;
    int64_t b = 0;
    for (int g = 0; g < G; ++g) {
        const int64_t r0 = offsets[g], r1 = offsets[g + 1];
        for (int64_t base = r0; base < r1; base += 128, ++b) {
            if ((b + 1) * nc * 512 > dst_bytes) return -1;
            for (int c = 0; c < nc; ++c) {
                uint8_t *blk = dst + (b * nc + c) * 512;
                for (int i = 0; i < 128; ++i)
                    for (int j = 0; j < 4; ++j) {
                        const int64_t r = base + i;
                        const int col = 4 * c + j;
                        blk[16 * (i % 32) + 4 * (i / 32) + j] =
                            (r < r1 && col < KS) ? src[r * KS + col] : (uint8_t)0x7F;
                    }
            }
        }
    }
    return b;
}

/*
 * MXFP8 Kgemm on a list of (expert, n) pairs: out[i, k] = dW[sel_e[i],
 * sel_n[i], k].  Every offset must be a multiple of 32.  Returns 0 or -1.
 */
int oracle_kgemm_mx_rows(const uint8_t *gq, const uint8_t *sg, const uint8_t *xq, const uint8_t *sx,
                         const int32_t *offsets, int E, int64_t M, int N, int K,
                         const int32_t *sel_e, const int32_t *sel_n, int64_t nsel, double *out) {
    if (N < 1 || K < 1 || M % 32 != 0 || check_offsets(offsets, E, M) != 0) return -1;
    for (int e = 0; e <= E; ++e)
        if (offsets[e] % 32 != 0) return -1;
    for (int64_t i = 0; i < nsel; ++i)
        if (sel_e[i] < 0 || sel_e[i] >= E || sel_n[i] < 0 || sel_n[i] >= N) return -1;
    const int64_t MS = M / 32;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nsel; ++i) {
        const int e = sel_e[i];
        const int n = sel_n[i];
        double *o = out + i * (int64_t)K;
        for (int k = 0; k < K; ++k) o[k] = 0.0;
        for (int64_t r = offsets[e]; r < (int64_t)offsets[e + 1]; ++r) {
            const double g = e4m3_to_double(gq[r * (int64_t)N + n]) * e8m0_to_double(sg[(int64_t)n * MS + r / 32]);
            for (int k = 0; k < K; ++k)
                o[k] += g * (e4m3_to_double(xq[r * (int64_t)K + k]) * e8m0_to_double(sx[(int64_t)k * MS + r / 32]));
        }
    }
    return 0;
}

/*
 * Blocked scale layout for groups along the contraction (the torchao PR's
 * conversion "for groups along K"): src [R, KS] holds, for each of R rows
 * (an operand's columns), KS scales along the contraction; offsets [G+1]
 * are contraction indices (multiples of 32, offsets[G] <= 32*KS), so group g
 * owns scale columns offsets[g]/32 .. offsets[g+1]/32 - 1.  Each group's
 * scale columns are cut into chunks of 4 from its first column; the chunks
 * of all groups are numbered in order (NQ in total).  Row block rb (rows
 * 128rb ..), chunk q is the 512 bytes at (rb * NQ + q) * 512, with row i
 * and column j of the chunk at byte 16*(i%32) + 4*(i/32) + j; positions past
 * row R-1 or past the group's last scale column hold 0x7F.  Returns NQ or -1.
 */
int64_t oracle_mx_blocked_k(const uint8_t *src, int64_t R, int KS, const int32_t *offsets, int G,
                            uint8_t *dst, int64_t dst_bytes) {
    if (R < 1 || KS < 1 || check_offsets(offsets, G, (int64_t)KS * 32) != 0) return -1;
    for (int g = 0; g <= G; ++g)
        if (offsets[g] % 32 != 0) return -1;
    int64_t NQ = 0;
    for (int g = 0; g < G; ++g) NQ += (offsets[g + 1] - offsets[g] + 127) / 128;
    const int64_t NRB = (R + 127) / 128;
    if (NRB * NQ * 512 > dst_bytes) return -1;
    int64_t q = 0;
    for (int g = 0; g < G; ++g) {
        const int c0 = offsets[g] / 32, c1 = offsets[g + 1] / 32;
        for (int cb = c0; cb < c1; cb += 4, ++q)
            for (int64_t rb = 0; rb < NRB; ++rb) {
                uint8_t *blk = dst + (rb * NQ + q) * 512;
                for (int i = 0; i < 128; ++i)
                    for (int j = 0; j < 4; ++j) {
                        const int64_t r = 128 * rb + i;
                        const int col = cb + j;
                        blk[16 * (i % 32) + 4 * (i / 32) + j] =
                            (r < R && col < c1) ? src[r * KS + col] : (uint8_t)0x7F;
                    }
            }
    }
    return NQ;
}

/* Decoded values of the 256 E4M3 codes and of the 256 E8M0 codes. */
void oracle_mx_decode_tables(double *e4m3, double *e8m0) {
    for (int c = 0; c < 256; ++c) {
        e4m3[c] = e4m3_to_double((uint8_t)c);
        e8m0[c] = e8m0_to_double((uint8_t)c);
    }
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

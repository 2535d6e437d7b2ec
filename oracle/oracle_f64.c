/*
 * oracle_f64.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the FP32 tiled
 * matrix multiply computes, used to check the CUDA path.  Nothing on the
 * product path may link, load or call this file; only the tests, the smoke
 * check and the benchmark's CPU-baseline leg do.  It shares no code, header
 * or constant with the CUDA library.
 *
 * Sources (the surveyed web pages):
 *  - "CUDA 深入浅出（五）: Vectorized Load 和 Shared Memory Layout"
 *    (csh0101.cc), section "这一篇放进 GEMM 路径里看": the product is the
 *    textbook C = A x B; the tiled kernel only reorders data movement.
 *  - same page, section "对齐也要从数据分配开始": rows of a stored matrix
 *    start lda / ldb / ldc elements apart (leading dimensions).
 *  - "CUDA 深入浅出（四）: 怎么高效访问 Shared Memory", section
 *    "padding 为什么有用": layout changes do not change the mathematics.
 *  - "Memory Bank 机制与加速计算" (ykliu.com), section "地址怎样落到 bank":
 *    bank = (byte_address / 4) % 32; section "四种访问，四种结果":
 *    a conflict is the same bank at a different 32-bit word, the same word
 *    is broadcast; section "为什么 double 和 float4 要另算": wide accesses
 *    naturally need several wavefronts and must be analysed by the words
 *    they touch.
 *
 * Arithmetic: every product of two FP32 values is exact in FP64 (24+24 <
 * 53 significand bits), and the sum runs over k in increasing order in FP64.
 * The absolute-value product (|A|.|B|)_ij is formed in the same pass; the
 * acceptance bound for FP32 results is stated in terms of it.
 *
 * Parity status: every function here is pinned by tests that do not use
 * this file's arithmetic (hand-computed cases, closed forms, numpy's float64
 * matmul, exact rational brute force, the pages' printed bank examples and
 * the gcd law from the bank page).
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of host threads the OpenMP loops use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * C[i*ldc + j] = sum_{k<K} A[i*lda + k] * B[k*ldb + j]   (FP64, increasing k)
 * absAB[i*ldc + j] = sum_{k<K} |A[i*lda + k]| * |B[k*ldb + j]|  (if non-NULL)
 *
 * A is M x K row-major with row stride lda, B is K x N row-major with row
 * stride ldb, C and absAB are M x N row-major with row stride ldc.
 * K == 0 gives C = 0 (the empty sum).  Returns 0, or -1 on a bad argument.
 * Loop order i-k-j: each output row is built up one k at a time, so each
 * C[i][j] still receives its terms in increasing k.
 */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    double *C, int64_t ldc, double *absAB) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return -1;
    if (M == 0 || N == 0) return 0;
    if (C == NULL) return -1;
    if (K > 0 && (A == NULL || B == NULL)) return -1;
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i) {
        double *c = C + i * ldc;
        double *s = absAB ? absAB + i * ldc : NULL;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        if (s) for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const float *b = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) c[j] += a * (double)b[j];
            if (s) {
                const double aa = a < 0 ? -a : a;
                for (int64_t j = 0; j < N; ++j) {
                    const double bb = (double)b[j];
                    s[j] += aa * (bb < 0 ? -bb : bb);
                }
            }
        }
    }
    return 0;
}

/*
 * The same definition evaluated only at n chosen outputs (rows[t], cols[t]):
 * out[t] = sum_k A[rows[t]*lda + k] * B[k*ldb + cols[t]], absout[t] likewise
 * with absolute values.  Used where the full product is too large for the
 * CPU.  Returns 0, or -1 on a bad argument or an index out of range.
 */
int oracle_gemm_sampled_f64(int64_t n, const int64_t *rows, const int64_t *cols,
                            int64_t M, int64_t N, int64_t K,
                            const float *A, int64_t lda,
                            const float *B, int64_t ldb,
                            double *out, double *absout) {
    if (n < 0 || M < 0 || N < 0 || K < 0) return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1)) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < n; ++t) {
        double c = 0.0, s = 0.0;
        const int64_t i = rows[t], j = cols[t];
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const double b = (double)B[k * ldb + j];
            c += a * b;
            s += (a < 0 ? -a : a) * (b < 0 ? -b : b);
        }
        out[t] = c;
        if (absout) absout[t] = s;
    }
    return 0;
}

/* ---------------------------------------------------------------------
 * Shared-memory bank model (bank page, "地址怎样落到 bank" and
 * "四种访问，四种结果"; wide accesses per "为什么 double 和 float4 要另算").
 * ------------------------------------------------------------------- */

/* bank = (byte_address / 4) % 32 : 32 banks, each 4 bytes wide, interleaved. */
int oracle_bank_of(uint64_t byte_address) {
    return (int)((byte_address / 4u) % 32u);
}

/*
 * One warp-wide shared-memory request.  Lane l (active[l] != 0) touches
 * width_bytes / 4 consecutive 32-bit words starting at byte_address[l]
 * (width_bytes is 4, 8 or 16 and each address is a multiple of it).
 *
 * Reading of the pages: one pass over the banks (a wavefront) can serve one
 * 32-bit word per bank and hand that word to every lane that asked for it
 * (broadcast); two different words in the same bank need two passes
 * (conflict).  So the passes the request needs are the largest number of
 * distinct words that fall in any one bank.  A wide request may need several
 * passes without any conflict simply because it moves more than 32 distinct
 * words; the least it can need is ceil(distinct_words / 32).
 *
 * Outputs: *wavefronts (passes needed), *ideal (ceil(distinct words / 32)),
 * *degree (the largest number of distinct words in one bank, as for a
 * scalar access), *distinct (number of distinct words).  Returns 0, or -1 on
 * a bad argument (width not 4/8/16, misaligned address, more than 32 lanes).
 */
int oracle_shared_request(int n_lanes, const uint64_t *byte_address,
                          const uint8_t *active, int width_bytes,
                          int *wavefronts, int *ideal, int *degree,
                          int *distinct) {
    if (n_lanes < 0 || n_lanes > 32) return -1;
    if (width_bytes != 4 && width_bytes != 8 && width_bytes != 16) return -1;
    const int wpl = width_bytes / 4;
    uint64_t words[32 * 4];
    int nw = 0;
    for (int l = 0; l < n_lanes; ++l) {
        if (active && !active[l]) continue;
        if (byte_address[l] % (uint64_t)width_bytes) return -1;
        for (int w = 0; w < wpl; ++w) {
            const uint64_t word = byte_address[l] / 4u + (uint64_t)w;
            int seen = 0;
            for (int q = 0; q < nw; ++q)
                if (words[q] == word) { seen = 1; break; }
            if (!seen) words[nw++] = word;
        }
    }
    int per_bank[32];
    memset(per_bank, 0, sizeof per_bank);
    int worst = 0;
    for (int q = 0; q < nw; ++q) {
        const int b = oracle_bank_of(words[q] * 4u);
        if (++per_bank[b] > worst) worst = per_bank[b];
    }
    if (wavefronts) *wavefronts = worst;
    if (ideal) *ideal = (nw + 31) / 32;
    if (degree) *degree = worst;
    if (distinct) *distinct = nw;
    return 0;
}

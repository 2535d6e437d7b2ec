/*
 * oracle_f64.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the FP32 tiled
 * matrix multiply computes, used to check the CUDA path.  Nothing on the
 * product path may link, load or call this file; only the tests, the smoke
 * check and the benchmark's CPU-baseline leg do.  It shares no code, header
 * or constant with the CUDA library.
 *
 * Sources (the web pages this follows):
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

/* Distinct 32-bit words touched by the active lanes lo..hi-1; returns count. */
static int collect_words(int lo, int hi, const uint64_t *byte_address, const uint8_t *active,
                         int wpl, uint64_t *words) {
    int nw = 0;
    for (int l = lo; l < hi; ++l) {
        if (active && !active[l]) continue;
        for (int w = 0; w < wpl; ++w) {
            const uint64_t word = byte_address[l] / 4u + (uint64_t)w;
            int seen = 0;
            for (int q = 0; q < nw; ++q)
                if (words[q] == word) { seen = 1; break; }
            if (!seen) words[nw++] = word;
        }
    }
    return nw;
}

/* The pages' rule inside one pass: the largest number of distinct words that
 * fall in one bank (the same word is broadcast).  Also returns the bank mask. */
static int pass_degree(int nw, const uint64_t *words, uint32_t *bank_mask) {
    int per_bank[32];
    memset(per_bank, 0, sizeof per_bank);
    int worst = 0;
    uint32_t mask = 0;
    for (int q = 0; q < nw; ++q) {
        const int b = oracle_bank_of(words[q] * 4u);
        mask |= 1u << b;
        if (++per_bank[b] > worst) worst = per_bank[b];
    }
    if (bank_mask) *bank_mask = mask;
    return worst;
}

/* Largest number of distinct accesses among the groups of 4 consecutive
 * active lanes ("quads") in lo..hi-1. */
static int max_quad_distinct(int lo, int hi, const uint64_t *addr, const uint8_t *act) {
    int worst = 0;
    for (int q = lo; q < hi; q += 4) {
        uint64_t seen[4];
        int n = 0;
        for (int l = q; l < q + 4 && l < hi; ++l) {
            if (!act[l]) continue;
            int dup = 0;
            for (int t = 0; t < n; ++t)
                if (seen[t] == addr[l]) { dup = 1; break; }
            if (!dup) seen[n++] = addr[l];
        }
        if (n > worst) worst = n;
    }
    return worst;
}

/* 1 when no two active lanes in lo..hi-1 access the same address. */
static int all_distinct(int lo, int hi, const uint64_t *addr, const uint8_t *act) {
    for (int a = lo; a < hi; ++a) {
        if (!act[a]) continue;
        for (int b = a + 1; b < hi; ++b)
            if (act[b] && addr[b] == addr[a]) return 0;
    }
    return 1;
}

/* Passes for the active lanes lo..hi-1 of one wide request (see below). */
static int wide_passes(int lo, int hi, const uint64_t *addr, const uint8_t *act, int wpl,
                       int split_quarters, int *max_degree) {
    uint64_t words[32 * 4];
    uint32_t m0, m1;
    const int nw = collect_words(lo, hi, addr, act, wpl, words);
    if (!nw) return 0;
    const int deg = pass_degree(nw, words, &m0);
    if (!all_distinct(lo, hi, addr, act) || !split_quarters) {
        if (max_degree && deg > *max_degree) *max_degree = deg;
        if (!all_distinct(lo, hi, addr, act))
            return (max_quad_distinct(lo, hi, addr, act) + 1) / 2 * deg;
        return deg;
    }
    const int mid = lo + (hi - lo) / 2;
    const int n0 = collect_words(lo, mid, addr, act, wpl, words);
    const int d0 = n0 ? pass_degree(n0, words, &m0) : 0;
    const int n1 = collect_words(mid, hi, addr, act, wpl, words);
    const int d1 = n1 ? pass_degree(n1, words, &m1) : 0;
    const int dq = d0 > d1 ? d0 : d1;
    if (max_degree && dq > *max_degree) *max_degree = dq;
    if (!n0 || !n1 || !(m0 & m1)) return dq;
    return d0 + d1;
}

/*
 * One warp-wide shared-memory request.  Lane l (active[l] != 0) touches
 * width_bytes / 4 consecutive 32-bit words starting at byte_address[l]
 * (width_bytes is 4, 8 or 16 and each address is a multiple of it).
 *
 * Within one pass over the banks (a wavefront) each bank serves one 32-bit
 * word, which may go to every lane that asked for it (broadcast); two
 * different words in one bank need two passes (conflict).  This is the bank
 * page's rule ("四种访问，四种结果"), and for 4-byte accesses the passes are
 * the largest number of distinct words in one bank (the conflict degree).
 *
 * For 8- and 16-byte accesses the same page says to analyse the lanes each
 * transaction actually serves ("为什么 double 和 float4 要另算").  The lane
 * grouping used here was fitted to ncu wavefront counts of 26 lane patterns
 * x 2 widths measured on sm_103 (tests/probes/lds_probe.cu, counts in
 * tests/golden/lds_wavefronts_sm103.txt), and reproduces all of them:
 *   8-byte : the whole warp is one group;
 *   16-byte: each half-warp is a group, and the two halves never share passes.
 * A group whose lanes all read different addresses needs as many passes as
 * its conflict degree (for 16 bytes: per 8-lane quarter, the two quarters
 * sharing passes when their banks are disjoint).  A group in which some
 * lanes share an address (a broadcast) is served 2 distinct accesses per
 * quad of 4 consecutive lanes per pass, each pass also limited by the
 * conflict degree: passes = ceil(most distinct accesses in a quad / 2) x
 * degree.
 *
 * Outputs: *wavefronts (passes needed), *ideal (least passes the same amount
 * of distinct data could need: one per 32 distinct words, counted per
 * half-warp for 16-byte accesses), *degree (largest number of distinct words
 * in one bank within one group), *distinct (distinct words over the warp).
 * Returns 0, or -1 on a bad argument (width not 4/8/16, misaligned address,
 * more than 32 lanes).
 */
int oracle_shared_request(int n_lanes, const uint64_t *byte_address,
                          const uint8_t *active, int width_bytes,
                          int *wavefronts, int *ideal, int *degree,
                          int *distinct) {
    if (n_lanes < 0 || n_lanes > 32) return -1;
    if (width_bytes != 4 && width_bytes != 8 && width_bytes != 16) return -1;
    const int wpl = width_bytes / 4;
    uint64_t addr[32];
    uint8_t act[32];
    for (int l = 0; l < 32; ++l) {
        const int on = l < n_lanes && (!active || active[l]);
        if (on && byte_address[l] % (uint64_t)width_bytes) return -1;
        addr[l] = on ? byte_address[l] : 0;
        act[l] = (uint8_t)on;
    }
    uint64_t words[32 * 4];
    const int nw = collect_words(0, 32, addr, act, wpl, words);
    int deg = 0, wf = 0, id = 0;
    if (width_bytes == 4) {
        uint32_t m;
        deg = nw ? pass_degree(nw, words, &m) : 0;
        wf = deg;
        id = (nw + 31) / 32;
    } else if (width_bytes == 8) {
        wf = wide_passes(0, 32, addr, act, wpl, 0, &deg);
        id = (nw + 31) / 32;
    } else {
        for (int h = 0; h < 2; ++h) {
            wf += wide_passes(16 * h, 16 * h + 16, addr, act, wpl, 1, &deg);
            const int nh = collect_words(16 * h, 16 * h + 16, addr, act, wpl, words);
            id += (nh + 31) / 32;
        }
    }
    if (wavefronts) *wavefronts = wf;
    if (ideal) *ideal = id;
    if (degree) *degree = deg;
    if (distinct) *distinct = nw;
    return 0;
}

/* ---------------------------------------------------------------------
 * Matrix transpose (bank page, "放进矩阵转置里看"): the input is a
 * rows x cols row-major FP32 matrix (row i at in + i*ld_in), the output the
 * cols x rows matrix with out[j][i] = in[i][j] (row j at out + j*ld_out); the
 * two must not overlap.  Pure data movement: bit-exact.
 * Returns 0, or -1 on a bad argument.
 * ------------------------------------------------------------------- */
int oracle_transpose_f32(int64_t rows, int64_t cols, const float *in, int64_t ld_in,
                         float *out, int64_t ld_out) {
    if (rows < 0 || cols < 0) return -1;
    if (ld_in < (cols > 1 ? cols : 1) || ld_out < (rows > 1 ? rows : 1)) return -1;
    if (rows == 0 || cols == 0) return 0;
    if (in == NULL || out == NULL) return -1;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j)
            memcpy(out + j * ld_out + i, in + i * ld_in + j, sizeof(float));
    return 0;
}

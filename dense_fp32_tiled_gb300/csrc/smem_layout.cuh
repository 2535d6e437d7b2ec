// smem_layout.cuh -- tile geometry and every shared-memory index map of the
// tiled FP32 matrix multiply kernel.
//
// The kernel computes its shared-memory addresses only through these
// functions, and the host-side layout query (sgemm_f32_smem_request) runs
// the same functions for every lane, so a host test can apply the bank rule
// (bank = (byte_address / 4) % 32; bank page, "地址怎样落到 bank") to exactly
// the addresses the kernel issues.
//
// Layout (per pipeline stage):
//   As: BK x BM floats, k-major ("transposed" A tile, as in the
//       vectorised-load page's "shared memory transpose 的基本想法"), with an
//       XOR swizzle of the 8-float block index inside each 32-float bank row:
//       logical (k, m) lives at word k*BM + (m ^ ((k & 3) << 3)).  The
//       swizzle ("Padding 之外的选择" on the bank page) keeps 4-float groups
//       contiguous and 16-byte aligned, so fragment reads stay 128-bit, and
//       spreads the transposing 4-byte copies of 4 consecutive k over 4
//       different bank groups.  +1 padding would break the 16-byte alignment
//       of the fragment reads.
//   Bs: BK x BN floats, row-major as in global memory (the page's
//       "原样写" variant); fragment reads along n are contiguous.
#pragma once

#if defined(__CUDACC__)
#define SG_HD __host__ __device__ __forceinline__
#else
#define SG_HD inline
#endif

namespace sg {

constexpr int BM = 128;          // CTA tile rows (M)
constexpr int BN = 128;          // CTA tile cols (N)
constexpr int BK = 16;           // K depth of one pipeline stage
constexpr int NT = 256;          // threads per CTA (8 warps)
constexpr int STAGES = 4;        // global->shared pipeline depth
constexpr int TM = 8;            // per-thread register tile rows
constexpr int TN = 8;            // per-thread register tile cols
constexpr int WARPS_M = 4;       // warp grid over the CTA tile
constexpr int WARPS_N = 2;
constexpr int WM = BM / WARPS_M; // 32 rows per warp
constexpr int WN = BN / WARPS_N; // 64 cols per warp
constexpr int A_STAGE_FLOATS = BK * BM;
constexpr int B_STAGE_FLOATS = BK * BN;
constexpr int STAGE_FLOATS = A_STAGE_FLOATS + B_STAGE_FLOATS;
constexpr int SMEM_BYTES = STAGES * STAGE_FLOATS * 4;
constexpr int A_COPIES = BM * BK / NT;  // 4-byte copies per thread per stage

static_assert(WARPS_M * WARPS_N * 32 == NT, "warp grid");
static_assert(WM == 4 * TM && WN == 8 * TN, "lane grid 4 x 8");
static_assert((STAGE_FLOATS * 4) % 128 == 0, "stages start on a bank row");

// ---- shared-memory word offsets inside one stage -----------------------
SG_HD int as_word(int k, int m) { return k * BM + (m ^ ((k & 3) << 3)); }
SG_HD int bs_word(int k, int n) { return A_STAGE_FLOATS + k * BN + n; }

// ---- global->shared copy maps -----------------------------------------
// A: 4-byte copies (a 16-byte copy cannot transpose).  Warp w owns rows
// [16w, 16w+16); copy q of lane l moves element (k, m) with
//   k = 4*(q & 3) + (l & 3),  m = 16w + 8*(q >> 2) + (l >> 2).
// A warp instruction therefore reads 8 rows x 16 contiguous bytes of A.
SG_HD void a_copy_coord(int tid, int q, int &k, int &m) {
    const int w = tid >> 5, l = tid & 31;
    k = 4 * (q & 3) + (l & 3);
    m = 16 * w + 8 * (q >> 2) + (l >> 2);
}

// B: vector copies of VB floats (VB = 4, 2, 1 by alignment class).  Copy q
// of thread t moves the VB floats at (k, n) with consecutive threads on
// consecutive vectors of one row, so a warp reads 32*VB contiguous floats.
template <int VB>
SG_HD void b_copy_coord(int tid, int q, int &k, int &n) {
    constexpr int PER_ROW = BN / VB;          // vectors per tile row
    constexpr int ROWS_PER_PASS = NT / PER_ROW;
    k = tid / PER_ROW + ROWS_PER_PASS * q;
    n = (tid % PER_ROW) * VB;
}
template <int VB>
SG_HD constexpr int b_copies() { return BK * BN / (NT * VB); }

// ---- register-tile maps ------------------------------------------------
// Warp w covers rows WM*(w / WARPS_N) and cols WN*(w % WARPS_N); lane l is
// (lr, lc) = (l >> 3, l & 7).  Thread rows: 4*lr + {0..3} and 16 + 4*lr +
// {0..3}; thread cols: 4*lc + {0..3} and 32 + 4*lc + {0..3}.  Each k step
// a thread reads two 4-float groups of As row k and two of Bs row k.
SG_HD int frag_row0(int tid) {
    const int w = tid >> 5, l = tid & 31;
    return WM * (w / WARPS_N) + 4 * (l >> 3);
}
SG_HD int frag_col0(int tid) {
    const int w = tid >> 5, l = tid & 31;
    return WN * (w % WARPS_N) + 4 * (l & 7);
}
// i, j in [0, 8): row / col of register-tile element (i, j).
SG_HD int frag_row(int tid, int i) { return frag_row0(tid) + (i & 3) + 16 * (i >> 2); }
SG_HD int frag_col(int tid, int j) { return frag_col0(tid) + (j & 3) + 32 * (j >> 2); }

// ---- tile rasterisation ------------------------------------------------
// Linear CTA index -> (tile row, tile col), walking GROUP_M tile rows at a
// time so CTAs resident together share A row panels and B column panels.
constexpr int GROUP_M = 8;
SG_HD void tile_of(int bid, int tiles_m, int tiles_n, int &tm, int &tn) {
    const int per_group = GROUP_M * tiles_n;
    const int g = bid / per_group;
    const int first = g * GROUP_M;
    const int rows = (tiles_m - first) < GROUP_M ? (tiles_m - first) : GROUP_M;
    const int r = bid - g * per_group;
    tm = first + r % rows;
    tn = r / rows;
}

}  // namespace sg

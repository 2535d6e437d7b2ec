// smem_layout.cuh -- tile geometry and every shared-memory index map of the
// tiled FP32 matrix multiply kernel.
//
// The kernel computes its shared-memory addresses only through these
// functions, and the host-side layout query (sgemm_f32_smem_request) runs
// the same functions for every lane, so a host test can apply the bank rule
// (bank = (byte_address / 4) % 32; bank page, "地址怎样落到 bank") to exactly
// the addresses the kernel issues.
//
// Layout.  A ring of STAGES stages, each holding
//   Bs : BK x BN floats, the B tile row-major as in global memory (the
//        vectorised-load page's "原样写" variant); fragment reads along n
//        are contiguous;
//   Ar : BM x BK floats, the A tile as it arrives from global memory (row m,
//        k contiguous), each 64-byte row split in four 16-byte groups stored
//        at group g ^ ((m >> 1) & 3) (an XOR swizzle, "Padding 之外的选择" on
//        the bank page: 16-byte copies of 8 rows and 128-bit reads of 32
//        consecutive rows both spread over all banks);
// followed by two buffers
//   As : BK x BM floats, k-major ("transposed" A tile, the vectorised-load
//        page's "shared memory transpose 的基本想法"): logical (k, m) at word
//        k*BM + m.  Each thread moves its share of Ar to As one tile ahead of
//        use (two 128-bit reads, eight 4-byte stores); each warp store writes
//        32 consecutive m of one k (one word per bank) and the fragment reads
//        take 4 consecutive m (16-byte aligned), so As needs no padding.
//
// With A supplied already transposed (the k-major copy At = A^T, K x M,
// that sgemm_f32_ws can make in its workspace), each stage of a separate
// STAGES_AT-deep ring receives a BK_AT x 128 tile of B (row-major, atb_word)
// and a BK_AT x 128 k-major tile of At (logical (k, m) at word k*BM + m, the
// As layout, at_word) directly from tensor copies, so the fragment reads are
// those of As and no shared store is needed.
//
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
constexpr int STAGES = 3;        // copy ring depth (tiles in flight: STAGES - 1)
constexpr int BK_AT = 32;        // K depth of one stage when A arrives k-major
constexpr int STAGES_AT = 3;     // ring depth when A arrives k-major (no As buffers)
constexpr int TM = 8;            // per-thread register tile rows
constexpr int TN = 8;            // per-thread register tile cols
constexpr int WARPS_M = 4;       // warp grid over the CTA tile
constexpr int WARPS_N = 2;
constexpr int WM = BM / WARPS_M; // 32 rows per warp
constexpr int WN = BN / WARPS_N; // 64 cols per warp
constexpr int B_STAGE_FLOATS = BK * BN;
constexpr int A_RAW_FLOATS = BM * BK;
constexpr int STAGE_FLOATS = B_STAGE_FLOATS + A_RAW_FLOATS;
constexpr int AS_FLOATS = BK * BM;
constexpr int AS_BASE = STAGES * STAGE_FLOATS;  // first As buffer (floats)
constexpr int SMEM_FLOATS = AS_BASE + 2 * AS_FLOATS;
constexpr int SMEM_ALIGN = 1024;  // all offsets above are from a 1024-byte aligned base
constexpr int SMEM_BYTES = SMEM_FLOATS * 4 + SMEM_ALIGN;  // dynamic size requested, with alignment slack
constexpr int A_VECS = BM * BK / (4 * NT);  // float4 of A a thread transposes per tile

static_assert(WARPS_M * WARPS_N * 32 == NT, "warp grid");
static_assert(WM == 4 * TM && WN == 8 * TN, "lane grid 4 x 8");
// the k-major ring: per stage a BK_AT x BN tile of B, then a BK_AT x BM tile of At
constexpr int AT_STAGE_FLOATS = BK_AT * BN + BK_AT * BM;
constexpr int SMEM_AT_BYTES = STAGES_AT * AT_STAGE_FLOATS * 4 + SMEM_ALIGN;
static_assert((STAGE_FLOATS * 4) % 128 == 0 && (AS_FLOATS * 4) % 128 == 0, "regions start on a bank row");
static_assert(NT == 256 && BM == 128 && BK == 16, "A copy and transpose maps cover 128 rows x 16 k");

// ---- shared-memory word offsets (floats from the start of the block) --
SG_HD int bs_word(int stage, int k, int n) { return stage * STAGE_FLOATS + k * BN + n; }
SG_HD int ar_word(int stage, int m, int k) {
    return stage * STAGE_FLOATS + B_STAGE_FLOATS + m * BK + 4 * ((k >> 2) ^ ((m >> 1) & 3)) + (k & 3);
}
SG_HD int as_word(int buf, int k, int m) { return AS_BASE + buf * AS_FLOATS + k * BM + m; }
SG_HD int atb_word(int stage, int k, int n) { return stage * AT_STAGE_FLOATS + k * BN + n; }
SG_HD int at_word(int stage, int k, int m) { return stage * AT_STAGE_FLOATS + BK_AT * BN + k * BM + m; }

// ---- global->shared copy maps -----------------------------------------
// A (16-byte class): copy q of thread t moves the 4 floats A[m][k..k+3] with
//   m = 64q + t/4,  k = 4 (t % 4),
// so a warp copies 8 rows x 64 contiguous bytes.
SG_HD void a_copy16_coord(int tid, int q, int &m, int &k) {
    m = 64 * q + (tid >> 2);
    k = 4 * (tid & 3);
}
constexpr int A_COPIES16 = BM * BK / (4 * NT);
// A (4-byte class, misaligned rows): copy q of thread t moves A[m][k] with
//   m = 16q + t/16,  k = t % 16.
SG_HD void a_copy4_coord(int tid, int q, int &m, int &k) {
    m = 16 * q + (tid >> 4);
    k = tid & 15;
}
constexpr int A_COPIES4 = BM * BK / NT;

// A transpose: float4 f (0 or 1) of lane l in warp w is A[m][k..k+3] with
//   m = 32(w % 4) + l,  k = 8(w / 4) + 4f,
// read from Ar (lanes on 32 consecutive rows) and written to As as 4 scalar
// stores, component c to (k + c, m): 32 consecutive words per store.
SG_HD void a_xpose_coord(int tid, int f, int &k, int &m) {
    const int w = tid >> 5, l = tid & 31;
    m = 32 * (w & 3) + l;
    k = 8 * (w >> 2) + 4 * f;
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
// Warp w covers rows WM*(w / WARPS_N) and cols WN*(w % WARPS_N).  Lane
// l = 16h + 4q + 2e1 + e0 (h half-warp, q quad, e1 e0 lane bits in the quad)
// sits at (lr, lc) = (2h + e0, 2q + e1) of a 4 x 8 lane grid: each quad holds
// 2 rows x 2 columns of the grid.  Thread rows: 4*lr + {0..3} and
// 16 + 4*lr + {0..3}; thread cols: 4*lc + {0..3} and 32 + 4*lc + {0..3}.
SG_HD int lane_lr(int l) { return 2 * (l >> 4) + (l & 1); }
SG_HD int lane_lc(int l) { return 2 * ((l >> 2) & 3) + ((l & 3) >> 1); }
SG_HD int frag_row0(int tid) {
    const int w = tid >> 5, l = tid & 31;
    return WM * (w / WARPS_N) + 4 * lane_lr(l);
}
SG_HD int frag_col0(int tid) {
    const int w = tid >> 5, l = tid & 31;
    return WN * (w % WARPS_N) + 4 * lane_lc(l);
}
// i, j in [0, 8): row / col of register-tile element (i, j).
SG_HD int frag_row(int tid, int i) { return frag_row0(tid) + (i & 3) + 16 * (i >> 2); }
SG_HD int frag_col(int tid, int j) { return frag_col0(tid) + (j & 3) + 32 * (j >> 2); }

// ---- register-tile maps of the k-major kernels (8 x 16 per thread) -------
// 128 threads: warp w covers rows 64*(w / 2) and cols 64*(w % 2) of the CTA
// tile.  Lane l = 16h + 4q + 2e1 + e0 sits at (lr, lc) = (2q + e0, 2h + e1)
// of an 8 x 4 lane grid (each quad again holds 2 rows x 2 columns of the
// grid, so each 128-bit fragment read costs the minimum 2 wavefronts).
// Thread rows: 4*lr + {0..3} and 32 + 4*lr + {0..3}; thread cols:
// 16g + 4*lc + {0..3} for g = 0..3.  Per k step: 2 A reads and 4 B reads of
// 128 bits for 64 packed FMAs.
constexpr int NT16 = 128;        // threads per CTA of the k-major kernels
constexpr int TN16 = 16;         // their register tile cols (rows: TM = 8)
SG_HD int lane16_lr(int l) { return 2 * ((l >> 2) & 3) + (l & 1); }
SG_HD int lane16_lc(int l) { return 2 * (l >> 4) + ((l >> 1) & 1); }
SG_HD int frag16_row0(int tid) { return 64 * ((tid >> 5) >> 1) + 4 * lane16_lr(tid & 31); }
SG_HD int frag16_col0(int tid) { return 64 * ((tid >> 5) & 1) + 4 * lane16_lc(tid & 31); }
// i in [0, 8), j in [0, 16): row / col of register-tile element (i, j).
SG_HD int frag16_row(int tid, int i) { return frag16_row0(tid) + (i & 3) + 32 * (i >> 2); }
SG_HD int frag16_col(int tid, int j) { return frag16_col0(tid) + (j & 3) + 16 * (j >> 2); }
static_assert(NT16 == 4 * 32 && 2 * (8 * 4 * 2) == BM && 2 * (4 * 4 * 4) == BN, "2 x 2 warps of 64 x 64");

// ---- partial tile of the cluster split of K --------------------------------
// After its K loop each CTA of a cluster leaves its 128 x 128 partial sums in
// its own shared memory (reusing the ring), logical (row, col) at
// row*BN + 4*((col/4) ^ (row % 8)) + col % 4: the 8 x 8 threads' 128-bit
// stores (a quarter-warp: 2 rows x 4 column groups, rows 4 apart) fall on 8
// distinct bank groups, and a warp reading one row (32 groups) needs the
// minimum 4 passes.
SG_HD int pt_word(int row, int col) { return row * BN + 4 * ((col >> 2) ^ (row & 7)) + (col & 3); }
static_assert(BM * BN <= SMEM_FLOATS, "the partial tile fits the shared block");
// Store q (0 .. 2 TM - 1) of thread tid: row q/2 of its 8 x 8 tile, the four
// columns of half q%2.
SG_HD void pt_store_coord(int tid, int q, int &row, int &col) {
    row = frag_row(tid, q >> 1);
    col = frag_col0(tid) + 32 * (q & 1);
}
// Read j of thread tid when summing the rows from r0 on: warp w takes rows
// r0 + w, r0 + w + 8, ..., lane l the columns 4 l .. 4 l + 3.
SG_HD void pt_sum_coord(int tid, int j, int r0, int &row, int &col) {
    row = r0 + (tid >> 5) + (NT / 32) * j;
    col = 4 * (tid & 31);
}

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

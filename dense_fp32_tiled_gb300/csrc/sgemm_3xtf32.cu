// sgemm_3xtf32.cu -- FP32 C = A.B on the 5th-generation tensor cores of GB300
// (sm_103a: tcgen05.mma with TMEM accumulators), by the 3xTF32 split.
//
// Each FP32 operand x is split into two TF32 values, hi = rna_tf32(x) and
// lo = rna_tf32(x - hi), so x = hi + lo + e with |e| <= 2^-22 |x|; then
//   A.B ~= Ahi.Bhi + Ahi.Blo + Alo.Bhi
// (the dropped Alo.Blo is below 2^-22 |a||b| per product).  The pages
// describe only the SIMT path (the textbook product C = A x B, vectorised-load
// page, "这一篇放进 GEMM 路径里看"); this is an additional implementation of
// the same product, checked against the same FP32 tolerance.
//
// Two kernels:
//   1. split: A -> A_hi, A_lo (M x Kp, row-major) and B -> Bt_hi, Bt_lo
//      (N x Kp: B transposed, so both operands are K-major), Kp = K rounded
//      up to 4, in the caller's workspace; the K padding is written as 0.
//   2. mma: one CTA pair (cluster of 2) per 256 x 256 tile of C.  In each CTA
//      one thread issues TMA copies (128 x 32 boxes, 128-byte swizzle) of its
//      halves of the four operand panels into a 3-stage ring; one thread of
//      CTA 0 issues, per 8-deep K step, tcgen05.mma.cta_group::2.kind::tf32
//      (M = N = 256) for Ahi.Bhi, Ahi.Blo and Alo.Bhi into one accumulator,
//      which restarts every 128 K in one of two tensor-memory buffer sets;
//      eight warps per CTA add each finished block into FP32 registers
//      (tcgen05.ld) and finally store C.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "ctx_key.cuh"
#include "nvtx_range.cuh"
#include "sgemm_f32.h"

namespace {

// ---- split kernel ----------------------------------------------------------
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

constexpr int ST = 64;  // split-transpose tile
constexpr int ST_STRIDE = ST + 1;

// Block (32, 8).  blockIdx.x < a_blocks: rows of A (one row per y-thread,
// 32 consecutive k per warp access); else tiles of B transposed through a
// padded 64 x 64 shared tile.
__global__ void __launch_bounds__(256) split_kernel(const float *__restrict__ A, int lda, const float *__restrict__ B,
                                                    int ldb, int M, int N, int K, int Kp, float *__restrict__ a_hi,
                                                    float *__restrict__ a_lo, float *__restrict__ bt_hi,
                                                    float *__restrict__ bt_lo, int a_blocks, int b_tiles_k) {
    __shared__ float tile[ST * ST_STRIDE];
    // the MMA grid queued behind this one may start its set-up now; it waits
    // for this grid to complete before its first copy of split data
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int tx = threadIdx.x, ty = threadIdx.y;
    if (static_cast<int>(blockIdx.x) < a_blocks) {
        // 8 rows of A per block, the whole padded K range
        const int row = blockIdx.x * 8 + ty;
        if (row >= M) return;
        const float *src = A + static_cast<size_t>(row) * lda;
        float *hi = a_hi + static_cast<size_t>(row) * Kp, *lo = a_lo + static_cast<size_t>(row) * Kp;
        for (int k = tx; k < Kp; k += 32) {
            const float x = k < K ? __ldg(src + k) : 0.0f;
            const float h = tf32_rna(x);
            hi[k] = h;
            lo[k] = tf32_rna(x - h);
        }
        return;
    }
    // B^T tile: input B rows k0.., cols n0..; output Bt rows n, cols k
    const int t = blockIdx.x - a_blocks;
    const int tk = t % b_tiles_k, tn = t / b_tiles_k;
    const int k0 = tk * ST, n0 = tn * ST;
#pragma unroll
    for (int h = 0; h < ST; h += 32)
#pragma unroll
        for (int j = 0; j < ST; j += 8) {
            const int k = k0 + ty + j, n = n0 + tx + h;
            tile[(ty + j) * ST_STRIDE + tx + h] = (k < K && n < N) ? __ldg(B + static_cast<size_t>(k) * ldb + n) : 0.0f;
        }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < ST; h += 32)
#pragma unroll
        for (int j = 0; j < ST; j += 8) {
            const int n = n0 + ty + j, k = k0 + tx + h;
            if (n < N && k < Kp) {
                const float x = tile[(tx + h) * ST_STRIDE + ty + j];
                const float hv = tf32_rna(x);
                bt_hi[static_cast<size_t>(n) * Kp + k] = hv;
                bt_lo[static_cast<size_t>(n) * Kp + k] = tf32_rna(x - hv);
            }
        }
}

// ---- tensor-core kernel ------------------------------------------------------
// A CTA pair (a cluster of 2, placed by the hardware on one TPC) computes a
// 256 x 256 tile of C with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 8).
// CTA r of the pair holds rows 128r .. 128r+127 of the tile's A panel and rows
// 128r .. 128r+127 of its Bt panel (C columns n0+128r ..) in shared memory;
// the tensor core of each SM reads its own A half and both B halves, and
// writes the accumulator for its 128 rows of C, all 256 columns, into its own
// tensor memory.  Per SM this reads 8 KiB of operands from shared memory per
// 128 x 256 x 8 MMA (the 1-CTA 128 x 128 shape needs the same 8 KiB for half
// the work), which keeps operand traffic below the shared-memory bandwidth.
constexpr int PM = 256, PN = 256;               // pair tile
constexpr int TBM = 128, TBK = 32;              // per-CTA box: 128 rows x 32 K (one 128-byte swizzle row)
constexpr int TSTAGES = 3;
constexpr int BOX_BYTES = TBM * TBK * 4;        // 16 KiB
constexpr int STAGE_BYTES = 4 * BOX_BYTES;      // halves of A_hi, A_lo, Bt_hi, Bt_lo
constexpr int MMA_SMEM = TSTAGES * STAGE_BYTES + 1024;  // + alignment slack
constexpr int KBLK = 4;                         // K tiles (128 K) per accumulation block
constexpr int ACC_COLS = PN;                    // one FP32 accumulator per column of C
constexpr int TMEM_COLS = 2 * ACC_COLS;         // two buffer sets
constexpr int EPI_WARPS = 8;                    // warp w: TMEM lanes 32(w%4).., columns EPI_COLS(w/4)..
constexpr int EPI_COLS = PN * 4 / EPI_WARPS;    // accumulator columns per summing thread
constexpr int COPY_WARP = EPI_WARPS, MMA_WARP = EPI_WARPS + 1;
constexpr int TC_THREADS = (EPI_WARPS + 2) * 32;
constexpr uint32_t kWaitPolls = 1u << 22;
static_assert(PM == 2 * TBM && PN == 2 * TBM, "each CTA holds half of both panels");

// Shared-memory matrix descriptor for a K-major operand box of 128 rows x
// 128 bytes stored with the 128-byte swizzle (the layout a TMA copy with
// CU_TENSOR_MAP_SWIZZLE_128B writes): 8-row groups of 1024 bytes, start
// address in 16-byte units (bits 0-13), leading-dimension offset (bits 16-29,
// unused for this layout, set to 1), stride between 8-row groups (bits
// 32-45, 1024 bytes), descriptor version 1 (bits 46-47), base offset 0
// (1024-byte aligned boxes), layout 2 = 128-byte swizzle (bits 61-63).
__host__ __device__ constexpr uint64_t smem_desc_sw128(uint32_t smem_addr) {
    return (static_cast<uint64_t>((smem_addr >> 4) & 0x3FFF)) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor for kind::tf32: D = F32 (bits 4-5 = 1), A and B =
// TF32 (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc_tf32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// Arrive on a barrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait: gives up after `limit` polls and records the timeout.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, unsigned *timeout_flag,
                                          uint32_t limit = kWaitPolls) {
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++polls > limit) {
            *timeout_flag = 1u;
            break;
        }
    }
}
// TMA box load into this CTA's shared memory; completion is counted on
// `cluster_bar`, which may belong to the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t cluster_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
        : "memory");
}
__device__ __forceinline__ void umma_tf32_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this shared address in both CTAs of the pair
// when all tcgen05 operations issued so far by this thread are complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    const uint16_t both = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
            bar),
        "h"(both)
        : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns of tensor memory -> 8 registers per
// thread (thread i reads lane base + i).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcMaps {
    CUtensorMap a_hi, a_lo, b_hi, b_lo;
};

// Schedule (persistent grid of P CTA pairs).  The first dp_tiles pair tiles
// (whole waves, a multiple of P) run data-parallel: pair p takes tiles p,
// p + P, ..., so the tiles in flight at one time are neighbours in the
// rasterised order and share their operand panels in L2.  The remaining
// tiles (the last partial wave plus one full wave) are cut into units
// (tile, K block), NB = ceil(KT / KBLK) blocks per tile, and pair p takes
// units [floor(pU/Psk), floor((p+1)U/Psk)) of them (stream-K; pairs p >= Psk
// take none), so every pair ends at the same time whatever the tile count.  A tile whose blocks all fall in
// one pair is stored directly; a tile cut between pairs is finished by
// whichever of its parts arrives last (an atomic count per tile half), which
// adds all parts in part order, so the result does not depend on timing and
// no CTA waits for another.
struct SkPlan {
    int U;         // stream-K units = (T - dp_tiles) * NB (checked on the host to fit an int)
    int P;         // CTA pairs
    int Psk;       // pairs that share the stream-K units (<= P, each gets at least MIN_UNITS)
    int NB;        // K blocks per tile
    int KT;        // K tiles (TBK deep) per tile
    int dp_tiles;  // tiles run data-parallel, round-robin over the pairs
    int tiles_m;   // pair-tile rows
    int tiles_n;   // pair-tile columns
};

__device__ __forceinline__ int unit_start(int p, const SkPlan &pl) {
    return p >= pl.Psk ? pl.U : static_cast<int>(static_cast<long long>(p) * pl.U / pl.Psk);
}
// The pair whose stream-K range holds unit u: the largest p with unit_start(p) <= u.
__device__ __forceinline__ int pair_of_unit(int u, const SkPlan &pl) {
    return static_cast<int>((static_cast<long long>(u + 1) * pl.Psk - 1) / pl.U);
}
// Pair tile t -> (row, column) of pair tiles, walking 8 rows at a time.
__device__ __forceinline__ void pair_tile_coords(int t, const SkPlan &pl, int &tm, int &tn) {
    const int per_group = 8 * pl.tiles_n;
    const int g = t / per_group, first = g * 8;
    const int rows_in_group = (pl.tiles_m - first) < 8 ? (pl.tiles_m - first) : 8;
    const int r_in = t - g * per_group;
    tm = first + r_in % rows_in_group;
    tn = r_in / rows_in_group;
}
// Partial-sum slot of pair p's part of stream-K tile ts (counted from the
// first stream-K tile): 2p for the pair's first tile, 2p + 1 for its last
// (tiles in between are whole).
__device__ __forceinline__ int part_slot(int p, int ts, const SkPlan &pl) {
    return 2 * p + (ts == unit_start(p, pl) / pl.NB ? 0 : 1);
}
// The pair's segments in order: its data-parallel tiles, then its stream-K
// range cut at tile boundaries.  Segment = tile t, K blocks [kb0, kb1).
struct SegIter {
    int dp_next, dp_left;  // next data-parallel tile, how many remain
    int u, u_end;          // stream-K units still to cover
    __device__ SegIter(int pair, const SkPlan &pl)
        : dp_next(pair),
          dp_left(pl.dp_tiles > pair ? (pl.dp_tiles - pair + pl.P - 1) / pl.P : 0),
          u(unit_start(pair, pl)),
          u_end(unit_start(pair + 1, pl)) {}
    __device__ bool next(const SkPlan &pl, int &t, int &kb0, int &kb1) {
        if (dp_left > 0) {
            t = dp_next;
            kb0 = 0;
            kb1 = pl.NB;
            dp_next += pl.P;
            --dp_left;
            return true;
        }
        if (u >= u_end) return false;
        const int ts = u / pl.NB;
        const int seg_end = min(u_end, (ts + 1) * pl.NB);
        t = pl.dp_tiles + ts;
        kb0 = u - ts * pl.NB;
        kb1 = seg_end - ts * pl.NB;
        u = seg_end;
        return true;
    }
};
constexpr int SLOT_FLOATS = TBM * PN;  // one CTA's half of a pair tile

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(EPI_WARPS * 32) : "memory"); }

// Warps 0-7 read tensor memory and own the C rows, warp 8 lane 0 issues the
// copies, warp 9 holds the tensor-memory allocation and, in CTA 0 of the
// pair, its lane 0 issues the MMAs for both CTAs.
//
// Tensor memory holds two buffer sets of 128 x 256 FP32 accumulators.  Block
// g (counted over the pair's whole range) accumulates Ahi.Bhi + Ahi.Blo +
// Alo.Bhi over its K tiles from zero in set g % 2, and warps 0-7 of both CTAs
// add each finished block into FP32 registers with round-to-nearest adds
// while the tensor cores work on the next block.  The tensor core's own
// accumulation thus never spans more than 128 K, which bounds the rounding
// bias of its accumulator adds.
//
// Barriers: full[s] (CTA 0 only) completes when both CTAs' copies of stage s
// have landed; empty[s] (both CTAs) when the MMAs reading stage s are done;
// blk_full[set] (both) when a block's MMAs are done; blk_empty[set] (CTA 0)
// when the 16 summing warps of the pair have read the set.
//
// Workspace: counts[2T] (zeroed before each launch) and partials[2P][2]
// [128 x 256], each slot stored 4-column chunk by chunk so that a warp's 32
// rows write 512 contiguous bytes.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
sgemm_3xtf32_kernel(const __grid_constant__ TcMaps maps, float *__restrict__ C, int ldc, int M, int N,
                    const SkPlan pl, unsigned *__restrict__ counts, float *__restrict__ partials, int vc,
                    unsigned *timeout_flag) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[TSTAGES], empty_bar[TSTAGES], blk_full[2], blk_empty[2];
    __shared__ uint32_t tmem_base_slot;
    __shared__ int last_part;
    // same offset in both CTAs: the MMA addresses the peer's boxes with this CTA's descriptors
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&blk_full[b]), 1);
            mbar_init(smem_u32(&blk_empty[b]), 2 * EPI_WARPS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == MMA_WARP) {  // one warp of each CTA allocates, collectively, in both
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "n"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any remote arrive or copy
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = tmem_base_slot;

    if (warp == COPY_WARP) {
        if (lane == 0) {
            // the split operands come from the grid this one may overlap: wait for it (a no-op
            // when launched without a programmatic dependency)
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            const uint32_t full0 = peer_addr(smem_u32(&full_bar[0]), 0);  // CTA 0 counts both CTAs' bytes
            uint32_t it = 0;                                               // K tiles issued so far
            SegIter seg(pair, pl);
            int t, kb0, kb1;
            while (seg.next(pl, t, kb0, kb1)) {
                int tm, tn;
                pair_tile_coords(t, pl, tm, tn);
                const int m0 = tm * PM + static_cast<int>(rank) * TBM, nb = tn * PN + static_cast<int>(rank) * TBM;
                const int kt1 = min(kb1 * KBLK, pl.KT);
                for (int kt = kb0 * KBLK; kt < kt1; ++kt, ++it) {
                    const uint32_t s = it % TSTAGES;
                    if (it >= TSTAGES) mbar_wait(smem_u32(&empty_bar[s]), ((it / TSTAGES) - 1) & 1, timeout_flag);
                    if (rank == 0) mbar_expect_tx(smem_u32(&full_bar[s]), 2 * STAGE_BYTES);
                    const uint32_t bar = full0 + 8u * s;
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    tma_load_2d_pair(st + 0 * BOX_BYTES, &maps.a_hi, kt * TBK, m0, bar);
                    tma_load_2d_pair(st + 1 * BOX_BYTES, &maps.a_lo, kt * TBK, m0, bar);
                    tma_load_2d_pair(st + 2 * BOX_BYTES, &maps.b_hi, kt * TBK, nb, bar);
                    tma_load_2d_pair(st + 3 * BOX_BYTES, &maps.b_lo, kt * TBK, nb, bar);
                }
            }
            // let the last releases of every stage land before this CTA can exit
            for (uint32_t j = it > TSTAGES ? it - TSTAGES : 0; j < it; ++j)
                mbar_wait(smem_u32(&empty_bar[j % TSTAGES]), (j / TSTAGES) & 1, timeout_flag);
        }
    } else if (warp == MMA_WARP) {
        if (rank == 0 && lane == 0) {
            constexpr uint32_t idesc = instr_desc_tf32(PM, PN);
            uint32_t it = 0, g = 0;  // K tiles and blocks consumed so far
            SegIter seg(pair, pl);
            int t, kb0, kb1;
            while (seg.next(pl, t, kb0, kb1)) {
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int kt0 = kb * KBLK, kt1 = min(kt0 + KBLK, pl.KT);
                    const uint32_t set = g & 1;
                    if (g >= 2) mbar_wait(smem_u32(&blk_empty[set]), ((g / 2) - 1) & 1, timeout_flag);
                    const uint32_t t_acc = tmem + set * ACC_COLS;
                    for (int kt = kt0; kt < kt1; ++kt, ++it) {
                        const uint32_t s = it % TSTAGES;
                        mbar_wait(smem_u32(&full_bar[s]), (it / TSTAGES) & 1, timeout_flag);
                        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
                        const uint32_t st = sbase + s * STAGE_BYTES;
#pragma unroll
                        for (int j = 0; j < TBK / 8; ++j) {  // 8 TF32 = 32 bytes per MMA along K
                            const uint64_t ahi = smem_desc_sw128(st + 0 * BOX_BYTES + 32 * j);
                            const uint64_t alo = smem_desc_sw128(st + 1 * BOX_BYTES + 32 * j);
                            const uint64_t bhi = smem_desc_sw128(st + 2 * BOX_BYTES + 32 * j);
                            const uint64_t blo = smem_desc_sw128(st + 3 * BOX_BYTES + 32 * j);
                            umma_tf32_pair(t_acc, ahi, bhi, idesc, (kt > kt0 || j > 0) ? 1u : 0u);
                            umma_tf32_pair(t_acc, ahi, blo, idesc, 1u);
                            umma_tf32_pair(t_acc, alo, bhi, idesc, 1u);
                        }
                        umma_commit_pair(smem_u32(&empty_bar[s]));  // stage s free in both CTAs once these are done
                    }
                    umma_commit_pair(smem_u32(&blk_full[set]));
                }
            }
        }
    } else {
        // summing warps: per tile segment, sum its blocks, then store or hand over
        const int q = warp & 3, h = warp >> 2;
        const int rloc = 32 * q + lane;  // this thread's row within the CTA's 128
        const uint32_t t_off = (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(h * (EPI_COLS));
        const uint32_t empty0 = peer_addr(smem_u32(&blk_empty[0]), 0);
        uint32_t g = 0;
        SegIter seg(pair, pl);
        int t, kb0, kb1;
        while (seg.next(pl, t, kb0, kb1)) {
            // a stream-K tile cut between pairs: its parts (pairs p_first ..
            // p_first + nparts - 1) and their slots, worked out before the
            // sums occupy the registers.  Pair p > p_first starts its range
            // inside tile ts, so its slot is 2 p; only p_first's depends on
            // where its range began.
            const bool cut = kb0 != 0 || kb1 != pl.NB;
            int p_first = 0, nparts = 0, first_slot = 0, my_slot = 0;
            if (cut) {
                const int ts = t - pl.dp_tiles;
                p_first = pair_of_unit(ts * pl.NB, pl);
                nparts = pair_of_unit((ts + 1) * pl.NB - 1, pl) - p_first + 1;
                first_slot = part_slot(p_first, ts, pl);
                my_slot = part_slot(pair, ts, pl);
            }
            float total[EPI_COLS];
#pragma unroll
            for (int c = 0; c < EPI_COLS; ++c) total[c] = 0.0f;
            for (int kb = kb0; kb < kb1; ++kb, ++g) {
                const uint32_t set = g & 1;
                mbar_wait(smem_u32(&blk_full[set]), (g / 2) & 1, timeout_flag);
                __syncwarp();
                asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
                const uint32_t t_set = tmem + set * ACC_COLS + t_off;
#pragma unroll
                for (int c = 0; c < EPI_COLS; c += 8) {
                    float v[8];
                    tmem_ld8(t_set + c, v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
                    for (int e = 0; e < 8; ++e) total[c + e] += v[e];
                }
                asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty0 + 8u * set);
            }
            bool store = true;
            if (cut) {  // hand over or finish
                float *mine = partials + (static_cast<size_t>(my_slot) * 2 + rank) * SLOT_FLOATS;
#pragma unroll
                for (int c = 0; c < EPI_COLS; c += 4) {
                    const int chunk = (h * (EPI_COLS) + c) / 4;
                    __stcg(reinterpret_cast<float4 *>(mine + (static_cast<size_t>(chunk) * TBM + rloc) * 4),
                           make_float4(total[c], total[c + 1], total[c + 2], total[c + 3]));
                }
                __threadfence();
                epi_bar();
                if (threadIdx.x == 0) {
                    __threadfence();
                    unsigned *cnt = counts + 2 * static_cast<size_t>(t) + rank;
                    const unsigned before = atomicAdd(cnt, 1u);
                    __threadfence();
                    last_part = before == static_cast<unsigned>(nparts - 1) ? 1 : 0;
                }
                epi_bar();
                if (last_part != 0) {
                    // C = the sum of the parts in part order, read back from
                    // the workspace four columns at a time and stored at once
                    // (the running sums of all columns would not fit the
                    // registers beside everything else live here)
                    int tm, tn;
                    pair_tile_coords(t, pl, tm, tn);
                    const int row = tm * PM + static_cast<int>(rank) * TBM + rloc;
                    const int col0 = tn * PN + h * (EPI_COLS);
                    if (row < M && col0 < N) {
                        float *crow = C + static_cast<size_t>(row) * ldc + col0;
                        const int left = N - col0;
                        for (int c = 0; c < EPI_COLS && c < left; c += 4) {
                            const size_t off = (static_cast<size_t>((h * (EPI_COLS) + c) / 4) * TBM + rloc) * 4;
                            float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            for (int k = 0; k < nparts; ++k) {
                                const int sl = k == 0 ? first_slot : 2 * (p_first + k);
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                    partials + (static_cast<size_t>(sl) * 2 + rank) * SLOT_FLOATS + off));
                                sum.x += v.x;
                                sum.y += v.y;
                                sum.z += v.z;
                                sum.w += v.w;
                            }
                            if (vc == 4 && c + 4 <= left) {
                                *reinterpret_cast<float4 *>(crow + c) = sum;
                            } else {
                                const float e4[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (c + e < left) crow[c + e] = e4[e];
                            }
                        }
                    }
                }
                store = false;
            }
            if (store) {
                int tm, tn;
                pair_tile_coords(t, pl, tm, tn);
                const int row = tm * PM + static_cast<int>(rank) * TBM + rloc;
                const int col0 = tn * PN + h * (EPI_COLS);
                if (row < M && col0 < N) {
                    float *crow = C + static_cast<size_t>(row) * ldc + col0;
                    const int left = N - col0;
                    if (vc == 4 && left >= EPI_COLS) {
#pragma unroll
                        for (int e = 0; e < EPI_COLS; e += 4)
                            *reinterpret_cast<float4 *>(crow + e) =
                                make_float4(total[e], total[e + 1], total[e + 2], total[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < EPI_COLS; ++e)
                            if (e < left) crow[e] = total[e];
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    cluster_sync();  // no remote arrive or tensor-memory read of either CTA is still pending
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(TMEM_COLS)
                     : "memory");
    }
}

// ---- host ------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        else
            (void)cudaGetLastError();
    });
    return g_encode;
}

// rows x Kp K-major operand in the workspace: boxes of 32 (K) x 128 (rows)
// with the 128-byte swizzle; out-of-range elements read 0.
bool encode_operand(CUtensorMap &map, const float *base, int rows, int Kp) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dim[2] = {static_cast<cuuint64_t>(Kp), static_cast<cuuint64_t>(rows)};
    const cuuint64_t stride[1] = {static_cast<cuuint64_t>(Kp) * 4};
    const cuuint32_t box[2] = {TBK, TBM};  // 32 K x 128 rows
    const cuuint32_t ones[2] = {1, 1};
    return enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dim, stride, box, ones,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t region_bytes(long long rows, long long Kp) { return (static_cast<size_t>(rows * Kp) * 4 + 255) / 256 * 256; }

// A pair gets at least this many K blocks (MIN_UNITS x 128 K), so that small
// products do not spread thinner than the pipeline can fill.
constexpr int MIN_UNITS = 2;
// Cost of handing a split tile over, in 128-K block-times (fitted to timings
// of 2048^3 .. 8192^3, 16384 x 256 x 4096 and 1024 x 1024 x 8192).
constexpr int SK_FIXUP_BLOCKS = 6;

std::mutex g_setup_mutex;
int g_setup_state[64];
int g_max_pairs[64];
unsigned long long g_setup_ctx[64];  // id of the CUDA context the set-up was made in

// Per device: the architecture check, the shared-memory opt-in and the number
// of CTA pairs that fit on the GPU at once (the persistent grid).
int setup(int dev) {
    if (dev < 0 || dev >= 64) return SGEMM_ERR_DEVICE;
    unsigned long long ctx = 0;
    const bool known = sg_ctx::current_id(dev, &ctx);
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (known && g_setup_state[dev] != 0 && g_setup_ctx[dev] != ctx) g_setup_state[dev] = 0;  // a new context
    if (g_setup_state[dev] == 0) {
        g_setup_ctx[dev] = ctx;
        int major = 0, minor = 0, sms = 0, st = SGEMM_OK;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || major != 10 ||
            minor != 3 || sms < 2 ||
            cudaFuncSetAttribute(sgemm_3xtf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM) !=
                cudaSuccess)
            st = SGEMM_ERR_DEVICE;
        int pairs = sms / 2;
        if (st == SGEMM_OK) {
            cudaLaunchConfig_t cfg;
            memset(&cfg, 0, sizeof cfg);
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 2;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
            cfg.blockDim = dim3(TC_THREADS);
            cfg.dynamicSmemBytes = MMA_SMEM;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, sgemm_3xtf32_kernel, &cfg) == cudaSuccess && clusters > 0)
                pairs = clusters < pairs ? clusters : pairs;
            else
                (void)cudaGetLastError();
        }
        if (st != SGEMM_OK) (void)cudaGetLastError();
        g_max_pairs[dev] = pairs;
        g_setup_state[dev] = st == SGEMM_OK ? 1 : st;
    }
    return g_setup_state[dev] > 0 ? SGEMM_OK : g_setup_state[dev];
}

// Workspace layout: A_hi, A_lo (M x Kp), Bt_hi, Bt_lo (N x Kp), the tile
// counts (2 per pair tile) and the partial-sum slots (2 per pair, 2 halves).
struct WsLayout {
    size_t a_lo, bt_hi, bt_lo, counts, partials, bytes;
};
WsLayout ws_layout(int M, int N, int K, int pairs) {
    const long long Kp = (static_cast<long long>(K) + 3) / 4 * 4;
    const long long T = ((static_cast<long long>(M) + PM - 1) / PM) * ((static_cast<long long>(N) + PN - 1) / PN);
    WsLayout w;
    w.a_lo = region_bytes(M, Kp);
    w.bt_hi = 2 * region_bytes(M, Kp);
    w.bt_lo = w.bt_hi + region_bytes(N, Kp);
    w.counts = w.bt_lo + region_bytes(N, Kp);
    w.partials = w.counts + (static_cast<size_t>(2 * T) * sizeof(unsigned) + 255) / 256 * 256;
    w.bytes = w.partials + static_cast<size_t>(pairs) * 4 * SLOT_FLOATS * sizeof(float);
    return w;
}

// device-side timeout word of the last call, per library instance
__device__ unsigned g_tc_timeout;

// Largest poll limit sgemm_f32_3xtf32_wait_selftest accepts.
constexpr unsigned kSelftestMaxPolls = 1u << 16;

// The pipeline's bounded mbarrier wait on a phase nothing completes (which =
// 0: no arrival) or one already complete (1: after an arrival), with a short
// poll limit; status[0] = 1 if the wait gave up.  One CTA of 32 threads.
__global__ void tc_wait_selftest_kernel(int which, unsigned limit, unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        if (which == 1) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(b) : "memory");
        unsigned gave_up = 0u;
        mbar_wait(b, 0, &gave_up, limit);
        status[0] = gave_up;
    }
}

}  // namespace

extern "C" size_t sgemm_f32_3xtf32_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return ws_layout(M, N, K, sms / 2 > 0 ? sms / 2 : 1).bytes;
}

extern "C" int sgemm_f32_3xtf32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                                int ldc, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_LD;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (K == 0) return sgemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream);  // C = 0
    if (C == nullptr || A == nullptr || B == nullptr) return SGEMM_ERR_NULL_PTR;
    if (workspace == nullptr) return SGEMM_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) % 4 ||
        reinterpret_cast<uintptr_t>(workspace) % 256)
        return SGEMM_ERR_INVALID_ARG;
    if (workspace_bytes < sgemm_f32_3xtf32_workspace_size(M, N, K)) return SGEMM_ERR_INVALID_ARG;
    auto span = [](const void *p, long long bytes) {
        return std::pair<uintptr_t, uintptr_t>(reinterpret_cast<uintptr_t>(p),
                                               reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes));
    };
    auto overl = [](std::pair<uintptr_t, uintptr_t> a, std::pair<uintptr_t, uintptr_t> b) {
        return a.first < b.second && b.first < a.second;
    };
    const auto sa = span(A, 4 * ((static_cast<long long>(M) - 1) * lda + K));
    const auto sb = span(B, 4 * ((static_cast<long long>(K) - 1) * ldb + N));
    const auto sc = span(C, 4 * ((static_cast<long long>(M) - 1) * ldc + N));
    const auto sw = span(workspace, static_cast<long long>(sgemm_f32_3xtf32_workspace_size(M, N, K)));
    if (overl(sc, sa) || overl(sc, sb)) return SGEMM_ERR_ALIAS;
    if (overl(sw, sa) || overl(sw, sb) || overl(sw, sc)) return SGEMM_ERR_ALIAS;
    const long long T = ((static_cast<long long>(M) + PM - 1) / PM) * ((N + PN - 1) / PN);  // pair tiles
    if (2 * T > INT_MAX) return SGEMM_ERR_INVALID_DIM;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    const int st = setup(dev);
    if (st != SGEMM_OK) return st;

    const int Kp = (K + 3) / 4 * 4;
    const WsLayout wl = ws_layout(M, N, K, g_max_pairs[dev]);
    char *ws = static_cast<char *>(workspace);
    float *a_hi = reinterpret_cast<float *>(ws);
    float *a_lo = reinterpret_cast<float *>(ws + wl.a_lo);
    float *bt_hi = reinterpret_cast<float *>(ws + wl.bt_hi);
    float *bt_lo = reinterpret_cast<float *>(ws + wl.bt_lo);
    unsigned *counts = reinterpret_cast<unsigned *>(ws + wl.counts);
    float *partials = reinterpret_cast<float *>(ws + wl.partials);
    TcMaps maps;
    memset(&maps, 0, sizeof maps);
    if (!encode_operand(maps.a_hi, a_hi, M, Kp) || !encode_operand(maps.a_lo, a_lo, M, Kp) ||
        !encode_operand(maps.b_hi, bt_hi, N, Kp) || !encode_operand(maps.b_lo, bt_lo, N, Kp))
        return SGEMM_ERR_DEVICE;

    const int a_blocks = (M + 7) / 8;
    const int b_tiles_k = (Kp + ST - 1) / ST, b_tiles_n = (N + ST - 1) / ST;
    const long long split_blocks = static_cast<long long>(a_blocks) + static_cast<long long>(b_tiles_k) * b_tiles_n;
    if (split_blocks > INT_MAX) return SGEMM_ERR_INVALID_DIM;
    if (cudaMemsetAsync(counts, 0, static_cast<size_t>(2 * T) * sizeof(unsigned), stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    {
        sg_nvtx::Range r("sgemm_f32_3xtf32: split");
        split_kernel<<<static_cast<unsigned>(split_blocks), dim3(32, 8), 0, stream>>>(
            A, lda, B, ldb, M, N, K, Kp, a_hi, a_lo, bt_hi, bt_lo, a_blocks, b_tiles_k);
    }
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    unsigned *timeout = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&timeout), g_tc_timeout) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    SkPlan pl;
    pl.tiles_m = (M + PM - 1) / PM;
    pl.tiles_n = (N + PN - 1) / PN;
    pl.KT = (Kp + TBK - 1) / TBK;
    pl.NB = (pl.KT + KBLK - 1) / KBLK;
    if (T * pl.NB > INT_MAX) return SGEMM_ERR_INVALID_DIM;
    const long long want = (T * pl.NB + MIN_UNITS - 1) / MIN_UNITS;
    pl.P = static_cast<int>(want < g_max_pairs[dev] ? want : g_max_pairs[dev]);
    // Data-parallel takes ceil(T/P) tiles of NB blocks on the longest pair;
    // splitting the partial last wave takes floor(T/P) tiles plus an equal
    // share of the rest, plus the hand-over of split tiles (measured at about
    // SK_FIXUP_BLOCKS block-times).  Pick the shorter.
    const long long waves = T / pl.P, rest = T % pl.P;
    const long long sk_units = rest * pl.NB;
    long long psk = sk_units / MIN_UNITS;
    psk = psk < 1 ? 1 : (psk > pl.P ? pl.P : psk);
    const long long dp_cost = (waves + (rest != 0 ? 1 : 0)) * pl.NB;
    const long long sk_cost = waves * pl.NB + (sk_units + psk - 1) / psk + SK_FIXUP_BLOCKS;
    if (rest == 0 || sk_cost >= dp_cost) {
        pl.dp_tiles = static_cast<int>(T);
        if (T < pl.P) pl.P = static_cast<int>(T);  // one tile per pair, no idle pairs
        pl.Psk = 1;
        pl.U = 0;
    } else {
        pl.dp_tiles = static_cast<int>(waves * pl.P);
        pl.Psk = static_cast<int>(psk);
        pl.U = static_cast<int>(sk_units);
    }
    const int vc = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 4 == 0) ? 4 : 1;
    // programmatic dependent launch: the MMA grid's CTAs may start (barriers,
    // tensor-memory allocation) as the split grid drains
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pl.P));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = MMA_SMEM;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    sg_nvtx::Range r_mma("sgemm_f32_3xtf32: MMA kernel");
    if (cudaLaunchKernelEx(&cfg, sgemm_3xtf32_kernel, maps, C, ldc, M, N, pl, counts, partials, vc, timeout) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

extern "C" int sgemm_f32_3xtf32_timeouts(unsigned *count) {
    if (count == nullptr) return SGEMM_ERR_NULL_PTR;
    if (cudaMemcpyFromSymbol(count, g_tc_timeout, sizeof(unsigned)) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    return SGEMM_OK;
}

extern "C" int sgemm_f32_3xtf32_wait_selftest(int which, unsigned polls, unsigned *timed_out) {
    if (timed_out == nullptr) return SGEMM_ERR_NULL_PTR;
    if (which < 0 || which > 1 || polls == 0 || polls > kSelftestMaxPolls) return SGEMM_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    const int st = setup(dev);
    if (st != SGEMM_OK) return st;
    unsigned *d = nullptr;
    if (cudaMalloc(&d, sizeof(unsigned)) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    int rc = SGEMM_OK;
    if (cudaMemset(d, 0, sizeof(unsigned)) != cudaSuccess) {
        rc = SGEMM_ERR_LAUNCH;
    } else {
        tc_wait_selftest_kernel<<<1, 32>>>(which, polls, d);
        if (cudaGetLastError() != cudaSuccess ||
            cudaMemcpy(timed_out, d, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
            rc = SGEMM_ERR_LAUNCH;
    }
    (void)cudaGetLastError();
    (void)cudaFree(d);
    return rc;
}

// sgemm_f32.cu -- tiled FP32 matrix multiply C = A.B for GB300 (sm_103a),
// and its C ABI (declared in include/sgemm_f32.h).
//
// Data path (vectorised-load page, "这一篇放进 GEMM 路径里看"):
//   global --(cp.async, coalesced, 16/8/4-byte by alignment class)-->
//   shared (k-major swizzled A tile, row-major B tile, STAGES-deep ring) -->
//   registers (two 128-bit reads of A and two of B per k) -->
//   8 x 8 register tile of FP32 FMAs --> guarded, vectorised stores of C.
//
// * Tiling: a CTA computes a BM x BN = 128 x 128 tile of C, walking K in
//   BK = 16 slices (shared-memory page, "register tiling 在干什么": each value
//   read from shared memory feeds 8 FMAs, (8+8)/64 = 0.25 reads per FMA).
// * Warp-level reuse: the 32 lanes of a warp form a 4 x 8 grid over a
//   32 x 64 warp tile; the 8 lanes of a row read the same A group (one word
//   per bank, broadcast) and the 4 lanes of a column the same B group
//   ("广播不是 bank conflict").
// * Transpose on store: A (row-major, k contiguous) is written k-major so a
//   thread's 4 consecutive rows are one 128-bit read ("shared memory transpose
//   的基本想法"); a 16-byte copy cannot split a vector across rows, so A moves
//   in 4-byte copies, spread over banks by the XOR swizzle in smem_layout.cuh.
// * Edges ("边界处理会破坏漂亮形状"): copies past M, N or K are issued with a
//   zero source size, which fills shared memory with 0; stores are guarded.
//   Misaligned leading dimensions ("对齐也要从数据分配开始") select 8- or
//   4-byte B copies and C stores instead of 16-byte ones.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "ctx_key.cuh"
#include "nvtx_range.cuh"
#include "sgemm_f32.h"
#include "smem_layout.cuh"
#include "transpose_f32.h"

namespace {

using namespace sg;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async with an explicit source size: bytes beyond `src_bytes` are
// written as zero in shared memory and not read from global memory.
template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const float *src, uint32_t src_bytes) {
    if constexpr (BYTES == 16) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    } else if constexpr (BYTES == 8) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    } else {
        static_assert(BYTES == 4, "copy width");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int PENDING>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(PENDING) : "memory");
}

// ---- mbarrier and tensor-memory-access (TMA) copies ---------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Polls one mbarrier phase at most `limit` times; a wait that runs out sets
// *timeout_flag to 1 and returns.
__device__ __forceinline__ void mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t limit,
                                                  unsigned *timeout_flag) {
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++polls > limit) {
            *timeout_flag = 1u;
            break;
        }
    }
}
// 2-D tiled bulk copy global -> shared; elements outside the tensor read 0.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Polls of one mbarrier phase before a wait is abandoned (each try_wait
// itself blocks for a while): far beyond any copy's latency.
constexpr uint32_t kWaitLimit = 1u << 22;
// Largest poll limit sgemm_f32_wait_selftest accepts (keeps the test short).
constexpr unsigned kSelftestMaxPolls = 1u << 16;
// Set to 1 by a CTA whose copy wait ran out (the result is then wrong; the
// kernel still finishes).  Stays set until the process exits.
__device__ unsigned g_copy_timeout;

// Global memory descriptions of A (dims K x M, box 16 x 128, 64-byte
// swizzle: the layout of the raw A tile) and B (dims N x K, box 128 x 16, no
// swizzle: the layout of the B tile).
struct Maps {
    CUtensorMap a, b;
};

struct Problem {
    int M, N, K;
    const float *__restrict__ A;
    int lda;
    const float *__restrict__ B;
    int ldb;
    float *__restrict__ C;
    int ldc;
    int tiles_m, tiles_n;
    int vc;  // C store width in floats (4, 2 or 1)
};

// The 8 x 8 register tile, held as 32 column pairs for the packed FP32 FMA
// (fma.rn.f32x2): c[r][j] = (acc[r][2j], acc[r][2j+1]) += (a_r, a_r) * (b_2j, b_2j+1).
// The B pairs are natural register pairs of the 128-bit fragment reads and
// a_r is used twice: 32 packed FMAs per k step, issued column pair by column
// pair so that consecutive ones share their B operand.
struct Acc {
    float2 c[TM][TN / 2];
};

__device__ __forceinline__ void acc_zero(Acc &acc) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc.c[i][j] = make_float2(0.0f, 0.0f);
}

// threadIdx.x, read afresh at each call: the compiler can neither keep it
// live across a loop nor merge two reads.
__device__ __forceinline__ int tid_fresh() {
    int t;
    asm volatile("mov.u32 %0, %%tid.x;\n" : "=r"(t));
    return t;
}

// Accumulates the product of the CTA's C tile (m0, n0) over K tiles
// [kt0, kt1) into acc.  VA = A copy width in floats (4 or 1), VB = B copy
// width in floats (4, 2 or 1), chosen on the host from alignment; with TMA
// (both 4) one thread moves each tile by two tensor copies instead.
//
// `pipe` counts the tiles this CTA has loaded before this range: load u goes
// to ring stage u % STAGES (its mbarrier completes phase u / STAGES) and is
// transposed into As buffer u % 2.
//
// Pipeline (one __syncthreads per K tile): at iteration kt
//   1. wait until tile kt+1 has landed (own cp.async copies, or the stage's
//      mbarrier), then barrier: tile kt+1's raw A and B, and the transposed
//      As of tile kt, are visible to all; every thread has finished tile kt-1;
//   2. issue the copies of tile kt+STAGES-1 into the stage tile kt-1 used;
//   3. transpose tile kt+1's raw A into the As buffer tile kt-1 used;
//   4. 16 k steps of fragment reads and packed FMAs on tile kt.
// On return every copy has landed; the caller must __syncthreads() before
// starting another range (other threads may still read shared memory).
//
// The tile origin (m0, n0) is read from shared memory (`org`, written before
// a barrier the whole CTA passed) and the copy coordinates from a fresh read
// of the thread index at each copy issue, so neither is held in registers
// through the K loop: with 64 accumulators in a 128-register budget the
// narrow-copy variants have no room to keep them.
template <int VA, int VB, bool TMA>
__device__ __forceinline__ void mma_k_range(const Problem &p, const Maps &maps, const int2 *org, const int kt0,
                                            const int kt1, uint32_t &pipe, float *smem, const uint32_t bars,
                                            Acc &acc) {
    static_assert(!TMA || (VA == 4 && VB == 4), "tensor copies need 16-byte aligned rows");
    constexpr uint32_t RING = STAGES;
    const int tid = threadIdx.x;
    const int K = p.K, M = p.M, N = p.N;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t u0 = pipe - static_cast<uint32_t>(kt0);  // load index of tile kt is u0 + kt

    // Copies: A (global -> raw staging tile) and B (global -> row-major tile).
    // Rows past M and columns past K or N are zero-filled by a zero or short
    // source size ("边界处理会破坏漂亮形状").
    constexpr int NA = VA == 4 ? A_COPIES16 : A_COPIES4;
    constexpr int NB = b_copies<VB>();

    auto issue_tile = [&](int kt) {
        const uint32_t stage = (u0 + kt) % RING;
        const int kb = kt * BK;
        const int2 o = *org;  // (m0, n0)
        if constexpr (TMA) {
            if (tid == 0) {
                const uint32_t bar = bars + 8 * stage;
                mbar_expect_tx(bar, STAGE_FLOATS * 4);
                tma_load_2d(sbase + ar_word(stage, 0, 0) * 4, &maps.a, kb, o.x, bar);
                tma_load_2d(sbase + bs_word(stage, 0, 0) * 4, &maps.b, o.y, kb, bar);
            }
        } else {
            const int t = tid_fresh();
#pragma unroll
            for (int q = 0; q < NA; ++q) {
                int m, k;
                if constexpr (VA == 4) a_copy16_coord(t, q, m, k);
                else a_copy4_coord(t, q, m, k);
                const int kg = kb + k;
                const int left = K - kg;  // valid floats from kg on
                const uint32_t bytes = (o.x + m < M && left > 0) ? (left >= VA ? VA * 4u : left * 4u) : 0u;
                const float *src = bytes ? p.A + (static_cast<size_t>(o.x + m) * p.lda + kg) : p.A;
                cp_async<VA * 4>(sbase + ar_word(stage, m, k) * 4, src, bytes);
            }
#pragma unroll
            for (int q = 0; q < NB; ++q) {
                int k, n;
                b_copy_coord<VB>(t, q, k, n);
                const int kg = kb + k;
                const int valid = N - (o.y + n);  // valid floats from column o.y + n on
                const uint32_t bytes =
                    kg < K && valid > 0 ? (valid >= VB ? VB * 4u : static_cast<uint32_t>(valid) * 4u) : 0u;
                const float *src = bytes ? p.B + (static_cast<size_t>(kg) * p.ldb + (o.y + n)) : p.B;
                cp_async<VB * 4>(sbase + bs_word(stage, k, n) * 4, src, bytes);
            }
            cp_async_commit();
        }
    };
    // Waits until tile kt's copies are visible to this thread.  cp.async:
    // PENDING later groups may stay in flight.  TMA: the stage's mbarrier
    // phase; a wait that runs out records g_copy_timeout and goes on.
    auto wait_tile = [&](int kt, auto pending) {
        if constexpr (TMA) {
            const uint32_t u = u0 + kt;
            mbar_wait_bounded(bars + 8 * (u % RING), (u / RING) & 1u, kWaitLimit, &g_copy_timeout);
        } else {
            cp_async_wait<decltype(pending)::value>();
        }
    };
    using Pending1 = std::integral_constant<int, STAGES - 2>;
    using Pending2 = std::integral_constant<int, STAGES - 3>;

    // ---- A transpose: raw staging tile -> k-major As buffer
    auto transpose_tile = [&](int kt) {
        const uint32_t stage = (u0 + kt) % STAGES;
        const int buf = (u0 + kt) & 1;
#pragma unroll
        for (int f = 0; f < A_VECS; ++f) {
            int k, m;
            a_xpose_coord(tid, f, k, m);
            const float4 v = *reinterpret_cast<const float4 *>(smem + ar_word(stage, m, k));
            smem[as_word(buf, k + 0, m)] = v.x;
            smem[as_word(buf, k + 1, m)] = v.y;
            smem[as_word(buf, k + 2, m)] = v.z;
            smem[as_word(buf, k + 3, m)] = v.w;
        }
    };

    // prologue: tiles kt0 .. kt0+STAGES-2 in flight, tile kt0 transposed
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (kt0 + s < kt1) issue_tile(kt0 + s);
        else if (!TMA) cp_async_commit();  // keep one cp.async group per slot
    }
    if (kt0 < kt1) {
        wait_tile(kt0, Pending1{});
        __syncthreads();
        transpose_tile(kt0);
    }

    for (int kt = kt0; kt < kt1; ++kt) {
        if (!TMA || kt + 1 < kt1) wait_tile(kt + 1, Pending2{});
        __syncthreads();
        if (kt + STAGES - 1 < kt1) issue_tile(kt + STAGES - 1);
        else if (!TMA) cp_async_commit();
        if (kt + 1 < kt1) transpose_tile(kt + 1);

        const uint32_t stage = (u0 + kt) % STAGES;
        const int buf = (u0 + kt) & 1;
        // fragment offsets: from a fresh thread index in the narrow-copy
        // variants (no room to keep them), else from tid
        const int tf = TMA ? tid : tid_fresh();
        const int ra = frag_row0(tf), cb = frag_col0(tf);
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(smem + as_word(buf, k, ra));
            const float4 a1 = *reinterpret_cast<const float4 *>(smem + as_word(buf, k, ra + 16));
            const float4 b0 = *reinterpret_cast<const float4 *>(smem + bs_word(stage, k, cb));
            const float4 b1 = *reinterpret_cast<const float4 *>(smem + bs_word(stage, k, cb + 32));
            const float a[TM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float2 bp[TN / 2] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                       make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
            // column pair outermost: consecutive packed FMAs share the B register
            // pair, so each reads only its A value and its accumulator pair
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) {
#pragma unroll
                for (int r = 0; r < TM; ++r) acc.c[r][j] = __ffma2_rn(make_float2(a[r], a[r]), bp[j], acc.c[r][j]);
            }
        }
    }
    if (!TMA) cp_async_wait<0>();
    pipe += static_cast<uint32_t>(kt1 > kt0 ? kt1 - kt0 : 0);
}

// 1024-byte aligned start of the dynamic shared memory block, and the
// mbarriers of the copy ring (initialised once per CTA).
__device__ __forceinline__ float *aligned_smem(float *raw) {
    const uint32_t s = smem_u32(raw);
    return raw + ((SMEM_ALIGN - (s & (SMEM_ALIGN - 1))) & (SMEM_ALIGN - 1)) / 4;
}
constexpr int kMaxRing = STAGES_AT > STAGES ? STAGES_AT : STAGES;
template <bool TMA>
__device__ __forceinline__ void init_bars(uint32_t bars) {
    if (TMA) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < kMaxRing; ++s) mbar_init(bars + 8 * s, 1);
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        }
        __syncthreads();
    }
}

// init_bars, and thread 0 publishes the CTA's tile origin (m0, n0) in `org`
// for mma_k_range; the barrier makes both visible to the CTA.
template <bool TMA>
__device__ __forceinline__ void init_cta(uint32_t bars, int2 *org, int m0, int n0) {
    if (threadIdx.x == 0) {
        if (TMA) {
            for (int s = 0; s < kMaxRing; ++s) mbar_init(bars + 8 * s, 1);
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        }
        *org = make_int2(m0, n0);
    }
    __syncthreads();
}

// Writes the register tile to C tile (m0, n0) with guarded stores,
// vectorised where C's alignment class allows.  With ADD_PARTIAL, the value
// already in C (a partial sum left there by another CTA) is read back from
// L2 and added first: final = this CTA's sum + the other part.
template <bool ADD_PARTIAL>
__device__ __forceinline__ void store_tile(const Problem &p, const int m0, const int n0, const Acc &acc) {
    const int tid = threadIdx.x;
    const int cb = frag_col0(tid);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + frag_row(tid, i);
        if (row >= p.M) continue;
        float *crow = p.C + static_cast<size_t>(row) * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + cb + 32 * h;
            float v[4] = {acc.c[i][2 * h].x, acc.c[i][2 * h].y, acc.c[i][2 * h + 1].x, acc.c[i][2 * h + 1].y};
            if (col + 3 < p.N && p.vc == 4) {
                if (ADD_PARTIAL) {
                    const float4 o = __ldcg(reinterpret_cast<const float4 *>(crow + col));
                    v[0] += o.x; v[1] += o.y; v[2] += o.z; v[3] += o.w;
                }
                *reinterpret_cast<float4 *>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else if (col + 3 < p.N && p.vc == 2) {
                if (ADD_PARTIAL) {
                    const float2 o0 = __ldcg(reinterpret_cast<const float2 *>(crow + col));
                    const float2 o1 = __ldcg(reinterpret_cast<const float2 *>(crow + col + 2));
                    v[0] += o0.x; v[1] += o0.y; v[2] += o1.x; v[3] += o1.y;
                }
                *reinterpret_cast<float2 *>(crow + col) = make_float2(v[0], v[1]);
                *reinterpret_cast<float2 *>(crow + col + 2) = make_float2(v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < p.N) crow[col + e] = ADD_PARTIAL ? v[e] + __ldcg(crow + col + e) : v[e];
            }
        }
    }
}

// Data-parallel schedule: one CTA per C tile, the whole K range.
template <int VA, int VB, bool TMA>
__global__ void __launch_bounds__(NT, 2) sgemm_f32_tiled_kernel(const Problem p, const __grid_constant__ Maps maps) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    // a split-tail grid queued behind this one may start as SMs free up: it
    // writes other tiles and reads nothing this grid writes
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    __shared__ int2 org;
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    int tm, tn;
    tile_of(blockIdx.x, p.tiles_m, p.tiles_n, tm, tn);
    init_cta<TMA>(bars, &org, tm * BM, tn * BN);
    Acc acc;
    acc_zero(acc);
    uint32_t pipe = 0;
    mma_k_range<VA, VB, TMA>(p, maps, &org, 0, (p.K + BK - 1) / BK, pipe, smem, bars, acc);
    store_tile<false>(p, org.x, org.y, acc);
}

// ---- cluster split of K ----------------------------------------------------
// For products with few tiles (at most half the CTAs the GPU holds at once) a
// cluster of S CTAs (2 <= S <= 8) computes one tile of C: CTA r of the
// cluster accumulates K tiles [KT r / S, KT (r+1) / S) with the 8 x 8
// kernels' main loop, leaves its partial sums in its own shared memory (the
// ring's space, pt_word layout), and after a cluster barrier sums rows
// [128 r / S, 128 (r+1) / S) of the tile over the S CTAs' shared memory
// (distributed shared memory, in rank order, so the result does not depend
// on timing) and stores them to C.  A second cluster barrier keeps every
// CTA's shared memory alive until its peers have read it.  No workspace, no
// flags and no wait between CTAs other than the hardware's cluster barrier.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(n));
    return n;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The address of shared-memory address `addr` of this CTA in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
// Stores 4 consecutive values of row `row` of C from column `col` on,
// guarded by M and N, with the widest stores C's alignment class allows.
__device__ __forceinline__ void store_c4(const Problem &p, const int row, const int col, const float4 v) {
    if (row >= p.M || col >= p.N) return;
    float *c = p.C + static_cast<size_t>(row) * p.ldc + col;
    if (col + 3 < p.N && p.vc == 4) {
        *reinterpret_cast<float4 *>(c) = v;
    } else if (col + 3 < p.N && p.vc == 2) {
        *reinterpret_cast<float2 *>(c) = make_float2(v.x, v.y);
        *reinterpret_cast<float2 *>(c + 2) = make_float2(v.z, v.w);
    } else {
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (col + i < p.N) c[i] = e[i];
    }
}

template <int VA, int VB, bool TMA>
__global__ void __launch_bounds__(NT, 2) sgemm_f32_clusterk_kernel(const Problem p, const __grid_constant__ Maps maps) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    __shared__ int2 org;
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    int k0, k1;
    {
        const int S = static_cast<int>(cluster_nctarank());
        const int rank = static_cast<int>(cluster_ctarank());
        int tm, tn;
        tile_of(static_cast<int>(blockIdx.x) / S, p.tiles_m, p.tiles_n, tm, tn);
        init_cta<TMA>(bars, &org, tm * BM, tn * BN);
        const int KT = (p.K + BK - 1) / BK;
        k0 = static_cast<int>(static_cast<long long>(KT) * rank / S);
        k1 = static_cast<int>(static_cast<long long>(KT) * (rank + 1) / S);
    }
    Acc acc;
    acc_zero(acc);
    uint32_t pipe = 0;
    mma_k_range<VA, VB, TMA>(p, maps, &org, k0, k1, pipe, smem, bars, acc);
    __syncthreads();  // every thread is done with the ring: its space becomes the partial tile
    // the cluster shape is read again here rather than kept through the K loop
    const int S = static_cast<int>(cluster_nctarank());
    const int rank = static_cast<int>(cluster_ctarank());
    const int tid = threadIdx.x;
#pragma unroll
    for (int q = 0; q < 2 * TM; ++q) {
        int row, col;
        pt_store_coord(tid, q, row, col);
        const int i = q >> 1, h = q & 1;
        *reinterpret_cast<float4 *>(smem + pt_word(row, col)) =
            make_float4(acc.c[i][2 * h].x, acc.c[i][2 * h].y, acc.c[i][2 * h + 1].x, acc.c[i][2 * h + 1].y);
    }
    cluster_barrier();  // every CTA's partial tile is complete and visible to the cluster
    // this CTA sums rows [r0, r1) of the tile
    const int r0 = BM * rank / S, r1 = BM * (rank + 1) / S;
    const uint32_t base = smem_u32(smem);
    for (int j = 0;; ++j) {
        int row, col;
        pt_sum_coord(tid, j, r0, row, col);
        if (row >= r1) break;
        const uint32_t addr = base + static_cast<uint32_t>(pt_word(row, col)) * 4u;
        float4 sum = ld_dsmem_f4(map_peer(addr, 0));
        for (int q = 1; q < S; ++q) {
            const float4 v = ld_dsmem_f4(map_peer(addr, static_cast<uint32_t>(q)));
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
        }
        store_c4(p, org.x + row, org.y + col, sum);
    }
    cluster_barrier();  // no CTA leaves while a peer may still read its shared memory
}

// ---- k-major kernels with 8 x 16 register tiles --------------------------
// The one-CTA-per-tile and split-tail kernels of the k-major path: 128
// threads (2 x 2 warps of 64 x 64), each holding an 8 x 16 register tile,
// so that a k step reads 2 + 4 fragments of 128 bits for 64 packed FMAs
// (0.09 reads per FMA instead of 0.125 with 8 x 8).  Measured on GB300 with
// the same ring and copies: 3072x4864x4096 1745 -> 1695 us, 8192^3 one CTA
// per tile 15462 -> 14953 us against the 8 x 8 tiles; results bit for bit
// the same (each output is the same FMA chain over k).
struct Acc16 {
    float2 c[TM][TN16 / 2];  // (acc[r][2j], acc[r][2j+1]) as in Acc
};

__device__ __forceinline__ void acc16_zero(Acc16 &acc) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN16 / 2; ++j) acc.c[i][j] = make_float2(0.0f, 0.0f);
}

// Accumulates the product of C tile (m0, n0) over K tiles [kt0, kt1) into
// acc, with A given as its k-major copy At (K x M; maps.a describes it) and
// K tiles BK_AT deep.  Each stage of a STAGES_AT-deep ring receives a
// BK_AT x 128 box of At and a BK_AT x 128 box of B by tensor copy,
// completing on the stage's mbarrier.  Iteration kt waits for tile kt, then a
// barrier (every thread has finished tile kt-1, whose stage is free), issues
// tile kt + STAGES_AT - 1 into that stage and runs BK_AT k steps.  `pipe`
// counts the tiles this CTA has loaded before this range (load u goes to
// stage u % STAGES_AT, whose mbarrier completes phase u / STAGES_AT), as in
// mma_k_range.
// With DRAIN (a diagnostic kernel, never dispatched by default) one tile is in
// flight at a time, issued after the k steps of the one before: no copy
// writes shared memory while the fragments are read.
template <bool DRAIN = false>
__device__ __forceinline__ void kmajor16_k_range(const Maps &maps, const int m0, const int n0, const int kt0,
                                                 const int kt1, uint32_t &pipe, float *smem, const uint32_t bars,
                                                 Acc16 &acc) {
    const int tid = threadIdx.x;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t u0 = pipe - static_cast<uint32_t>(kt0);
    auto issue_tile = [&](int kt) {
        if (tid == 0) {
            const uint32_t stage = (u0 + kt) % STAGES_AT;
            const uint32_t bar = bars + 8 * stage;
            mbar_expect_tx(bar, AT_STAGE_FLOATS * 4);
            tma_load_2d(sbase + at_word(stage, 0, 0) * 4, &maps.a, m0, kt * BK_AT, bar);
            tma_load_2d(sbase + atb_word(stage, 0, 0) * 4, &maps.b, n0, kt * BK_AT, bar);
        }
    };
    const int ra = frag16_row0(tid);
    const int cb = frag16_col0(tid);
    if constexpr (DRAIN) {
        if (kt0 < kt1) issue_tile(kt0);
    } else {
#pragma unroll
        for (int s = 0; s < STAGES_AT - 1; ++s)
            if (kt0 + s < kt1) issue_tile(kt0 + s);
    }
    for (int kt = kt0; kt < kt1; ++kt) {
        const uint32_t u = u0 + kt;
        mbar_wait_bounded(bars + 8 * (u % STAGES_AT), (u / STAGES_AT) & 1u, kWaitLimit, &g_copy_timeout);
        __syncthreads();
        if (!DRAIN && kt + STAGES_AT - 1 < kt1) issue_tile(kt + STAGES_AT - 1);
        const uint32_t stage = u % STAGES_AT;
#pragma unroll
        for (int k = 0; k < BK_AT; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(smem + at_word(stage, k, ra));
            const float4 a1 = *reinterpret_cast<const float4 *>(smem + at_word(stage, k, ra + 32));
            const float a[TM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float2 bp[TN16 / 2];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 b = *reinterpret_cast<const float4 *>(smem + atb_word(stage, k, cb + 16 * g));
                bp[2 * g] = make_float2(b.x, b.y);
                bp[2 * g + 1] = make_float2(b.z, b.w);
            }
            // column pair outermost, as in mma_k_range
#pragma unroll
            for (int j = 0; j < TN16 / 2; ++j) {
#pragma unroll
                for (int r = 0; r < TM; ++r) acc.c[r][j] = __ffma2_rn(make_float2(a[r], a[r]), bp[j], acc.c[r][j]);
            }
        }
        if constexpr (DRAIN) {
            __syncthreads();  // every thread is done with this stage before the next copy lands
            if (kt + 1 < kt1) issue_tile(kt + 1);
        }
    }
    pipe += static_cast<uint32_t>(kt1 > kt0 ? kt1 - kt0 : 0);
}

// store_tile for the 8 x 16 register tile: row i of the thread's tile, its
// 16 columns as 4 groups of 4 (guarded, vectorised by C's class).  With
// ADD_PARTIAL the value already in C is read back from L2 and added first.
template <bool ADD_PARTIAL>
__device__ __forceinline__ void store_tile16(const Problem &p, const int m0, const int n0, const Acc16 &acc) {
    const int tid = threadIdx.x;
    const int cb = frag16_col0(tid);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + frag16_row(tid, i);
        if (row >= p.M) continue;
        float *crow = p.C + static_cast<size_t>(row) * p.ldc;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int col = n0 + cb + 16 * g;
            float v[4] = {acc.c[i][2 * g].x, acc.c[i][2 * g].y, acc.c[i][2 * g + 1].x, acc.c[i][2 * g + 1].y};
            if (col + 3 < p.N && p.vc == 4) {
                if (ADD_PARTIAL) {
                    const float4 o = __ldcg(reinterpret_cast<const float4 *>(crow + col));
                    v[0] += o.x; v[1] += o.y; v[2] += o.z; v[3] += o.w;
                }
                *reinterpret_cast<float4 *>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else if (col + 3 < p.N && p.vc == 2) {
                if (ADD_PARTIAL) {
                    const float2 o0 = __ldcg(reinterpret_cast<const float2 *>(crow + col));
                    const float2 o1 = __ldcg(reinterpret_cast<const float2 *>(crow + col + 2));
                    v[0] += o0.x; v[1] += o0.y; v[2] += o1.x; v[3] += o1.y;
                }
                *reinterpret_cast<float2 *>(crow + col) = make_float2(v[0], v[1]);
                *reinterpret_cast<float2 *>(crow + col + 2) = make_float2(v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < p.N) crow[col + e] = ADD_PARTIAL ? v[e] + __ldcg(crow + col + e) : v[e];
            }
        }
    }
}
// Partial sums of the 8 x 16 tiles, one 128 x 128 slot per CTA: thread t's
// 32 float4 go to floats 4 * (q * NT16 + t), q = 0..31, so each warp store
// covers 512 contiguous bytes.
__device__ __forceinline__ void store_partial16(float *slot, const Acc16 &acc) {
#pragma unroll
    for (int q = 0; q < TM * TN16 / 4; ++q) {
        const float2 lo = acc.c[q >> 2][2 * (q & 3)], hi = acc.c[q >> 2][2 * (q & 3) + 1];
        *reinterpret_cast<float4 *>(slot + 4 * (q * NT16 + threadIdx.x)) = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
}
__device__ __forceinline__ void add_partial16(const float *slot, Acc16 &acc) {
#pragma unroll
    for (int q = 0; q < TM * TN16 / 4; ++q) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(slot + 4 * (q * NT16 + threadIdx.x)));
        float2 &lo = acc.c[q >> 2][2 * (q & 3)], &hi = acc.c[q >> 2][2 * (q & 3) + 1];
        lo.x += v.x; lo.y += v.y; hi.x += v.z; hi.y += v.w;
    }
}

// Data-parallel schedule on the k-major copy of A: one CTA per C tile.  The
// DRAIN instantiation is the drained-ring diagnostic (see kmajor16_k_range).
template <bool DRAIN = false>
__global__ void __launch_bounds__(NT16, 2) sgemm_f32_kmajor_kernel(const Problem p, const __grid_constant__ Maps maps) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    // a split-tail grid queued behind this one may start as SMs free up
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    init_bars<true>(bars);
    int tm, tn;
    tile_of(blockIdx.x, p.tiles_m, p.tiles_n, tm, tn);
    Acc16 acc;
    acc16_zero(acc);
    uint32_t pipe = 0;
    kmajor16_k_range<DRAIN>(maps, tm * BM, tn * BN, 0, (p.K + BK_AT - 1) / BK_AT, pipe, smem, bars, acc);
    store_tile16<false>(p, tm * BM, tn * BN, acc);
}

// ---- flags between CTAs (stream-K fix-up) ------------------------------
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
constexpr unsigned kSpinLimit = 1u << 24;  // x ~64 ns sleeps: about a second, then give up

// Partial sums of a split tile, one 128 x 128 slot per CTA: thread t's 16
// float4 go to floats 4 * (q * NT + t), q = 0..15, so each warp store
// covers 512 contiguous bytes.
__device__ __forceinline__ void store_partial(float *slot, const Acc &acc) {
#pragma unroll
    for (int q = 0; q < TM * TN / 4; ++q) {
        const float2 lo = acc.c[q >> 1][2 * (q & 1)], hi = acc.c[q >> 1][2 * (q & 1) + 1];
        *reinterpret_cast<float4 *>(slot + 4 * (q * NT + threadIdx.x)) = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
}
// (at most 4 loads in flight: with the 64 accumulators live, loading all 16
// first would not fit the 128-register budget)
__device__ __forceinline__ void add_partial(const float *slot, Acc &acc) {
#pragma unroll
    for (int q = 0; q < TM * TN / 4; ++q) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(slot + 4 * (q * NT + threadIdx.x)));
        float2 &lo = acc.c[q >> 1][2 * (q & 1)], &hi = acc.c[q >> 1][2 * (q & 1) + 1];
        lo.x += v.x; lo.y += v.y; hi.x += v.z; hi.y += v.w;
        if ((q & 3) == 3) asm volatile("" ::: "memory");
    }
}
// Thread 0 waits for a flag raised by another CTA; a wait longer than
// `limit` polls sets bit 0 of *error and gives up (wrong result, no hang).
__device__ __forceinline__ void wait_flag(const unsigned *flag, unsigned *error, unsigned limit = kSpinLimit) {
    if (threadIdx.x == 0) {
        unsigned spins = 0;
        while (ld_acquire(flag) == 0u) {
            if (++spins > limit) {
                atomicOr(error, 1u);
                break;
            }
            __nanosleep(64);
        }
    }
    __syncthreads();
}
__device__ __forceinline__ void raise_flag(unsigned *flag) {
    __syncthreads();  // every thread's partial stores are issued
    if (threadIdx.x == 0) {
        __threadfence();
        st_release(flag, 1u);
    }
}

// The segments of one CTA of the stream-K schedules (below): first whole
// data-parallel tiles (tile c, c + G, ...), then its share of the (tile,
// K tile) iterations of the remaining tiles, cut at tile boundaries.  K tiles
// are bk deep (BK, or BK_AT for the k-major kernels).  The walk lives in
// shared memory, one per CTA, and only thread 0 advances it, between the
// barriers that already separate segments: in registers its 64-bit positions
// would stay live through the K loop, where the 8 x 8 kernels have none to
// spare.
struct SkWalk {
    long long it, it_end;  // this CTA's stream-K iterations not yet taken: [it, it_end)
    int dp_lin;            // its next data-parallel tile
    int lin, k0, k1;       // the current segment: tile lin, K tiles [k0, k1)
    int last;              // the last CTA holding a part of tile lin (see sk_last_part)
    int more;              // 0 once the CTA is done
    int2 org;              // the segment's tile origin (m0, n0)
    int KT;                // K tiles per tile
    unsigned pipe;         // K tiles this CTA loaded before the segment (see mma_k_range)
};
// Stream-K iterations (tile, K tile) after the dp_tiles data-parallel tiles.
__device__ __forceinline__ long long sk_total(const Problem &p, int dp_tiles, int KT) {
    return static_cast<long long>(p.tiles_m * p.tiles_n - dp_tiles) * KT;
}
// Thread 0 only: this CTA's range, CTA c of G taking iterations
// [total c / G, total (c+1) / G) after the data-parallel ones.
__device__ __forceinline__ void sk_begin(SkWalk &w, const Problem &p, int dp_tiles, int KT) {
    const long long total = sk_total(p, dp_tiles, KT), base = static_cast<long long>(dp_tiles) * KT;
    w.it = base + total * blockIdx.x / gridDim.x;
    w.it_end = base + total * (blockIdx.x + 1) / gridDim.x;
    w.dp_lin = blockIdx.x;
    w.KT = KT;
    w.k0 = w.k1 = 0;
    w.pipe = 0u;
}
// The last CTA holding a part of tile lin: the owner adds the parts of CTAs
// blockIdx.x + 1 .. sk_last_part(lin).
__device__ __forceinline__ int sk_last_part(const Problem &p, int dp_tiles, int KT, int lin) {
    const long long total = sk_total(p, dp_tiles, KT);
    const long long last = static_cast<long long>(lin + 1) * KT - 1 - static_cast<long long>(dp_tiles) * KT;
    return static_cast<int>(((last + 1) * gridDim.x + total - 1) / total - 1);
}
// Thread 0 only: the next segment (whole data-parallel tiles first, then the
// range cut at tile boundaries), or more = 0 when the CTA is done.
__device__ __forceinline__ void sk_next(SkWalk &w, const Problem &p, int dp_tiles) {
    const int KT = w.KT;
    w.pipe += static_cast<unsigned>(w.k1 - w.k0);  // the segment just finished
    int lin, k0, k1;
    if (w.dp_lin < dp_tiles) {
        lin = w.dp_lin;
        k0 = 0;
        k1 = KT;
        w.dp_lin += gridDim.x;
    } else if (w.it < w.it_end) {
        lin = static_cast<int>(w.it / KT);
        k0 = static_cast<int>(w.it % KT);
        k1 = static_cast<int>(k0 + (w.it_end - w.it) < KT ? k0 + (w.it_end - w.it) : KT);
        w.it += k1 - k0;
    } else {
        w.more = 0;
        return;
    }
    int tm, tn;
    tile_of(lin, p.tiles_m, p.tiles_n, tm, tn);
    w.lin = lin;
    w.k0 = k0;
    w.k1 = k1;
    w.last = lin >= dp_tiles ? sk_last_part(p, dp_tiles, KT, lin) : static_cast<int>(blockIdx.x);
    w.org = make_int2(tm * BM, tn * BN);
    w.more = 1;
}

// Stream-K schedule.  A persistent, co-resident grid of G CTAs first computes
// tiles 0 .. dp_tiles-1 one whole tile at a time (tile c, c+G, ...: CTAs
// running together work on neighbouring tiles, which keeps A and B panels in
// L2), then splits the (tile, K tile) iterations of the remaining tiles into
// G equal contiguous ranges, so every CTA ends with the same amount of FMA
// work.  A tile cut by range boundaries is finished by the CTA holding its
// K = 0 part (the owner, whose last segment it is); every other CTA holding a
// part of it starts its range there and hands its partial sums over first:
//   * partials == nullptr (more remaining tiles than CTAs, so every range is
//     longer than a tile and a tile has at most two parts): the other CTA
//     stores its partial sums into the tile of C itself and raises
//     flags[tile]; the owner adds that tile of C to its sums.
//   * partials != nullptr (any number of parts): CTA c writes its partial
//     sums to slot c of `partials` and raises flags[c]; the owner adds the
//     slots of the following CTAs in CTA order.
// Every hand-over comes first in its CTA's range, so no wait can form a
// cycle, and the order of the additions is fixed: results are deterministic.
// A wait longer than kSpinLimit polls sets bit 0 of the word after the flags
// and stores without that part: a wrong result, never a hang.
template <int VA, int VB, bool TMA>
__global__ void __launch_bounds__(NT, 2)
sgemm_f32_streamk_kernel(const Problem p, const __grid_constant__ Maps maps, const int dp_tiles, unsigned *flags,
                         float *partials) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    __shared__ SkWalk w;  // advanced by thread 0 between barriers
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    init_bars<TMA>(bars);
    if (threadIdx.x == 0) sk_begin(w, p, dp_tiles, (p.K + BK - 1) / BK);
    // One loop over segments (whole data-parallel tiles first, then this CTA's
    // stream-K range cut at tile boundaries), so the main loop is inlined once.
    for (;;) {
        if (threadIdx.x == 0) sk_next(w, p, dp_tiles);
        __syncthreads();  // the segment is visible to the CTA
        if (!w.more) break;
        Acc acc;
        acc_zero(acc);
        uint32_t pipe = w.pipe;
        mma_k_range<VA, VB, TMA>(p, maps, &w.org, w.k0, w.k1, pipe, smem, bars, acc);
        const int lin = w.lin, k0 = w.k0;
        if (k0 == 0 && w.k1 == w.KT) {
            store_tile<false>(p, w.org.x, w.org.y, acc);
        } else if (k0 > 0) {  // hand the partial sums for k >= k0 over to the owner
            if (partials) {
                store_partial(partials + static_cast<size_t>(blockIdx.x) * (BM * BN), acc);
                raise_flag(flags + blockIdx.x);
            } else {
                store_tile<false>(p, w.org.x, w.org.y, acc);
                raise_flag(flags + lin);
            }
        } else if (partials) {  // owner: add the parts of CTAs blockIdx.x+1 .. c_last
            const int c_last = w.last;
            for (int c = blockIdx.x + 1; c <= c_last; ++c) {
                wait_flag(flags + c, flags + gridDim.x);
                add_partial(partials + static_cast<size_t>(c) * (BM * BN), acc);
            }
            store_tile<false>(p, w.org.x, w.org.y, acc);
            if (threadIdx.x == 0)
                for (int c = blockIdx.x + 1; c <= c_last; ++c) flags[c] = 0u;
        } else {  // owner of a two-part tile
            wait_flag(flags + lin, flags + p.tiles_m * p.tiles_n);
            store_tile<true>(p, w.org.x, w.org.y, acc);
            if (threadIdx.x == 0) flags[lin] = 0u;
        }
        __syncthreads();  // shared memory (ring and segment) free for the next segment
    }
}

// The stream-K schedule of sgemm_f32_streamk_kernel on the k-major copy of
// A, with the 8 x 16 register tiles of sgemm_f32_kmajor_kernel (the segment
// walk, the hand-overs and their order are the same).
__global__ void __launch_bounds__(NT16, 2)
sgemm_f32_kmajor_streamk_kernel(const Problem p, const __grid_constant__ Maps maps, const int dp_tiles,
                                unsigned *flags, float *partials) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    __shared__ SkWalk w;  // advanced by thread 0 between barriers
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    init_bars<true>(bars);
    if (threadIdx.x == 0) sk_begin(w, p, dp_tiles, (p.K + BK_AT - 1) / BK_AT);
    for (;;) {
        if (threadIdx.x == 0) sk_next(w, p, dp_tiles);
        __syncthreads();  // the segment is visible to the CTA
        if (!w.more) break;
        Acc16 acc;
        acc16_zero(acc);
        uint32_t pipe = w.pipe;
        kmajor16_k_range(maps, w.org.x, w.org.y, w.k0, w.k1, pipe, smem, bars, acc);
        const int lin = w.lin, k0 = w.k0;
        if (k0 == 0 && w.k1 == w.KT) {
            store_tile16<false>(p, w.org.x, w.org.y, acc);
        } else if (k0 > 0) {  // hand the partial sums for k >= k0 over to the owner
            if (partials) {
                store_partial16(partials + static_cast<size_t>(blockIdx.x) * (BM * BN), acc);
                raise_flag(flags + blockIdx.x);
            } else {
                store_tile16<false>(p, w.org.x, w.org.y, acc);
                raise_flag(flags + lin);
            }
        } else if (partials) {  // owner: add the parts of CTAs blockIdx.x+1 .. c_last
            const int c_last = w.last;
            for (int c = blockIdx.x + 1; c <= c_last; ++c) {
                wait_flag(flags + c, flags + gridDim.x);
                add_partial16(partials + static_cast<size_t>(c) * (BM * BN), acc);
            }
            store_tile16<false>(p, w.org.x, w.org.y, acc);
            if (threadIdx.x == 0)
                for (int c = blockIdx.x + 1; c <= c_last; ++c) flags[c] = 0u;
        } else {  // owner of a two-part tile
            wait_flag(flags + lin, flags + p.tiles_m * p.tiles_n);
            store_tile16<true>(p, w.org.x, w.org.y, acc);
            if (threadIdx.x == 0) flags[lin] = 0u;
        }
        __syncthreads();  // shared memory (ring and segment) free for the next segment
    }
}

// Split tail.  The last R = T mod G tiles (G = co-resident CTAs) would leave
// a partial last wave; instead each is cut into S equal K ranges and the S*R
// CTAs of this grid, queued behind the one-CTA-per-tile grid of the other
// tiles, start as soon as SMs free up (programmatic dependent launch).  CTA
// c computes part c % S of tile dp_tiles + c / S into partial-sum slot c and
// counts itself in counts[c / S]; the part that arrives last adds all S
// slots in part order and stores the tile: deterministic, and no CTA waits
// for another.
template <int VA, int VB, bool TMA>
__global__ void __launch_bounds__(NT, 2)
sgemm_f32_tail_kernel(const Problem p, const __grid_constant__ Maps maps, const int dp_tiles, const int parts,
                      unsigned *counts, float *slots) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    __shared__ int last;
    __shared__ int2 org;
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    const int c = blockIdx.x, tile = c / parts, part = c - tile * parts;
    const int KT = (p.K + BK - 1) / BK;
    const int k0 = static_cast<int>(static_cast<long long>(KT) * part / parts);
    const int k1 = static_cast<int>(static_cast<long long>(KT) * (part + 1) / parts);
    int tm, tn;
    tile_of(dp_tiles + tile, p.tiles_m, p.tiles_n, tm, tn);
    init_cta<TMA>(bars, &org, tm * BM, tn * BN);
    Acc acc;
    acc_zero(acc);
    uint32_t pipe = 0;
    mma_k_range<VA, VB, TMA>(p, maps, &org, k0, k1, pipe, smem, bars, acc);
    store_partial(slots + static_cast<size_t>(c) * (BM * BN), acc);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned before = atomicAdd(counts + tile, 1u);
        __threadfence();
        last = before == static_cast<unsigned>(parts - 1) ? 1 : 0;
    }
    __syncthreads();
    if (last) {
        if (threadIdx.x == 0) counts[tile] = 0u;  // every part has counted itself: leave the word zero
        acc_zero(acc);
        for (int k = 0; k < parts; ++k) add_partial(slots + static_cast<size_t>(tile * parts + k) * (BM * BN), acc);
        store_tile<false>(p, org.x, org.y, acc);
    }
}

// The split tail of sgemm_f32_tail_kernel on the k-major copy of A, with the
// 8 x 16 register tiles of sgemm_f32_kmajor_kernel.
__global__ void __launch_bounds__(NT16, 2)
sgemm_f32_kmajor_tail_kernel(const Problem p, const __grid_constant__ Maps maps, const int dp_tiles, const int parts,
                             unsigned *counts, float *slots) {
    extern __shared__ float smem_raw[];
    __shared__ __align__(8) uint64_t bar_mem[kMaxRing];
    __shared__ int last;
    float *smem = aligned_smem(smem_raw);
    const uint32_t bars = smem_u32(bar_mem);
    init_bars<true>(bars);
    const int c = blockIdx.x, tile = c / parts, part = c - tile * parts;
    const int KT = (p.K + BK_AT - 1) / BK_AT;
    const int k0 = static_cast<int>(static_cast<long long>(KT) * part / parts);
    const int k1 = static_cast<int>(static_cast<long long>(KT) * (part + 1) / parts);
    int tm, tn;
    tile_of(dp_tiles + tile, p.tiles_m, p.tiles_n, tm, tn);
    Acc16 acc;
    acc16_zero(acc);
    uint32_t pipe = 0;
    kmajor16_k_range(maps, tm * BM, tn * BN, k0, k1, pipe, smem, bars, acc);
    store_partial16(slots + static_cast<size_t>(c) * (BM * BN), acc);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned before = atomicAdd(counts + tile, 1u);
        __threadfence();
        last = before == static_cast<unsigned>(parts - 1) ? 1 : 0;
    }
    __syncthreads();
    if (last) {
        if (threadIdx.x == 0) counts[tile] = 0u;  // every part has counted itself: leave the word zero
        acc16_zero(acc);
        for (int k = 0; k < parts; ++k)
            add_partial16(slots + static_cast<size_t>(tile * parts + k) * (BM * BN), acc);
        store_tile16<false>(p, tm * BM, tn * BN, acc);
    }
}

// Copies a rows x cols row-major matrix whose rows are not 16-byte aligned
// (leading dimension ld_src, any 4-byte alignment) into dst, whose leading
// dimension ld_dst is cols rounded up to 4 and whose base is 16-byte aligned,
// so that the tensor-copy kernels can read it.  Vector q of a row holds
// columns 4q .. 4q+3 (zeros past cols); consecutive threads take consecutive
// vectors of a row, so the scalar loads of a warp cover 512 contiguous bytes
// and each 16-byte store is aligned.  Grid-stride over rows x ld_dst / 4.
__global__ void __launch_bounds__(256) repack_rows_kernel(const float *__restrict__ src, long long ld_src, int rows,
                                                          int cols, float *__restrict__ dst, long long ld_dst) {
    const long long per_row = ld_dst / 4;
    const long long total = static_cast<long long>(rows) * per_row;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / per_row;
        const int c = static_cast<int>(i - r * per_row) * 4;
        const float *s = src + r * ld_src + c;
        float4 v;
        v.x = c < cols ? __ldg(s) : 0.0f;
        v.y = c + 1 < cols ? __ldg(s + 1) : 0.0f;
        v.z = c + 2 < cols ? __ldg(s + 2) : 0.0f;
        v.w = c + 3 < cols ? __ldg(s + 3) : 0.0f;
        *reinterpret_cast<float4 *>(dst + r * ld_dst + c) = v;
    }
}

// Runs one of the bounded waits above on a target that nothing completes
// (which = 0: a copy-ring mbarrier phase with no arrival and no copy; 1: a
// partner flag nobody raises) or on one that is already complete (2: the
// phase after an arrival; 3: a raised flag), with a short poll limit.
// status[0] = 1 if the wait gave up.  status[1] is the flag, status[2] the
// error word (both zeroed by the host).  One CTA of 32 threads.
__global__ void wait_selftest_kernel(int which, unsigned limit, unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    if (which == 0 || which == 2) {
        if (threadIdx.x == 0) {
            const uint32_t b = smem_u32(&bar);
            mbar_init(b, 1);
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
            if (which == 2) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(b) : "memory");
            mbar_wait_bounded(b, 0, limit, status);  // status[0] was zeroed by the host
        }
    } else {
        if (which == 3 && threadIdx.x == 0) st_release(status + 1, 1u);
        __syncthreads();
        wait_flag(status + 1, status + 2, limit);
        if (threadIdx.x == 0) status[0] = ld_acquire(status + 2) != 0u ? 1u : 0u;
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

constexpr int kMaxDevices = 64;
// Dynamic shared memory the cta_per_sm=1 diagnostic asks for: more than half
// of an SM's, so two CTAs never share one.
constexpr int kOneCtaSmem = 120 * 1024;
// Kernel variants: (VA, VB) in {4, 1} x {4, 2, 1} with cp.async (0..5) and
// (4, 4) with TMA (6), for the 8 x 8 row-major kernels; 7 is the 8 x 16
// kernel on the k-major copy of A.
constexpr int kVariants = 8;
constexpr int kTmaVariant = 6;
constexpr int kAtVariant = 7;
using DpKernel = void (*)(Problem, Maps);
using SkKernel = void (*)(Problem, Maps, int, unsigned *, float *);
const DpKernel kDp[kVariants] = {
    sgemm_f32_tiled_kernel<4, 4, false>, sgemm_f32_tiled_kernel<4, 2, false>,
    sgemm_f32_tiled_kernel<4, 1, false>, sgemm_f32_tiled_kernel<1, 4, false>,
    sgemm_f32_tiled_kernel<1, 2, false>, sgemm_f32_tiled_kernel<1, 1, false>,
    sgemm_f32_tiled_kernel<4, 4, true>,  sgemm_f32_kmajor_kernel<false>};
const SkKernel kSk[kVariants] = {
    sgemm_f32_streamk_kernel<4, 4, false>, sgemm_f32_streamk_kernel<4, 2, false>,
    sgemm_f32_streamk_kernel<4, 1, false>, sgemm_f32_streamk_kernel<1, 4, false>,
    sgemm_f32_streamk_kernel<1, 2, false>, sgemm_f32_streamk_kernel<1, 1, false>,
    sgemm_f32_streamk_kernel<4, 4, true>,  sgemm_f32_kmajor_streamk_kernel};
// The cluster split of K for the 8 x 8 variants (none for the k-major one).
const DpKernel kCk[kVariants] = {
    sgemm_f32_clusterk_kernel<4, 4, false>, sgemm_f32_clusterk_kernel<4, 2, false>,
    sgemm_f32_clusterk_kernel<4, 1, false>, sgemm_f32_clusterk_kernel<1, 4, false>,
    sgemm_f32_clusterk_kernel<1, 2, false>, sgemm_f32_clusterk_kernel<1, 1, false>,
    sgemm_f32_clusterk_kernel<4, 4, true>,  nullptr};
using TailKernel = void (*)(Problem, Maps, int, int, unsigned *, float *);
// tensor-copy variants only: [0] A row-major, [1] A k-major (8 x 16 tiles)
const TailKernel kTail[2] = {sgemm_f32_tail_kernel<4, 4, true>, sgemm_f32_kmajor_tail_kernel};
// The drained-ring diagnostic kernel of the k-major variant (one CTA per
// tile; SGEMM_F32_TUNE drain=on).
const DpKernel kDrained[1] = {sgemm_f32_kmajor_kernel<true>};
DpKernel dp_kernel(int v, bool drain) { return drain && v == kAtVariant ? kDrained[0] : kDp[v]; }
bool is_tma(int v) { return v == kTmaVariant || v == kAtVariant; }
// threads per CTA, dynamic shared memory and K-tile depth of variant v's kernels
unsigned threads(int v) { return v == kAtVariant ? NT16 : NT; }
int smem_of(int v) { return v == kAtVariant ? SMEM_AT_BYTES : SMEM_BYTES; }
int bk_of(int v) { return v == kAtVariant ? BK_AT : BK; }

// ---- tuning overrides --------------------------------------------------
// SGEMM_F32_TUNE = "key=value,key=value" (read once, at the first call) forces
// choices the cost models otherwise make, for tuning sweeps without a
// rebuild.  Keys (any other key or value is ignored; "auto" = the default):
//   kernels  = rowmajor8 | kmajor16 : the 8 x 8 row-major kernels only, or
//              the k-major copy of A whenever the workspace has room;
//   schedule = 0 | 1 | 2 | 3 : the schedule of sgemm_f32_ws when the
//              workspace has room for it (3 needs tensor copies);
//   parts    = 2 .. 16 : K parts of each split-tail tile;
//   cluster  = 2 .. 16 | off : the cluster size of the cluster split of K
//              wherever that size fits (T clusters resident at once, at
//              least 2 K tiles per CTA), whatever the cost model says, or
//              no cluster split;
//   drain    = on : a diagnostic: the one-CTA-per-tile grid of the k-major
//              kernels keeps one tile in flight and issues
//              it only after the k steps of the one before, so no copy
//              writes shared memory while fragments are read (slow; it
//              exists to count shared-memory bank conflicts without the
//              copy engines' concurrent writes);
//   cta_per_sm = 1 : a diagnostic: the one-CTA-per-tile grid asks for
//              enough shared memory that only one CTA fits on an SM (the
//              kernels use the first SMEM_BYTES of it), so that no second
//              CTA's copies or loads share the SM.
// A forced choice changes only how the work is split, so the product stays
// within the same FP32 bound (not bit for bit the default's).
struct Tune {
    int kernels = -1;   // -1 auto, 0 rowmajor8, 1 kmajor16
    int schedule = -1;
    int parts = -1;
    int cluster = -1;   // -1 auto, 0 off, 2 .. 16 forced
    bool drain = false; // the drained-ring diagnostic kernels
    bool one_cta = false; // one CTA per SM in the one-CTA-per-tile grid (diagnostic)
};
const Tune &tune() {
    static Tune t;
    static std::once_flag once;
    std::call_once(once, [] {
        const char *env = getenv("SGEMM_F32_TUNE");
        if (env == nullptr) return;
        char buf[256];
        strncpy(buf, env, sizeof buf - 1);
        buf[sizeof buf - 1] = 0;
        for (char *item = buf; item != nullptr && *item != 0;) {
            char *next = strchr(item, ',');
            if (next != nullptr) *next++ = 0;
            char *eq = strchr(item, '=');
            if (eq == nullptr) {
                item = next;
                continue;
            }
            *eq = 0;
            const char *key = item, *val = eq + 1;
            item = next;
            const long num = strtol(val, nullptr, 10);
            if (!strcmp(key, "kernels")) {
                t.kernels = !strcmp(val, "rowmajor8") ? 0 : !strcmp(val, "kmajor16") ? 1 : -1;
            } else if (!strcmp(key, "schedule")) {
                t.schedule = (val[0] >= '0' && val[0] <= '3' && val[1] == 0) ? static_cast<int>(num) : -1;
            } else if (!strcmp(key, "parts")) {
                t.parts = (num >= 2 && num <= 16) ? static_cast<int>(num) : -1;
            } else if (!strcmp(key, "cluster")) {
                t.cluster = !strcmp(val, "off") ? 0 : (num >= 2 && num <= 16) ? static_cast<int>(num) : -1;
            } else if (!strcmp(key, "drain")) {
                t.drain = !strcmp(val, "on");
            } else if (!strcmp(key, "cta_per_sm")) {
                t.one_cta = num == 1;
            }
        }
    });
    return t;
}

// When a call takes the k-major copy of A: never (at = 0), where it pays
// (1, the default) or whenever the workspace has room (2).
struct Policy {
    int at;
};
Policy policy() {
    switch (tune().kernels) {
        case 0: return {0};
        case 1: return {2};
        default: return {1};
    }
}

// cuTensorMapEncodeTiled, fetched from the driver at run time (no link
// against libcuda).  Null when unavailable: the cp.async kernels are used.
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

// Describes A (K x M elements, rows lda apart; box 16 x 128, 64-byte
// swizzle) and B (N x K, rows ldb apart; box 128 x 16, no swizzle) for the
// tensor copies.  With a_kmajor, A is the k-major copy At (M x K elements in
// the map's order, rows lda apart: box 128 x BK_AT, no swizzle, the As
// layout) and B's box is 128 x BK_AT.  Needs 16-byte aligned bases and row
// strides.
bool encode_maps(Maps &maps, int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                 bool a_kmajor = false) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t a_dim[2] = {static_cast<cuuint64_t>(a_kmajor ? M : K), static_cast<cuuint64_t>(a_kmajor ? K : M)};
    const cuuint64_t a_stride[1] = {static_cast<cuuint64_t>(lda) * 4};
    const cuuint32_t a_box[2] = {static_cast<cuuint32_t>(a_kmajor ? BM : BK),
                                 static_cast<cuuint32_t>(a_kmajor ? BK_AT : BM)};
    const cuuint64_t b_dim[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K)};
    const cuuint64_t b_stride[1] = {static_cast<cuuint64_t>(ldb) * 4};
    const cuuint32_t b_box[2] = {BN, a_kmajor ? static_cast<cuuint32_t>(BK_AT) : static_cast<cuuint32_t>(BK)};
    const cuuint32_t ones[2] = {1, 1};
    return enc(&maps.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(A), a_dim, a_stride, a_box, ones,
               CU_TENSOR_MAP_INTERLEAVE_NONE, a_kmajor ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
           enc(&maps.b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(B), b_dim, b_stride, b_box, ones,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int state;                    // 0 = not yet set up, 1 = ready, < 0 = status
    int sms;                      // multiprocessors
    int sk_per_sm[kVariants];     // co-resident stream-K CTAs per SM
    int max_cluster;              // largest cluster of the cluster split of K (0 = none, else 2 .. 16)
    int active_clusters[17];      // clusters of S CTAs the GPU holds at once (index S, 2 .. 16)
    unsigned long long ctx;       // id of the CUDA context the set-up was made in
};
std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];

int setup_device(int dev, DeviceInfo *out) {
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    unsigned long long ctx = 0;
    const bool known = sg_ctx::current_id(dev, &ctx);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (known && d.state != 0 && d.ctx != ctx) d.state = 0;  // a new context (e.g. after cudaDeviceReset)
    if (d.state == 0) {
        d.ctx = ctx;
        int major = 0, minor = 0, st = SGEMM_OK;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || major != 10 ||
            minor != 3) {
            st = SGEMM_ERR_DEVICE;
        } else {
            for (int v = 0; v < kVariants && st == SGEMM_OK; ++v) {
                const void *fns[2] = {reinterpret_cast<const void *>(kDp[v]), reinterpret_cast<const void *>(kSk[v])};
                for (const void *f : fns) {
                    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_of(v)) !=
                            cudaSuccess ||
                        cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
                        st = SGEMM_ERR_DEVICE;
                        break;
                    }
                }
                // co-resident CTAs per SM: the smaller of the stream-K and the
                // one-CTA-per-tile kernels' figures (the waves of both)
                int sk = 0, dp = 0;
                if (st == SGEMM_OK &&
                    (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sk, kSk[v], threads(v), smem_of(v)) !=
                         cudaSuccess ||
                     cudaOccupancyMaxActiveBlocksPerMultiprocessor(&dp, kDp[v], threads(v), smem_of(v)) !=
                         cudaSuccess))
                    st = SGEMM_ERR_DEVICE;
                d.sk_per_sm[v] = sk < dp ? sk : dp;
            }
            for (int v = 0; v < kVariants && st == SGEMM_OK; ++v)
                if (kCk[v] != nullptr &&
                    (cudaFuncSetAttribute(kCk[v], cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
                         cudaSuccess ||
                     cudaFuncSetAttribute(kCk[v], cudaFuncAttributePreferredSharedMemoryCarveout,
                                          cudaSharedmemCarveoutMaxShared) != cudaSuccess))
                    st = SGEMM_ERR_DEVICE;
            // The cluster split of K: every variant opts in to clusters beyond
            // the portable 8 CTAs, and the runtime reports, for each size S up
            // to 16, how many clusters of S of these CTAs the GPU holds at once
            // (a cluster must fit in one GPC, so this can be fewer than G / S).
            // All variants share block size and shared memory, so one variant's
            // figures stand for all.  Sizes it cannot place are not used.
            d.max_cluster = 0;
            for (int S = 0; S <= 16; ++S) d.active_clusters[S] = 0;
            if (st == SGEMM_OK) {
                bool nonportable = true;
                for (int v = 0; v < kVariants; ++v)
                    if (kCk[v] != nullptr &&
                        cudaFuncSetAttribute(kCk[v], cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
                        nonportable = false;
                for (int S = 2; S <= (nonportable ? 16 : 8); ++S) {
                    cudaLaunchAttribute attr;
                    attr.id = cudaLaunchAttributeClusterDimension;
                    attr.val.clusterDim.x = static_cast<unsigned>(S);
                    attr.val.clusterDim.y = 1;
                    attr.val.clusterDim.z = 1;
                    cudaLaunchConfig_t q = {};
                    q.gridDim = dim3(static_cast<unsigned>(S) * 64u);
                    q.blockDim = dim3(NT);
                    q.dynamicSmemBytes = SMEM_BYTES;
                    q.attrs = &attr;
                    q.numAttrs = 1;
                    int n = 0;
                    if (cudaOccupancyMaxActiveClusters(&n, kCk[kTmaVariant], &q) == cudaSuccess && n > 0) {
                        d.active_clusters[S] = n;
                        d.max_cluster = S;
                    }
                    (void)cudaGetLastError();
                }
            }
            // the one-CTA-per-tile kernels may be launched with the padded
            // request of the cta_per_sm=1 diagnostic
            for (int v = 0; v < kVariants && st == SGEMM_OK; ++v)
                if (cudaFuncSetAttribute(kDp[v], cudaFuncAttributeMaxDynamicSharedMemorySize, kOneCtaSmem) !=
                    cudaSuccess)
                    st = SGEMM_ERR_DEVICE;
            for (const DpKernel f : kDrained)
                if (st == SGEMM_OK &&
                    (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kOneCtaSmem) != cudaSuccess ||
                     cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                          cudaSharedmemCarveoutMaxShared) != cudaSuccess))
                    st = SGEMM_ERR_DEVICE;
            for (int t = 0; t < 2; ++t)
                if (st == SGEMM_OK &&
                    (cudaFuncSetAttribute(kTail[t], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          t == 1 ? SMEM_AT_BYTES : SMEM_BYTES) != cudaSuccess ||
                     cudaFuncSetAttribute(kTail[t], cudaFuncAttributePreferredSharedMemoryCarveout,
                                          cudaSharedmemCarveoutMaxShared) != cudaSuccess))
                    st = SGEMM_ERR_DEVICE;
        }
        if (st != SGEMM_OK) (void)cudaGetLastError();  // do not leave our failure sticky for the caller
        d.state = st == SGEMM_OK ? 1 : st;
    }
    if (d.state < 0) return d.state;
    *out = d;
    return SGEMM_OK;
}

// Largest v in {4, 2, 1} floats such that the pointer and every row start are
// 4*v-byte aligned.
int vector_class(const void *p, long long ld) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (a % 16 == 0 && ld % 4 == 0) return 4;
    if (a % 8 == 0 && ld % 2 == 0) return 2;
    return 1;
}

bool ranges_overlap(const void *p, long long p_bytes, const void *q, long long q_bytes) {
    if (p_bytes <= 0 || q_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + static_cast<uintptr_t>(p_bytes);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(q), b1 = b0 + static_cast<uintptr_t>(q_bytes);
    return a0 < b1 && b0 < a1;
}

long long extent(long long rows, long long cols, long long ld) {
    return (rows == 0 || cols == 0) ? 0 : (rows - 1) * ld + cols;
}

long long tile_count(int M, int N) {
    return ((static_cast<long long>(M) + BM - 1) / BM) * ((static_cast<long long>(N) + BN - 1) / BN);
}

// Host-side argument checks shared by every entry point; touches no GPU.
int check_args(int M, int N, int K, const float *A, int lda, const float *B, int ldb, const float *C, int ldc) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_LD;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_NULL_PTR;
    if (K > 0 && (A == nullptr || B == nullptr)) return SGEMM_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(C) % 4 != 0) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && (reinterpret_cast<uintptr_t>(A) % 4 != 0 || reinterpret_cast<uintptr_t>(B) % 4 != 0))
        return SGEMM_ERR_INVALID_ARG;
    const long long c_bytes = 4 * extent(M, N, ldc);
    if (K > 0 && (ranges_overlap(C, c_bytes, A, 4 * extent(M, K, lda)) ||
                  ranges_overlap(C, c_bytes, B, 4 * extent(K, N, ldb))))
        return SGEMM_ERR_ALIAS;
    if (tile_count(M, N) > INT_MAX) return SGEMM_ERR_INVALID_DIM;
    return SGEMM_OK;
}

// How one product is scheduled.  kind 0: one CTA per tile.  kind 1:
// stream-K over the last wave-and-a-bit of tiles, partial sums handed over
// through C (needs flags only).  kind 2: stream-K over all tiles with any
// number of parts per tile, partial sums handed over through per-CTA slots
// (for fewer tiles than co-resident CTAs).  kind 3: one CTA per tile for
// all whole waves, and the R leftover tiles cut into S parts each in a
// split-tail grid (tensor-copy variant only).
struct Plan {
    int kind;
    long long grid, dp_tiles;
    long long flag_words;      // flags (tile counts for kind 3) plus the error word
    size_t partials_offset;    // byte offset of the partial slots (kinds 2 and 3)
    size_t bytes;              // workspace bytes needed
    int tail_parts;            // S (kind 3)
    long long tail_tiles;      // R (kind 3)
};
// K tiles per CTA below which splitting stops paying.  Measured on GB300
// (stream-K kernel, fewer tiles than resident CTAs): 4 beats 8 at 256^3
// (22.5 -> 18.5 us) and 512^3 (24.6 -> 22.5 us); 2 is slower at 512^3
// (32.5 us), where the owner's serial fix-up of more parts dominates.
constexpr long long kMinItersPerCta = 4;

// Chooses the schedule for T output tiles of KT K tiles each, with G CTAs
// resident at once on `sms` multiprocessors.
//   More tiles than resident CTAs, with a partial last wave (R = T mod G):
//   with `allow_tail`, kind 3.  Measured on GB300 for 2500x2100x4096 ..
//   8192^3 it beat one CTA per tile everywhere (+0.7 % .. +5.5 %).  S = 4
//   parts when R <= sms, else min(8, 4G/R): within about 1 % of the best S
//   at every shape measured, and the partial-sum slots stay below 4G tiles.
//   Without it, the cost model fitted to timings of 340..1024-tile products:
//   one CTA per tile takes floor(T/G) full rounds plus, for a last partial
//   wave, 0.55 of a round when it has at most one CTA per SM (a lone CTA runs
//   faster) or a full round otherwise; the split schedule takes T/G rounds
//   plus about 4.5 %, and is chosen only when it is at least 3 % better.
//   Fewer tiles than resident CTAs: the multi-part split is used when it
//   adds more than 10 % CTAs.
// SGEMM_F32_TUNE may force the schedule and the part count S.
Plan plan_schedule(long long T, long long KT, long long G, long long sms, bool allow_tail) {
    Plan pl = {0, T, 0, 0, 0, 0, 0, 0};
    if (KT <= 0 || G <= 0) return pl;
    const int forced = tune().schedule;
    if (forced == 0) return pl;
    const bool want_tail = forced == 3 || (forced < 0 && T > G);
    if (forced != 2 && T > G) {
        const long long W = T / G, R = T % G;
        if (R == 0 && forced < 0) return pl;  // whole waves: already balanced
        if (want_tail && allow_tail && KT >= 2 && R > 0) {
            long long S = R <= sms ? 4 : (4 * G / R < 4 ? 4 : (4 * G / R > 8 ? 8 : 4 * G / R));
            if (tune().parts > 0) S = tune().parts;
            if (S > KT) S = KT;
            pl.kind = 3;
            pl.grid = S * R;
            pl.dp_tiles = T - R;
            pl.tail_parts = static_cast<int>(S);
            pl.tail_tiles = R;
            pl.flag_words = R;
            pl.partials_offset = (static_cast<size_t>(R) * sizeof(unsigned) + 255) / 256 * 256;
            pl.bytes = pl.partials_offset + static_cast<size_t>(S * R) * BM * BN * sizeof(float);
            return pl;
        }
        const double dp_rounds = static_cast<double>(W) + (R <= sms ? 0.55 : 1.0);
        const double sk_rounds = static_cast<double>(T) / static_cast<double>(G) * 1.045;
        if (forced != 1 && sk_rounds > 0.97 * dp_rounds) return pl;
        pl.kind = 1;
        pl.grid = G;
        pl.dp_tiles = (W - 1) * G;  // the last T - dp_tiles tiles (between G and 2G) are split
        pl.flag_words = T + 1;
        pl.bytes = static_cast<size_t>(pl.flag_words) * sizeof(unsigned);
        return pl;
    }
    long long g = (T * KT / kMinItersPerCta < G) ? T * KT / kMinItersPerCta : G;
    if (forced != 2 && static_cast<double>(g) <= 1.1 * static_cast<double>(T)) return pl;  // too few extra CTAs
    if (g < 1) g = 1;
    pl.kind = 2;
    pl.grid = g;
    pl.flag_words = g + 1;
    pl.partials_offset = (static_cast<size_t>(pl.flag_words) * sizeof(unsigned) + 255) / 256 * 256;
    pl.bytes = pl.partials_offset + static_cast<size_t>(g) * BM * BN * sizeof(float);
    return pl;
}

// Kernel variant for these operands: copy widths by alignment class, and
// the tensor-copy variant when both are 16-byte aligned and the tensor maps
// encode (then filled into `maps`).
int choose_variant(int M, int N, int K, const float *A, int lda, const float *B, int ldb, Maps &maps) {
    const int va = K > 0 ? (vector_class(A, lda) == 4 ? 4 : 1) : 4;
    const int vb = K > 0 ? vector_class(B, ldb) : 4;
    int v = (va == 4 ? 0 : 3) + (vb == 4 ? 0 : vb == 2 ? 1 : 2);
    memset(&maps, 0, sizeof maps);
    if (v == 0 && K > 0 && encode_maps(maps, M, N, K, A, lda, B, ldb)) v = kTmaVariant;
    return v;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Products below this many FLOPs copy no operand (and get no room for copies
// from sgemm_f32_workspace_size_for).  Measured on GB300 with a workspace
// large enough for every copy (us, narrow copies -> copies first):
// 300 x 262 x 190 13.1 -> 34.6, 512^3 with lda = ldb = 513 23.1 -> 32.8,
// 700 x 900 x 333 30.1 -> 32.5, 1000 x 1030 x 777 52.8 -> 59.8 (or 54.5 with
// rows repacked instead of the k-major copy); from about 2 GFLOP on the
// copies win: 1024 x 1024 x 1025 60.9 -> 57.5, 2000 x 1030 x 777 91.7 -> 84.4
// (earlier, before the cluster split: 1536^3 153.7 -> 131.3,
// 2048 x 2048 x 2049 362.1 -> 289.3).
constexpr double kRepackMinFlops = 2e9;

// Whether transposing a 16-byte aligned A into its k-major copy first pays.
// Measured on GB300, transpose included (TFLOP/s, row-major 8 x 8 kernels ->
// k-major 8 x 16 kernels with 32-deep K tiles, the same schedule rules): the
// k-major kernels take about 6 % less time than the row-major ones:
//   one CTA per tile / split tail: 3072^3 64.51 -> 67.66, 4096^3 69.34 ->
//     73.04, 6144^3 70.14 -> 74.27, 8192^3 70.39 -> 74.64;
//   stream-K (fewer tiles than resident CTAs): 2048^3 62.10 -> 64.39,
//     2048x2048x4096 64.02 -> 66.87, 256x16384x4096 63.93 -> 67.80; but
//     1024^3 40.36 -> 37.19, 16384x256x4096 63.81 -> 58.98, 16384x512x4096
//     67.32 -> 66.10 and 32768x256x4096 67.32 -> 61.62, where the transpose
//     costs more than it saves (A is large next to the product).
// The transpose moves 8 M K bytes at about 5.5 TB/s plus a launch (4096^2
// 21 us, 16384 x 4096 84 us).  So the copy is taken when the expected
// saving, 6 % of 2MNK at 68 TFLOP/s, exceeds 1.2 x the transpose's time.  An
// A whose rows are not 16-byte aligned is copied anyway, and then always
// into the k-major copy.
bool kmajor_pays(int M, int N, int K) {
    const double saving = 0.06 * 2.0 * M * N * K / 68e12;
    const double copy = 8.0 * M * K / 5.5e12 + 4e-6;
    return saving > 1.2 * copy;
}

// Copies of the operands in the workspace (workspace entry point only),
// placed after the schedule's own words and slots.
//   * k-major A: when the workspace has room for it, A is first transposed
//     into At = A^T (K rows of M floats, row stride M rounded up to 4) by
//     the transpose kernel, whatever A's alignment, and the product runs on
//     the k-major tensor-copy kernels (kAtVariant), which load the fragment
//     layout directly and store nothing to shared memory in their K loop.
//   * Otherwise an operand whose rows are not 16-byte aligned is copied into
//     16-byte aligned rows when there is room, and the product runs on the
//     tensor-copy kernels and their schedules; else on the cp.async kernels
//     with narrower copies.
//   B is repacked in both cases when its rows are not 16-byte aligned.
struct Repack {
    bool a, b;            // A / B repacked
    bool at;              // A transposed into the k-major copy (instead of repacked)
    int lda2, ldb2;       // the repacked leading dimensions (K, N rounded up to 4)
    int ldat;             // the k-major copy's row stride (M rounded up to 4)
    size_t a_off, b_off;  // byte offsets of the copies in the workspace
    size_t at_off;
    size_t plan_bytes;    // the schedule's region at the start of the workspace
    size_t bytes;         // total workspace bytes this needs
};
Repack plan_repack(int M, int N, int K, const float *A, int lda, const float *B, int ldb, const DeviceInfo &info,
                   size_t avail, const Policy &pol) {
    Repack r = {false, false, false, 0, 0, 0, 0, 0, 0, 0, 0};
    if (K <= 0 || encode_fn() == nullptr) return r;
    // Below kRepackMinFlops the narrow-copy kernels (and their cluster split
    // of K) beat every copy, whatever room the workspace has (see there),
    // unless SGEMM_F32_TUNE picks the kernel family.
    if (pol.at == 1 && 2.0 * M * N * K < kRepackMinFlops) return r;
    const bool ra = vector_class(A, lda) != 4, rb = vector_class(B, ldb) != 4;
    const bool want_at = pol.at == 2 || (pol.at == 1 && (ra || kmajor_pays(M, N, K)));
    if (!ra && !rb && !want_at) return r;
    const int v = want_at ? kAtVariant : kTmaVariant;
    const long long T = tile_count(M, N), KT = (K + bk_of(v) - 1) / bk_of(v);
    const Plan pl = plan_schedule(T, KT, static_cast<long long>(info.sk_per_sm[v]) * info.sms, info.sms, true);
    r.lda2 = (K + 3) / 4 * 4;
    r.ldb2 = (N + 3) / 4 * 4;
    r.ldat = (M + 3) / 4 * 4;
    r.plan_bytes = round256(pl.bytes);
    if (want_at) {
        size_t off = r.plan_bytes;
        r.at_off = off;
        off += round256(static_cast<size_t>(K) * r.ldat * sizeof(float));
        if (rb) {
            r.b_off = off;
            off += round256(static_cast<size_t>(K) * r.ldb2 * sizeof(float));
        }
        r.bytes = off;
        if (off <= avail) {
            r.at = true;
            r.b = rb;
            return r;
        }
        if (!ra && !rb) return r;  // no room: nothing else to copy
    }
    size_t off = r.plan_bytes;
    if (ra) {
        r.a_off = off;
        off += round256(static_cast<size_t>(M) * r.lda2 * sizeof(float));
    }
    if (rb) {
        r.b_off = off;
        off += round256(static_cast<size_t>(K) * r.ldb2 * sizeof(float));
    }
    if (!want_at) r.bytes = off;
    if (off <= avail) {
        r.a = ra;
        r.b = rb;
    }
    return r;
}

// The schedule run() uses: plan_schedule, then the fallbacks run() takes when
// the workspace region (avail bytes) is too small for it.
Plan effective_plan(long long T, long long KT, long long G, long long sms, bool tma, size_t avail) {
    Plan pl = plan_schedule(T, KT, G, sms, tma);
    if (pl.kind == 3 && avail < pl.bytes) pl = plan_schedule(T, KT, G, sms, false);
    if (pl.kind != 0 && avail < pl.bytes) pl = Plan{0, T, 0, 0, 0, 0, 0, 0};
    return pl;
}

// Cluster size of the cluster split of K for T output tiles of KT K tiles
// with G CTAs resident at once, or 0 when it does not apply: products with at
// most G / 2 tiles (the split then fills the GPU without a second wave), at
// least 2 K tiles per CTA, on the 8 x 8 kernels (variant v).  S = the most
// CTAs per tile that keep all T clusters resident at once (at most G / T, and
// T at most the clusters of S the GPU holds at once: a cluster must fit in
// one GPC), at most 8 (the portable cluster size), or at most the largest
// size the GPU places (16 on GB300) when T clusters of it take at most a
// quarter of the resident CTAs.  Measured on GB300 (us, clusters of at most 8 -> of at
// most 16): 256 x 256 x 1024 (S = 16) 20.7 -> 16.9, 256 x 256 x 4096 52.0 ->
// 33.2; but with more tiles larger clusters lost: 512^3 (16 tiles, S = 16)
// 20.6 -> 25.0, 768 x 512 x 512 (S = 12) 22.6 -> 25.7, 1024 x 512 x 1024
// (S = 9) 32.7 -> 41.4, 128 x 4096 x 4096 (S = 9) 90.2 -> 117.1.
// When the multi-part stream-K schedule `sk` (kind 2, g CTAs) could run
// instead, the split is taken only if it is expected to be faster.  Cost in
// K tiles of one CTA with two CTAs per SM (about 2.4 us each); a grid that
// fills at most half the SMs runs one CTA per SM, whose K tile costs 0.55 of
// that.  Fitted to GB300 timings of both schedules:
//   cluster split: 4.7 + ceil(KT / S) (launch, the two cluster barriers and
//                  the sum over distributed shared memory);
//   stream-K:      7.5 + T KT / g + 0.3 ceil(g / T) (flag reset, hand-over
//                  waits, and the owner's serial sum of ceil(g / T) parts).
// Measured, split against stream-K (us): 1024^3 49.7 / 53.1, 512 x 512 x
// 1024 30.9 / 38.9, 384 x 384 x 2048 31.5 / 61.2, 256 x 256 x 4096 33.2 /
// 101.7; stream-K faster at 2048 x 1024 x 1024 88.3 / 83.9, 1024 x 1024 x
// 2048 88.1 / 86.0, 1024 x 1024 x 4096 165 / 149.5, 512 x 512 x 4096 88.4 /
// 63.3.  The model picks the faster of the two at every one of these shapes.
// SGEMM_F32_TUNE schedule=0..3 or cluster=off turns the split off; cluster=S
// forces its size where it fits.
int cluster_split(long long T, long long KT, long long G, int v, const Plan *sk, const DeviceInfo &info) {
    if (v >= kAtVariant || kCk[v] == nullptr || tune().schedule >= 0 || tune().cluster == 0 || T <= 0 || 2 * T > G)
        return 0;
    if (const int forced = tune().cluster; forced >= 2)
        return forced <= info.max_cluster && forced <= KT / 2 && T * forced <= G && T <= info.active_clusters[forced]
                   ? forced
                   : 0;
    // clusters above the portable 8 only while all of them use at most a
    // quarter of the resident CTAs (at most 4 tiles here)
    const long long cap = 4 * T * info.max_cluster <= G ? info.max_cluster : (info.max_cluster < 8 ? info.max_cluster : 8);
    long long S = cap < KT / 2 ? cap : KT / 2;
    while (S >= 2 && (T * S > G || T > info.active_clusters[S])) --S;  // one wave of clusters
    if (S < 2) return 0;
    if (sk != nullptr && sk->grid > 0) {
        const double g = static_cast<double>(sk->grid);
        const double lone = 0.55;  // K tile of a CTA alone on its SM
        const double split = 4.7 + static_cast<double>((KT + S - 1) / S) * (4 * T * S <= G ? lone : 1.0);
        const double streamk = 7.5 + static_cast<double>(T * KT) / g * (4 * sk->grid <= G ? lone : 1.0) +
                               0.3 * static_cast<double>((sk->grid + T - 1) / T);
        if (split > streamk) return 0;
    }
    return static_cast<int>(S);
}

// Runs one product whose arguments passed check_args (M, N > 0).  Uses a
// stream-K schedule when the workspace `flags` (flag_bytes long) is large
// enough for the plan chosen for this shape; else one CTA per tile.
int run(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
        unsigned *flags, size_t flag_bytes, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    DeviceInfo info;
    const int st = setup_device(dev, &info);
    if (st != SGEMM_OK) return st;

    const Policy pol = policy();
    const Repack rp = plan_repack(M, N, K, A, lda, B, ldb, info, flags != nullptr ? flag_bytes : 0, pol);
    Maps maps;
    if (rp.at) {
        // every copy's address is known before anything is launched: encode
        // the tensor maps of the copies first, so a failure launches nothing
        char *ws = reinterpret_cast<char *>(flags);
        float *at = reinterpret_cast<float *>(ws + rp.at_off);
        float *b2 = rp.b ? reinterpret_cast<float *>(ws + rp.b_off) : nullptr;
        memset(&maps, 0, sizeof maps);
        if (!encode_maps(maps, M, N, K, at, rp.ldat, rp.b ? b2 : B, rp.b ? rp.ldb2 : ldb, true))
            return SGEMM_ERR_DEVICE;
        sg_nvtx::Range r("sgemm_f32: k-major copy of A");
        if (transpose_f32(M, K, A, lda, at, rp.ldat, stream) != TRANSPOSE_OK) {
            (void)cudaGetLastError();
            return SGEMM_ERR_LAUNCH;
        }
        A = at;
        lda = rp.ldat;
        if (rp.b) {
            repack_rows_kernel<<<static_cast<unsigned>(info.sms) * 8, 256, 0, stream>>>(B, ldb, K, N, b2, rp.ldb2);
            if (cudaPeekAtLastError() != cudaSuccess) {
                (void)cudaGetLastError();
                return SGEMM_ERR_LAUNCH;
            }
            B = b2;
            ldb = rp.ldb2;
        }
        flag_bytes = rp.plan_bytes;  // the schedule keeps to the region before the copies
    } else if (rp.a || rp.b) {
        sg_nvtx::Range r("sgemm_f32: repack rows");
        char *ws = reinterpret_cast<char *>(flags);
        const unsigned blocks = static_cast<unsigned>(info.sms) * 8;
        if (rp.a) {
            float *a2 = reinterpret_cast<float *>(ws + rp.a_off);
            repack_rows_kernel<<<blocks, 256, 0, stream>>>(A, lda, M, K, a2, rp.lda2);
            A = a2;
            lda = rp.lda2;
        }
        if (rp.b) {
            float *b2 = reinterpret_cast<float *>(ws + rp.b_off);
            repack_rows_kernel<<<blocks, 256, 0, stream>>>(B, ldb, K, N, b2, rp.ldb2);
            B = b2;
            ldb = rp.ldb2;
        }
        if (cudaPeekAtLastError() != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_LAUNCH;
        }
        flag_bytes = rp.plan_bytes;  // the schedule keeps to the region before the copies
    }

    const int v = rp.at ? kAtVariant : choose_variant(M, N, K, A, lda, B, ldb, maps);
    Problem p;
    p.M = M; p.N = N; p.K = K; p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.vc = vector_class(C, ldc);
    const long long T = static_cast<long long>(p.tiles_m) * p.tiles_n;
    const long long G = static_cast<long long>(info.sk_per_sm[v]) * info.sms;
    const long long KT = (K + bk_of(v) - 1) / bk_of(v);
    Plan pl = plan_schedule(T, KT, G, info.sms, is_tma(v));

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem_of(v);
    cfg.stream = stream;
    const bool streamk = flags != nullptr && pl.kind == 2 && flag_bytes >= pl.bytes;
    if (const int S = cluster_split(T, KT, G, v, streamk ? &pl : nullptr, info)) {
        sg_nvtx::Range r("sgemm_f32: cluster split of K");
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(S);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(T * S));
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kCk[v], p, maps) == cudaSuccess) return SGEMM_OK;
        // The runtime refused the clusters (e.g. a process granted fewer SMs
        // than the set-up's occupancy figures assume): run the schedule the
        // call would run without the split.
        (void)cudaGetLastError();
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
    }
    if (pl.kind == 3) {
        if (flags != nullptr && flag_bytes >= pl.bytes) {
            unsigned *counts = flags;
            float *slots = reinterpret_cast<float *>(reinterpret_cast<char *>(flags) + pl.partials_offset);
            if (cudaMemsetAsync(counts, 0, static_cast<size_t>(pl.flag_words) * sizeof(unsigned), stream) !=
                cudaSuccess) {
                (void)cudaGetLastError();
                return SGEMM_ERR_LAUNCH;
            }
            sg_nvtx::Range r("sgemm_f32: whole waves + split tail");
            cfg.gridDim = dim3(static_cast<unsigned>(pl.dp_tiles));
            cfg.blockDim = dim3(threads(v));
            if (cudaLaunchKernelEx(&cfg, dp_kernel(v, tune().drain), p, maps) != cudaSuccess) {
                (void)cudaGetLastError();
                return SGEMM_ERR_LAUNCH;
            }
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr.val.programmaticStreamSerializationAllowed = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            if (cudaLaunchKernelEx(&cfg, kTail[v == kAtVariant ? 1 : 0], p, maps, static_cast<int>(pl.dp_tiles),
                                   pl.tail_parts, counts,
                                   slots) != cudaSuccess) {
                (void)cudaGetLastError();
                return SGEMM_ERR_LAUNCH;
            }
            return SGEMM_OK;
        }
        pl = plan_schedule(T, KT, G, info.sms, false);  // workspace too small for the split tail
    }
    cudaError_t err = cudaErrorUnknown;
    bool done = false;
    if (flags != nullptr && pl.kind != 0 && flag_bytes >= pl.bytes) {
        float *partials =
            pl.kind == 2 ? reinterpret_cast<float *>(reinterpret_cast<char *>(flags) + pl.partials_offset) : nullptr;
        sg_nvtx::Range r("sgemm_f32: stream-K");
        err = cudaMemsetAsync(flags, 0, static_cast<size_t>(pl.flag_words) * sizeof(unsigned), stream);
        if (err == cudaSuccess) {
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeCooperative;
            attr.val.cooperative = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
            cfg.blockDim = dim3(threads(v));
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            err = cudaLaunchKernelEx(&cfg, kSk[v], p, maps, static_cast<int>(pl.dp_tiles), flags, partials);
            done = err == cudaSuccess;
            if (err == cudaErrorCooperativeLaunchTooLarge) {  // fewer SMs free than set up for
                (void)cudaGetLastError();
                err = cudaSuccess;
            }
            cfg.attrs = nullptr;
            cfg.numAttrs = 0;
        }
    }
    if (!done && err != cudaSuccess && err != cudaErrorUnknown) {
        (void)cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    if (!done) {
        sg_nvtx::Range r("sgemm_f32: one CTA per tile");
        cfg.gridDim = dim3(static_cast<unsigned>(T));
        cfg.blockDim = dim3(threads(v));
        if (tune().one_cta) cfg.dynamicSmemBytes = kOneCtaSmem;
        err = cudaLaunchKernelEx(&cfg, dp_kernel(v, tune().drain), p, maps);
        if (err != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_LAUNCH;
        }
    }
    return SGEMM_OK;
}

// ---- fixed scratch for sgemm_f32_static_scratch ----------------------
// One 32-bit flag per output tile plus the error word, for callers that
// cannot allocate device memory.  Every GPU that loads this library holds
// the array (64 KiB) until the process exits.
constexpr int kStaticScratchWords = 16384;
constexpr long long kStaticMaxTiles = kStaticScratchWords - 1;
static __device__ __align__(256) unsigned g_static_scratch[kStaticScratchWords];

std::mutex g_static_mutex;
unsigned *g_static_ptr[kMaxDevices];   // device address of g_static_scratch
int g_static_state[kMaxDevices];       // 0 = not yet looked up, 1 = ready, < 0 = status
unsigned long long g_static_ctx[kMaxDevices];  // context the address belongs to

// Looks up, once per device (and again in a new context of that device, e.g.
// after cudaDeviceReset) and with that device current, the device address of
// g_static_scratch (the host-side name is only a stand-in).
int static_scratch(int dev, unsigned **out) {
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    unsigned long long ctx = 0;
    const bool known = sg_ctx::current_id(dev, &ctx);
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (known && g_static_state[dev] != 0 && g_static_ctx[dev] != ctx) g_static_state[dev] = 0;
    if (g_static_state[dev] == 0) {
        g_static_ctx[dev] = ctx;
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            g_static_state[dev] = SGEMM_ERR_DEVICE;
        } else {
            g_static_ptr[dev] = static_cast<unsigned *>(ptr);
            g_static_state[dev] = 1;
        }
    }
    if (g_static_state[dev] < 0) return g_static_state[dev];
    *out = g_static_ptr[dev];
    return SGEMM_OK;
}

}  // namespace

extern "C" int sgemm_f32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                         cudaStream_t stream) {
    const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    return run(M, N, K, A, lda, B, ldb, C, ldc, nullptr, 0, stream);
}

extern "C" size_t sgemm_f32_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K < 0) return 0;
    const long long T = tile_count(M, N);
    size_t bytes = static_cast<size_t>(T + 1) * sizeof(unsigned);  // flags of the two-part schedule
    int dev = 0;
    DeviceInfo info;
    if (cudaGetDevice(&dev) == cudaSuccess && setup_device(dev, &info) == SGEMM_OK) {
        int per_sm = 0;
        for (int v = 0; v < kVariants; ++v) per_sm = info.sk_per_sm[v] > per_sm ? info.sk_per_sm[v] : per_sm;
        for (const bool tail : {true, false}) {
            const Plan pl = plan_schedule(T, (K + BK - 1) / BK, static_cast<long long>(per_sm) * info.sms, info.sms, tail);
            if (pl.bytes > bytes) bytes = pl.bytes;
        }
    } else {
        (void)cudaGetLastError();
    }
    return (bytes + 255) / 256 * 256;
}

extern "C" size_t sgemm_f32_workspace_size_for(int M, int N, int K, const float *A, int lda, const float *B,
                                               int ldb) {
    const size_t base = sgemm_f32_workspace_size(M, N, K);
    // Smaller products copy nothing (kRepackMinFlops), so no room is asked
    // for them.
    if (base == 0 || K == 0 || 2.0 * M * N * K < kRepackMinFlops) return base;
    int dev = 0;
    DeviceInfo info;
    if (cudaGetDevice(&dev) != cudaSuccess || setup_device(dev, &info) != SGEMM_OK) {
        (void)cudaGetLastError();
        return base;
    }
    const Repack rp = plan_repack(M, N, K, A, lda, B, ldb, info, SIZE_MAX, policy());
    return rp.bytes > base ? round256(rp.bytes) : base;
}

extern "C" int sgemm_f32_ws_schedule(int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                                     const float *C, int ldc, size_t workspace_bytes, int *kind, long long *words) {
    if (kind == nullptr || words == nullptr) return SGEMM_ERR_NULL_PTR;
    *kind = 0;
    *words = 0;
    const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    int dev = 0;
    DeviceInfo info;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    const int sd = setup_device(dev, &info);
    if (sd != SGEMM_OK) return sd;
    const Policy pol = policy();
    const Repack rp = plan_repack(M, N, K, A, lda, B, ldb, info, workspace_bytes, pol);
    int v = rp.at ? kAtVariant : kTmaVariant;  // the copies have 16-byte aligned rows
    if (!rp.a && !rp.b && !rp.at) {
        Maps maps;
        v = choose_variant(M, N, K, A, lda, B, ldb, maps);
    }
    const size_t avail = (rp.a || rp.b || rp.at) ? rp.plan_bytes : workspace_bytes;
    const long long T = tile_count(M, N), KT = (K + bk_of(v) - 1) / bk_of(v);
    const long long G = static_cast<long long>(info.sk_per_sm[v]) * info.sms;
    const int copies = (rp.a ? 4 : 0) | (rp.b ? 8 : 0) | (rp.at ? 16 : 0);
    const Plan pl = effective_plan(T, KT, G, info.sms, is_tma(v), avail);
    if (const int S = K > 0 ? cluster_split(T, KT, G, v, pl.kind == 2 ? &pl : nullptr, info) : 0) {
        *kind = 32 | copies | (S << 8);  // cluster split of K: no schedule words
        return SGEMM_OK;
    }
    *kind = pl.kind | copies;
    *words = pl.flag_words;
    return SGEMM_OK;
}

extern "C" int sgemm_f32_ws(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                            int ldc, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    if (workspace == nullptr && workspace_bytes != 0) return SGEMM_ERR_NULL_PTR;
    if (workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SGEMM_ERR_INVALID_ARG;
    const long long wb = static_cast<long long>(workspace_bytes);
    if (workspace != nullptr &&
        (ranges_overlap(workspace, wb, C, 4 * extent(M, N, ldc)) ||
         (K > 0 && (ranges_overlap(workspace, wb, A, 4 * extent(M, K, lda)) ||
                    ranges_overlap(workspace, wb, B, 4 * extent(K, N, ldb))))))
        return SGEMM_ERR_ALIAS;
    return run(M, N, K, A, lda, B, ldb, C, ldc, static_cast<unsigned *>(workspace), workspace_bytes, stream);
}

extern "C" int sgemm_f32_static_scratch(int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                                        float *C, int ldc, cudaStream_t stream) {
    const int st = check_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    if (tile_count(M, N) > kStaticMaxTiles) return SGEMM_ERR_SCRATCH_LIMIT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    unsigned *scratch = nullptr;
    const int sst = static_scratch(dev, &scratch);
    if (sst != SGEMM_OK) return sst;
    return run(M, N, K, A, lda, B, ldb, C, ldc, scratch, sizeof(g_static_scratch), stream);
}

extern "C" const char *sgemm_f32_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "success";
        case SGEMM_ERR_INVALID_DIM: return "invalid dimension (negative M, N or K, or too many tiles)";
        case SGEMM_ERR_INVALID_LD: return "invalid leading dimension (lda < max(1,K), ldb or ldc < max(1,N))";
        case SGEMM_ERR_NULL_PTR: return "null pointer for a non-empty matrix";
        case SGEMM_ERR_ALIAS: return "C overlaps A or B";
        case SGEMM_ERR_LAUNCH: return "kernel launch rejected by the CUDA runtime";
        case SGEMM_ERR_DEVICE: return "current device is not sm_103 or its set-up failed";
        case SGEMM_ERR_INVALID_ARG: return "invalid argument (misaligned pointer or out-of-range value)";
        case SGEMM_ERR_SCRATCH_LIMIT:
            return "more than 16383 output tiles of 128 x 128: beyond the fixed scratch of sgemm_f32_static_scratch";
        default: return "unknown status";
    }
}

extern "C" int sgemm_f32_smem_shape(int kind, int *n_warps, int *n_steps, int *n_stages) {
    int steps;
    switch (kind) {
        case 0: steps = A_COPIES16; break;
        case 1: steps = b_copies<4>(); break;
        case 2:
        case 3: steps = 2 * BK; break;
        case 11: steps = 2 * BK_AT; break;
        case 12: steps = 4 * BK_AT; break;
        case 4: steps = b_copies<2>(); break;
        case 5: steps = b_copies<1>(); break;
        case 6: steps = A_COPIES4; break;
        case 7: steps = A_VECS; break;
        case 8: steps = 4 * A_VECS; break;
        case 13: steps = 2 * TM; break;
        case 14: steps = BM / (NT / 32); break;
        default: return SGEMM_ERR_INVALID_ARG;
    }
    if (n_warps) *n_warps = (kind == 11 || kind == 12) ? NT16 / 32 : NT / 32;
    if (n_steps) *n_steps = steps;
    if (n_stages) *n_stages = (kind == 2 || kind == 8) ? 2 : kind >= 13 ? 1 : kind >= 11 ? STAGES_AT : STAGES;
    return SGEMM_OK;
}

extern "C" int sgemm_f32_smem_request(int kind, int warp, int step, int stage, int64_t byte_offset[32],
                                      int *width_bytes) {
    int n_warps, n_steps, n_stages;
    if (sgemm_f32_smem_shape(kind, &n_warps, &n_steps, &n_stages) != SGEMM_OK) return SGEMM_ERR_INVALID_ARG;
    if (warp < 0 || warp >= n_warps || step < 0 || step >= n_steps || stage < 0 || stage >= n_stages ||
        byte_offset == nullptr)
        return SGEMM_ERR_INVALID_ARG;
    int width = 16;
    for (int lane = 0; lane < 32; ++lane) {
        const int tid = warp * 32 + lane;
        int word = 0, k = 0, x = 0;
        switch (kind) {
            case 0: a_copy16_coord(tid, step, x, k); word = ar_word(stage, x, k); width = 16; break;
            case 6: a_copy4_coord(tid, step, x, k); word = ar_word(stage, x, k); width = 4; break;
            case 1: b_copy_coord<4>(tid, step, k, x); word = bs_word(stage, k, x); width = 16; break;
            case 4: b_copy_coord<2>(tid, step, k, x); word = bs_word(stage, k, x); width = 8; break;
            case 5: b_copy_coord<1>(tid, step, k, x); word = bs_word(stage, k, x); width = 4; break;
            case 7: a_xpose_coord(tid, step, k, x); word = ar_word(stage, x, k); width = 16; break;
            case 8: a_xpose_coord(tid, step >> 2, k, x); word = as_word(stage, k + (step & 3), x); width = 4; break;
            case 2: word = as_word(stage, step >> 1, frag_row0(tid) + 16 * (step & 1)); width = 16; break;
            case 3: word = bs_word(stage, step >> 1, frag_col0(tid) + 32 * (step & 1)); width = 16; break;
            case 11: word = at_word(stage, step >> 1, frag16_row0(tid) + 32 * (step & 1)); width = 16; break;
            case 12: word = atb_word(stage, step >> 2, frag16_col0(tid) + 16 * (step & 3)); width = 16; break;
            case 13: pt_store_coord(tid, step, x, k); word = pt_word(x, k); width = 16; break;
            case 14: pt_sum_coord(tid, step, 0, x, k); word = pt_word(x, k); width = 16; break;
        }
        byte_offset[lane] = static_cast<int64_t>(word) * 4;
    }
    if (width_bytes) *width_bytes = width;
    return SGEMM_OK;
}

extern "C" int sgemm_f32_timeouts(unsigned *count) {
    if (count == nullptr) return SGEMM_ERR_NULL_PTR;
    if (cudaMemcpyFromSymbol(count, g_copy_timeout, sizeof(unsigned)) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    return SGEMM_OK;
}

extern "C" int sgemm_f32_wait_selftest(int which, unsigned polls, unsigned *timed_out) {
    if (timed_out == nullptr) return SGEMM_ERR_NULL_PTR;
    if (which < 0 || which > 3 || polls == 0 || polls > kSelftestMaxPolls) return SGEMM_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    DeviceInfo info;
    const int st = setup_device(dev, &info);
    if (st != SGEMM_OK) return st;
    unsigned *d = nullptr;
    if (cudaMalloc(&d, 3 * sizeof(unsigned)) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    int rc = SGEMM_OK;
    if (cudaMemset(d, 0, 3 * sizeof(unsigned)) != cudaSuccess) {
        rc = SGEMM_ERR_LAUNCH;
    } else {
        wait_selftest_kernel<<<1, 32>>>(which, polls, d);
        if (cudaGetLastError() != cudaSuccess || cudaMemcpy(timed_out, d, sizeof(unsigned), cudaMemcpyDeviceToHost) !=
                                                     cudaSuccess)
            rc = SGEMM_ERR_LAUNCH;
    }
    (void)cudaGetLastError();
    (void)cudaFree(d);
    return rc;
}

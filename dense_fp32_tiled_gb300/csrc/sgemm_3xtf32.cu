// sgemm_3xtf32.cu -- FP32 C = A.B on the 5th-generation tensor cores of GB300
// (sm_103a: tcgen05.mma with TMEM accumulators), by the 3xTF32 split.
//
// Each FP32 operand x is split into two TF32 values, hi = rna_tf32(x) and
// lo = rna_tf32(x - hi), so x = hi + lo + e with |e| <= 2^-22 |x|; then
//   A.B ~= Ahi.Bhi + (Ahi.Blo + Alo.Bhi)
// (the dropped Alo.Blo is below 2^-22 |a||b| per product).  The two groups
// accumulate in separate FP32 TMEM accumulators and are added in FP32 at
// the end.  The pages describe only the SIMT path (the textbook product
// C = A x B, vectorised-load page, "这一篇放进 GEMM 路径里看"); this is an
// additional implementation of the same product, checked against the same
// FP32 tolerance.
//
// Two kernels:
//   1. split: A -> A_hi, A_lo (M x Kp, row-major) and B -> Bt_hi, Bt_lo
//      (N x Kp: B transposed, so both operands are K-major), Kp = K rounded
//      up to 4, in the caller's workspace; the K padding is written as 0.
//   2. mma: one CTA per 128 x 128 tile of C.  One thread issues TMA copies
//      (128 x 32 boxes, 128-byte swizzle) of the four operand tiles into a
//      3-stage ring; one thread issues, per 8-deep K step,
//        main += Ahi.Bhi,  corr += Ahi.Blo,  corr += Alo.Bhi
//      (tcgen05.mma kind::tf32, M = 128, N = 128) and releases each stage
//      with tcgen05.commit; the accumulators restart every 256 K in one of two
//      tensor-memory buffer sets, and four warps add each finished block into
//      FP32 registers (tcgen05.ld) and finally store C.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

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
constexpr int TBM = 128, TBN = 128, TBK = 32;  // tile; 32 FP32 = one 128-byte swizzle row
constexpr int TSTAGES = 3;
constexpr int TILE_BYTES = TBM * TBK * 4;      // 16 KiB per operand tile (TBN == TBM)
constexpr int STAGE_BYTES = 4 * TILE_BYTES;    // A_hi, A_lo, Bt_hi, Bt_lo
constexpr int MMA_SMEM = TSTAGES * STAGE_BYTES + 1024;  // + alignment slack
constexpr int KBLK = 8;                        // K tiles (256 K) per tensor-memory block
constexpr int TMEM_COLS = 512;                 // 2 buffer sets x (main, corr) x 128 columns
constexpr int TC_THREADS = 192;                // warps 0-3 sum and store, 4 copies, 5 MMAs
constexpr uint32_t kWaitPolls = 1u << 22;
static_assert(TBM == TBN, "one tile size for both operands");

// Shared-memory matrix descriptor for a K-major operand tile of 128 rows x
// 128 bytes stored with the 128-byte swizzle (the layout a TMA copy with
// CU_TENSOR_MAP_SWIZZLE_128B writes): 8-row groups of 1024 bytes, start
// address in 16-byte units (bits 0-13), leading-dimension offset (bits 16-29,
// unused for this layout, set to 1), stride between 8-row groups (bits
// 32-45, 1024 bytes), descriptor version 1 (bits 46-47), base offset 0
// (1024-byte aligned tiles), layout 2 = 128-byte swizzle (bits 61-63).
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
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
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
// Bounded wait: gives up after kWaitPolls polls and records the timeout.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, unsigned *timeout_flag) {
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++polls > kWaitPolls) {
            *timeout_flag = 1u;
            break;
        }
    }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcMaps {
    CUtensorMap a_hi, a_lo, b_hi, b_lo;
};

// Warps 0-3 read tensor memory (warp w: lanes = tile rows 32w .. 32w+31),
// warp 4 lane 0 issues the copies, warp 5 owns the TMEM allocation and its
// lane 0 issues the MMAs.
//
// Tensor memory holds two buffer sets, each a (main, corr) pair of 128 x 128
// FP32 accumulators.  The K range is cut into blocks of KBLK K tiles; block b
// accumulates from zero in set b % 2, and warps 0-3 add each finished block
// (main + corr) into FP32 registers with round-to-nearest adds while the
// tensor core works on the next block.  The tensor core's own accumulation
// thus never runs over more than 256 K, which keeps its rounding bias from
// growing with K.
__global__ void __launch_bounds__(TC_THREADS, 1)
sgemm_3xtf32_kernel(const __grid_constant__ TcMaps maps, float *__restrict__ C, int ldc, int M, int N, int KT,
                    int tiles_m, int tiles_n, int vc, unsigned *timeout_flag) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[TSTAGES], empty_bar[TSTAGES], blk_full[2], blk_empty[2];
    __shared__ uint32_t tmem_base_slot;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = (KT + KBLK - 1) / KBLK;

    // rasterise 8 tile rows at a time
    const int per_group = 8 * tiles_n;
    const int g = blockIdx.x / per_group, first = g * 8;
    const int rows_in_group = (tiles_m - first) < 8 ? (tiles_m - first) : 8;
    const int r_in = blockIdx.x - g * per_group;
    const int tm = first + r_in % rows_in_group, tn = r_in / rows_in_group;
    const int m0 = tm * TBM, n0 = tn * TBN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&blk_full[b]), 1);
            mbar_init(smem_u32(&blk_empty[b]), 128);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "n"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = tmem_base_slot;

    if (warp == 4) {
        if (lane == 0) {  // copies
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % TSTAGES;
                if (kt >= TSTAGES) mbar_wait(smem_u32(&empty_bar[s]), ((kt / TSTAGES) - 1) & 1, timeout_flag);
                const uint32_t bar = smem_u32(&full_bar[s]);
                const uint32_t st = sbase + s * STAGE_BYTES;
                mbar_expect_tx(bar, STAGE_BYTES);
                tma_load_2d(st + 0 * TILE_BYTES, &maps.a_hi, kt * TBK, m0, bar);
                tma_load_2d(st + 1 * TILE_BYTES, &maps.a_lo, kt * TBK, m0, bar);
                tma_load_2d(st + 2 * TILE_BYTES, &maps.b_hi, kt * TBK, n0, bar);
                tma_load_2d(st + 3 * TILE_BYTES, &maps.b_lo, kt * TBK, n0, bar);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {  // MMAs
            constexpr uint32_t idesc = instr_desc_tf32(TBM, TBN);
            for (int kt = 0; kt < KT; ++kt) {
                const int b = kt / KBLK, set = b & 1;
                const bool block_start = kt % KBLK == 0;
                if (block_start && b >= 2) mbar_wait(smem_u32(&blk_empty[set]), ((b / 2) - 1) & 1, timeout_flag);
                const int s = kt % TSTAGES;
                mbar_wait(smem_u32(&full_bar[s]), (kt / TSTAGES) & 1, timeout_flag);
                asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
                const uint32_t t_main = tmem + set * 2 * TBN, t_corr = t_main + TBN;
                const uint32_t st = sbase + s * STAGE_BYTES;
#pragma unroll
                for (int j = 0; j < TBK / 8; ++j) {  // 8 TF32 = 32 bytes per MMA along K
                    const uint64_t ahi = smem_desc_sw128(st + 0 * TILE_BYTES + 32 * j);
                    const uint64_t alo = smem_desc_sw128(st + 1 * TILE_BYTES + 32 * j);
                    const uint64_t bhi = smem_desc_sw128(st + 2 * TILE_BYTES + 32 * j);
                    const uint64_t blo = smem_desc_sw128(st + 3 * TILE_BYTES + 32 * j);
                    const uint32_t acc = (!block_start || j > 0) ? 1u : 0u;
                    umma_tf32(t_main, ahi, bhi, idesc, acc);
                    umma_tf32(t_corr, ahi, blo, idesc, acc);
                    umma_tf32(t_corr, alo, bhi, idesc, 1u);
                }
                umma_commit(smem_u32(&empty_bar[s]));  // stage s free once these MMAs are done
                if (kt % KBLK == KBLK - 1 || kt == KT - 1) umma_commit(smem_u32(&blk_full[set]));
            }
        }
    } else {
        // warps 0-3: sum the blocks, then store C = sum
        float total[TBN];
#pragma unroll
        for (int c = 0; c < TBN; ++c) total[c] = 0.0f;
        const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
        for (int b = 0; b < NB; ++b) {
            const int set = b & 1;
            mbar_wait(smem_u32(&blk_full[set]), (b / 2) & 1, timeout_flag);
            __syncwarp();
            asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
            const uint32_t t_main = tmem + set * 2 * TBN + lane_off;  // corr follows at + TBN
#pragma unroll
            for (int c = 0; c < 2 * TBN; c += 32) {  // main columns, then corr columns
                float v[32];
                tmem_ld32(t_main + c, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
                for (int e = 0; e < 32; ++e) total[(c % TBN) + e] += v[e];
            }
            asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
            mbar_arrive(smem_u32(&blk_empty[set]));
        }
        const int row = m0 + 32 * warp + lane;
        if (row < M) {
            float *crow = C + static_cast<size_t>(row) * ldc + n0;
            const int left = N - n0;
            if (vc == 4 && left >= TBN) {
#pragma unroll
                for (int e = 0; e < TBN; e += 4)
                    *reinterpret_cast<float4 *>(crow + e) = make_float4(total[e], total[e + 1], total[e + 2], total[e + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < TBN; ++e)
                    if (e < left) crow[e] = total[e];
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    if (warp == 5) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(TMEM_COLS)
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
    const cuuint32_t box[2] = {TBK, TBM};
    const cuuint32_t ones[2] = {1, 1};
    return enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dim, stride, box, ones,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t region_bytes(long long rows, long long Kp) { return (static_cast<size_t>(rows * Kp) * 4 + 255) / 256 * 256; }

std::mutex g_setup_mutex;
int g_setup_state[64];

int setup(int dev) {
    if (dev < 0 || dev >= 64) return SGEMM_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_setup_state[dev] == 0) {
        int major = 0, minor = 0, st = SGEMM_OK;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
            minor != 3 ||
            cudaFuncSetAttribute(sgemm_3xtf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MMA_SMEM) !=
                cudaSuccess)
            st = SGEMM_ERR_DEVICE;
        if (st != SGEMM_OK) (void)cudaGetLastError();
        g_setup_state[dev] = st == SGEMM_OK ? 1 : st;
    }
    return g_setup_state[dev] > 0 ? SGEMM_OK : g_setup_state[dev];
}

// device-side timeout word of the last call, per library instance
__device__ unsigned g_tc_timeout;

}  // namespace

extern "C" size_t sgemm_f32_3xtf32_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const long long Kp = (static_cast<long long>(K) + 3) / 4 * 4;
    return 2 * region_bytes(M, Kp) + 2 * region_bytes(N, Kp);
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
    const long long tiles = ((static_cast<long long>(M) + TBM - 1) / TBM) * ((N + TBN - 1) / TBN);
    if (tiles > INT_MAX) return SGEMM_ERR_INVALID_DIM;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    const int st = setup(dev);
    if (st != SGEMM_OK) return st;

    const int Kp = (K + 3) / 4 * 4;
    char *ws = static_cast<char *>(workspace);
    float *a_hi = reinterpret_cast<float *>(ws);
    float *a_lo = reinterpret_cast<float *>(ws + region_bytes(M, Kp));
    float *bt_hi = reinterpret_cast<float *>(ws + 2 * region_bytes(M, Kp));
    float *bt_lo = reinterpret_cast<float *>(ws + 2 * region_bytes(M, Kp) + region_bytes(N, Kp));
    TcMaps maps;
    memset(&maps, 0, sizeof maps);
    if (!encode_operand(maps.a_hi, a_hi, M, Kp) || !encode_operand(maps.a_lo, a_lo, M, Kp) ||
        !encode_operand(maps.b_hi, bt_hi, N, Kp) || !encode_operand(maps.b_lo, bt_lo, N, Kp))
        return SGEMM_ERR_DEVICE;

    const int a_blocks = (M + 7) / 8;
    const int b_tiles_k = (Kp + ST - 1) / ST, b_tiles_n = (N + ST - 1) / ST;
    const long long split_blocks = static_cast<long long>(a_blocks) + static_cast<long long>(b_tiles_k) * b_tiles_n;
    if (split_blocks > INT_MAX) return SGEMM_ERR_INVALID_DIM;
    split_kernel<<<static_cast<unsigned>(split_blocks), dim3(32, 8), 0, stream>>>(
        A, lda, B, ldb, M, N, K, Kp, a_hi, a_lo, bt_hi, bt_lo, a_blocks, b_tiles_k);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    unsigned *timeout = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&timeout), g_tc_timeout) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    const int tiles_m = (M + TBM - 1) / TBM, tiles_n = (N + TBN - 1) / TBN;
    const int vc = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 4 == 0) ? 4 : 1;
    sgemm_3xtf32_kernel<<<static_cast<unsigned>(tiles), TC_THREADS, MMA_SMEM, stream>>>(
        maps, C, ldc, M, N, (Kp + TBK - 1) / TBK, tiles_m, tiles_n, vc, timeout);
    if (cudaPeekAtLastError() != cudaSuccess) {
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

// transpose_f32.cu -- FP32 matrix transpose out[j][i] = in[i][j] for GB300
// (sm_103a), the second workload of the shared-memory pages, and its C ABI
// (declared in include/transpose_f32.h).
//
// The bank page ("放进矩阵转置里看") stages a 32 x 32 tile in shared memory so
// that both the global read and the global write are coalesced, and pads the
// tile to [32][33] so that reading a column of it touches 32 different banks;
// "Padding 之外的选择" offers an XOR swizzle instead.  transpose_f32_layout
// runs that kernel shape with the three layouts (padded, unpadded control,
// swizzled) for measurement.  transpose_f32 is the same design scaled up for
// bandwidth: 64 x 64 tiles, 16 elements per thread, with 16-byte vector
// accesses and a chunk-swizzled tile when rows are 16-byte aligned, else
// scalar accesses and a [64][65] padded tile.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "transpose_f32.h"

namespace {

// ---- the pages' 32 x 32 tile kernel -------------------------------------
constexpr int T32 = 32;
constexpr int T32_ROWS = 8;  // block (32, 8): each thread moves 4 elements

// Word index of logical tile element (r, c) for each layout.
__host__ __device__ __forceinline__ int tile32_word(int layout, int r, int c) {
    switch (layout) {
        case TRANSPOSE_LAYOUT_PADDED: return r * (T32 + 1) + c;   // tile[32][33]
        case TRANSPOSE_LAYOUT_UNPADDED: return r * T32 + c;       // tile[32][32]
        default: return r * T32 + (c ^ r);                        // tile[r][c ^ r]
    }
}

template <int LAYOUT>
__global__ void __launch_bounds__(T32 *T32_ROWS) transpose_tile32_kernel(const float *__restrict__ in, int ld_in,
                                                                        float *__restrict__ out, int ld_out,
                                                                        int rows, int cols) {
    __shared__ float tile[LAYOUT == TRANSPOSE_LAYOUT_PADDED ? T32 * (T32 + 1) : T32 * T32];  // 4224 or 4096 B
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int c0 = blockIdx.x * T32, r0 = blockIdx.y * T32;
    // coalesced read of input rows, row-wise writes into the tile
#pragma unroll
    for (int j = 0; j < T32; j += T32_ROWS) {
        const int r = r0 + ty + j, c = c0 + tx;
        if (r < rows && c < cols) tile[tile32_word(LAYOUT, ty + j, tx)] = in[static_cast<size_t>(r) * ld_in + c];
    }
    __syncthreads();  // every thread reaches it, edge tiles included
    // column reads of the tile, coalesced writes of output rows
#pragma unroll
    for (int j = 0; j < T32; j += T32_ROWS) {
        const int orow = c0 + ty + j, ocol = r0 + tx;  // out[orow][ocol] = in[ocol][orow]
        if (orow < cols && ocol < rows)
            out[static_cast<size_t>(orow) * ld_out + ocol] = tile[tile32_word(LAYOUT, tx, ty + j)];
    }
}

// ---- bandwidth-oriented 64 x 64 kernel -----------------------------------
// The pages' kernel scaled up so that more bytes are in flight per SM: a
// 64 x 64 tile padded to [64][65] ("多一列": row stride 65 puts the 32
// consecutive rows of a column read in 32 different banks), block (32, 8),
// each thread moving 16 elements.  A warp reads and writes 128 contiguous
// bytes of one row per instruction on both sides; 4-byte accesses need no
// alignment class.
constexpr int TT = 64;         // tile rows and cols
constexpr int TT_STRIDE = TT + 1;
constexpr int TT_ROWS = 8;     // block (32, 8)

__host__ __device__ __forceinline__ int tt_word(int r, int c) { return r * TT_STRIDE + c; }

__global__ void __launch_bounds__(32 * TT_ROWS) transpose_f32_kernel(const float *__restrict__ in, int ld_in,
                                                                     float *__restrict__ out, int ld_out,
                                                                     int rows, int cols, int tiles_c) {
    __shared__ float tile[TT * TT_STRIDE];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int tr = blockIdx.x / tiles_c, tc = blockIdx.x - tr * tiles_c;
    const int r0 = tr * TT, c0 = tc * TT;
#pragma unroll
    for (int h = 0; h < TT; h += 32) {
#pragma unroll
        for (int j = 0; j < TT; j += TT_ROWS) {
            const int r = r0 + ty + j, c = c0 + tx + h;
            if (r < rows && c < cols) tile[tt_word(ty + j, tx + h)] = __ldg(in + static_cast<size_t>(r) * ld_in + c);
        }
    }
    __syncthreads();  // every thread reaches it, edge tiles included
#pragma unroll
    for (int h = 0; h < TT; h += 32) {
#pragma unroll
        for (int j = 0; j < TT; j += TT_ROWS) {
            const int orow = c0 + ty + j, ocol = r0 + tx + h;  // out[orow][ocol] = in[ocol][orow]
            if (orow < cols && ocol < rows)
                out[static_cast<size_t>(orow) * ld_out + ocol] = tile[tt_word(tx + h, ty + j)];
        }
    }
}

// ---- 16-byte vector kernel (aligned rows, sizes multiples of 4) -----------
// Same 64 x 64 tile and block, but every global access is a 16-byte vector:
// a warp reads 2 input rows x 256 bytes per instruction and writes 4 output
// rows x 128 bytes.  The tile is stored unpadded, its 16-byte chunks
// XOR-swizzled by row ("Padding 之外的选择"): element (r, c) at word
//   64 r + 4 ((c / 4) ^ ((r / 4) % 8)) + c % 4,
// so that the 128-bit tile writes of a quarter-warp cover 8 distinct chunk
// positions, and the scalar tile reads (lane l: rows 4(l/4) + e apart by 4,
// column 4j + l % 4) fall in 32 distinct banks.
__host__ __device__ __forceinline__ int tv_word(int r, int c) {
    return r * TT + 4 * ((c >> 2) ^ ((r >> 2) & 7)) + (c & 3);
}
// Thread t's q-th tile write: input row r, columns 4 c4 .. 4 c4 + 3.
__host__ __device__ __forceinline__ void tv_load_coord(int t, int q, int &r, int &c4) {
    const int idx = q * 256 + t;
    r = idx >> 4;
    c4 = idx & 15;
}
// Lane l of warp w, q-th output vector: output row (tile column) C, output
// columns (tile rows) 4 oc4 .. 4 oc4 + 3.
__host__ __device__ __forceinline__ void tv_store_coord(int w, int l, int q, int &C, int &oc4) {
    const int i = w * 4 + q;
    C = 4 * (i >> 1) + (l & 3);
    oc4 = (l >> 2) + 8 * (i & 1);
}

__global__ void __launch_bounds__(32 * TT_ROWS) transpose_f32_vec_kernel(const float *__restrict__ in, int ld_in,
                                                                         float *__restrict__ out, int ld_out,
                                                                         int rows, int cols, int tiles_c) {
    __shared__ __align__(16) float tile[TT * TT];
    const int t = threadIdx.y * 32 + threadIdx.x;
    const int tr = blockIdx.x / tiles_c, tc = blockIdx.x - tr * tiles_c;
    const int r0 = tr * TT, c0 = tc * TT;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        int r, c4;
        tv_load_coord(t, q, r, c4);
        if (r0 + r < rows && c0 + 4 * c4 < cols)
            *reinterpret_cast<float4 *>(tile + tv_word(r, 4 * c4)) =
                __ldg(reinterpret_cast<const float4 *>(in + static_cast<size_t>(r0 + r) * ld_in + c0 + 4 * c4));
    }
    __syncthreads();  // every thread reaches it, edge tiles included
    const int w = threadIdx.y, l = threadIdx.x;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        int C, oc4;
        tv_store_coord(w, l, q, C, oc4);
        if (c0 + C < cols && r0 + 4 * oc4 < rows) {
            const float4 v = make_float4(tile[tv_word(4 * oc4 + 0, C)], tile[tv_word(4 * oc4 + 1, C)],
                                         tile[tv_word(4 * oc4 + 2, C)], tile[tv_word(4 * oc4 + 3, C)]);
            *reinterpret_cast<float4 *>(out + static_cast<size_t>(c0 + C) * ld_out + r0 + 4 * oc4) = v;
        }
    }
}

bool overlap(const void *p, long long pb, const void *q, long long qb) {
    if (pb <= 0 || qb <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(q);
    return a0 < b0 + static_cast<uintptr_t>(qb) && b0 < a0 + static_cast<uintptr_t>(pb);
}

int check(int rows, int cols, const float *in, int ld_in, const float *out, int ld_out) {
    if (rows < 0 || cols < 0) return TRANSPOSE_ERR_INVALID_DIM;
    if (ld_in < (cols > 1 ? cols : 1) || ld_out < (rows > 1 ? rows : 1)) return TRANSPOSE_ERR_INVALID_LD;
    if (rows == 0 || cols == 0) return TRANSPOSE_OK;
    if (in == nullptr || out == nullptr) return TRANSPOSE_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(in) % 4 || reinterpret_cast<uintptr_t>(out) % 4) return TRANSPOSE_ERR_INVALID_ARG;
    const long long in_bytes = 4 * ((static_cast<long long>(rows) - 1) * ld_in + cols);
    const long long out_bytes = 4 * ((static_cast<long long>(cols) - 1) * ld_out + rows);
    if (overlap(in, in_bytes, out, out_bytes)) return TRANSPOSE_ERR_ALIAS;
    return TRANSPOSE_OK;
}

}  // namespace

extern "C" int transpose_f32(int rows, int cols, const float *in, int ld_in, float *out, int ld_out,
                             cudaStream_t stream) {
    const int st = check(rows, cols, in, ld_in, out, ld_out);
    if (st != TRANSPOSE_OK || rows == 0 || cols == 0) return st;
    const long long tiles_r = (rows + TT - 1) / TT, tiles_c = (cols + TT - 1) / TT;
    if (tiles_r * tiles_c > INT_MAX) return TRANSPOSE_ERR_INVALID_DIM;
    const bool vec = (reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 == 0 &&
                     ld_in % 4 == 0 && ld_out % 4 == 0 && rows % 4 == 0 && cols % 4 == 0;
    if (vec)
        transpose_f32_vec_kernel<<<static_cast<unsigned>(tiles_r * tiles_c), dim3(32, TT_ROWS), 0, stream>>>(
            in, ld_in, out, ld_out, rows, cols, static_cast<int>(tiles_c));
    else
        transpose_f32_kernel<<<static_cast<unsigned>(tiles_r * tiles_c), dim3(32, TT_ROWS), 0, stream>>>(
            in, ld_in, out, ld_out, rows, cols, static_cast<int>(tiles_c));
    return cudaPeekAtLastError() == cudaSuccess ? TRANSPOSE_OK : (cudaGetLastError(), TRANSPOSE_ERR_LAUNCH);
}

extern "C" int transpose_f32_layout(int rows, int cols, const float *in, int ld_in, float *out, int ld_out,
                                    int layout, cudaStream_t stream) {
    if (layout != TRANSPOSE_LAYOUT_PADDED && layout != TRANSPOSE_LAYOUT_UNPADDED &&
        layout != TRANSPOSE_LAYOUT_SWIZZLED)
        return TRANSPOSE_ERR_INVALID_ARG;
    const int st = check(rows, cols, in, ld_in, out, ld_out);
    if (st != TRANSPOSE_OK || rows == 0 || cols == 0) return st;
    const long long gx = (cols + T32 - 1) / T32, gy = (rows + T32 - 1) / T32;
    if (gx > INT_MAX || gy > 65535) return TRANSPOSE_ERR_INVALID_DIM;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), block(T32, T32_ROWS);
    switch (layout) {
        case TRANSPOSE_LAYOUT_PADDED:
            transpose_tile32_kernel<TRANSPOSE_LAYOUT_PADDED><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols);
            break;
        case TRANSPOSE_LAYOUT_UNPADDED:
            transpose_tile32_kernel<TRANSPOSE_LAYOUT_UNPADDED><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols);
            break;
        default:
            transpose_tile32_kernel<TRANSPOSE_LAYOUT_SWIZZLED><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols);
            break;
    }
    return cudaPeekAtLastError() == cudaSuccess ? TRANSPOSE_OK : (cudaGetLastError(), TRANSPOSE_ERR_LAUNCH);
}

extern "C" int transpose_f32_smem_request(int layout, int kind, int warp, int step, int64_t byte_offset[32],
                                          int *width_bytes) {
    if (byte_offset == nullptr || (kind != 0 && kind != 1) || warp < 0 || step < 0) return TRANSPOSE_ERR_INVALID_ARG;
    if (layout == TRANSPOSE_LAYOUT_FAST) {
        // block (32, 8): warp w is threadIdx.y == w; step s = 8 * h32 + j8 covers
        // tile rows (writes) or tile columns (reads) w + 8 * j8 at lane offset 32 * h32
        if (warp >= TT_ROWS || step >= (TT / 32) * (TT / TT_ROWS)) return TRANSPOSE_ERR_INVALID_ARG;
        const int h = 32 * (step / (TT / TT_ROWS)), j = TT_ROWS * (step % (TT / TT_ROWS));
        for (int lane = 0; lane < 32; ++lane) {
            const int word = kind == 0 ? tt_word(warp + j, lane + h) : tt_word(lane + h, warp + j);
            byte_offset[lane] = 4 * static_cast<int64_t>(word);
        }
        if (width_bytes) *width_bytes = 4;
        return TRANSPOSE_OK;
    }
    if (layout == TRANSPOSE_LAYOUT_FAST_VEC) {
        // kind 0: step q = 0..3, one 128-bit write per lane; kind 1: step
        // 4 q + e = 0..15, the scalar read of component e of the q-th vector
        if (warp >= TT_ROWS || step >= (kind == 0 ? 4 : 16)) return TRANSPOSE_ERR_INVALID_ARG;
        for (int lane = 0; lane < 32; ++lane) {
            int word;
            if (kind == 0) {
                int r, c4;
                tv_load_coord(warp * 32 + lane, step, r, c4);
                word = tv_word(r, 4 * c4);
            } else {
                int C, oc4;
                tv_store_coord(warp, lane, step >> 2, C, oc4);
                word = tv_word(4 * oc4 + (step & 3), C);
            }
            byte_offset[lane] = 4 * static_cast<int64_t>(word);
        }
        if (width_bytes) *width_bytes = kind == 0 ? 16 : 4;
        return TRANSPOSE_OK;
    }
    if (layout != TRANSPOSE_LAYOUT_PADDED && layout != TRANSPOSE_LAYOUT_UNPADDED &&
        layout != TRANSPOSE_LAYOUT_SWIZZLED)
        return TRANSPOSE_ERR_INVALID_ARG;
    if (warp >= T32_ROWS || step >= T32 / T32_ROWS) return TRANSPOSE_ERR_INVALID_ARG;
    // block (32, 8): warp w is threadIdx.y == w, lanes are threadIdx.x
    for (int lane = 0; lane < 32; ++lane) {
        const int r = warp + T32_ROWS * step;
        const int word = kind == 0 ? tile32_word(layout, r, lane) : tile32_word(layout, lane, r);
        byte_offset[lane] = 4 * static_cast<int64_t>(word);
    }
    if (width_bytes) *width_bytes = 4;
    return TRANSPOSE_OK;
}

extern "C" const char *transpose_f32_status_string(int status) {
    switch (status) {
        case TRANSPOSE_OK: return "success";
        case TRANSPOSE_ERR_INVALID_DIM: return "invalid dimension (negative rows or cols, or too many tiles)";
        case TRANSPOSE_ERR_INVALID_LD: return "invalid leading dimension (ld_in < max(1,cols) or ld_out < max(1,rows))";
        case TRANSPOSE_ERR_NULL_PTR: return "null pointer for a non-empty matrix";
        case TRANSPOSE_ERR_ALIAS: return "input and output overlap";
        case TRANSPOSE_ERR_LAUNCH: return "kernel launch rejected by the CUDA runtime";
        case TRANSPOSE_ERR_INVALID_ARG: return "invalid argument (misaligned pointer or unknown layout)";
        default: return "unknown status";
    }
}

// transpose_f32.cu -- FP32 matrix transpose out[j][i] = in[i][j] for GB300
// (sm_103a), the second workload of the shared-memory pages, and its C ABI
// (declared in include/transpose_f32.h).
//
// The bank page ("放进矩阵转置里看") stages a 32 x 32 tile in shared memory so
// that both the global read and the global write are coalesced, and pads the
// tile to [32][33] so that reading a column of it touches 32 different banks;
// "Padding 之外的选择" offers an XOR swizzle instead.  transpose_f32_layout
// runs that kernel shape with the three layouts (padded, unpadded control,
// swizzled) for measurement.  transpose_f32 is the bandwidth-oriented kernel:
// 64 x 64 tiles, 128-bit global loads and stores where the alignment class
// allows, and a tile stored k-major ("transposed on store", vectorised-load
// page) by 32-bit stores of 32 consecutive words, read back by 128-bit loads.
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
constexpr int TT = 64;        // tile rows and cols
constexpr int TNT = 256;      // threads
constexpr int TT_STRIDE = TT; // k-major tile row stride (floats)

// Load map: float4 q (0..3) of thread t covers input rows r = 32*(w & 1) + l
// (w = t / 32, l = t % 32) and columns 4*(4*(w >> 1) + q) .. +3: a warp load
// touches one 16-byte group in 32 consecutive rows, and the 4 components go
// to the k-major tile as 32-bit stores of 32 consecutive words.
__host__ __device__ __forceinline__ void tt_load_coord(int tid, int q, int &r, int &c) {
    const int w = tid >> 5, l = tid & 31;
    r = 32 * (w & 1) + l;
    c = 4 * (4 * (w >> 1) + q);
}
// k-major tile: logical (r, c) of the input tile at word c * TT_STRIDE + r.
__host__ __device__ __forceinline__ int tt_word(int r, int c) { return c * TT_STRIDE + r; }
// Store map: float4 q (0..3) of thread t is output row (tile column)
// c = 16q + t/16 and output columns (tile rows) 4*(t % 16) .. +3.
__host__ __device__ __forceinline__ void tt_store_coord(int tid, int q, int &c, int &r) {
    c = 16 * q + (tid >> 4);
    r = 4 * (tid & 15);
}

template <int VI, int VO>  // 4 or 1: 128-bit or 32-bit global access for in / out
__global__ void __launch_bounds__(TNT) transpose_f32_kernel(const float *__restrict__ in, int ld_in,
                                                            float *__restrict__ out, int ld_out, int rows,
                                                            int cols, int tiles_c) {
    __shared__ __align__(16) float tile[TT * TT_STRIDE];
    const int tid = threadIdx.x;
    const int tr = blockIdx.x / tiles_c, tc = blockIdx.x - tr * tiles_c;
    const int r0 = tr * TT, c0 = tc * TT;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        int r, c;
        tt_load_coord(tid, q, r, c);
        const int gr = r0 + r, gc = c0 + c;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (gr < rows) {
            const float *p = in + static_cast<size_t>(gr) * ld_in + gc;
            if (VI == 4 && gc + 3 < cols) {
                v = __ldg(reinterpret_cast<const float4 *>(p));
            } else {
                if (gc + 0 < cols) v.x = __ldg(p + 0);
                if (gc + 1 < cols) v.y = __ldg(p + 1);
                if (gc + 2 < cols) v.z = __ldg(p + 2);
                if (gc + 3 < cols) v.w = __ldg(p + 3);
            }
        }
        tile[tt_word(r, c + 0)] = v.x;
        tile[tt_word(r, c + 1)] = v.y;
        tile[tt_word(r, c + 2)] = v.z;
        tile[tt_word(r, c + 3)] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        int c, r;
        tt_store_coord(tid, q, c, r);
        const int orow = c0 + c, ocol = r0 + r;  // out[orow][ocol] = in[ocol][orow]
        if (orow >= cols) continue;
        const float4 v = *reinterpret_cast<const float4 *>(tile + tt_word(r, c));
        float *p = out + static_cast<size_t>(orow) * ld_out + ocol;
        if (VO == 4 && ocol + 3 < rows) {
            *reinterpret_cast<float4 *>(p) = v;
        } else {
            if (ocol + 0 < rows) p[0] = v.x;
            if (ocol + 1 < rows) p[1] = v.y;
            if (ocol + 2 < rows) p[2] = v.z;
            if (ocol + 3 < rows) p[3] = v.w;
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

int vec_class(const void *p, int ld) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 4 == 0) ? 4 : 1;
}

}  // namespace

extern "C" int transpose_f32(int rows, int cols, const float *in, int ld_in, float *out, int ld_out,
                             cudaStream_t stream) {
    const int st = check(rows, cols, in, ld_in, out, ld_out);
    if (st != TRANSPOSE_OK || rows == 0 || cols == 0) return st;
    const long long tiles_r = (rows + TT - 1) / TT, tiles_c = (cols + TT - 1) / TT;
    if (tiles_r * tiles_c > INT_MAX) return TRANSPOSE_ERR_INVALID_DIM;
    const int vi = vec_class(in, ld_in), vo = vec_class(out, ld_out);
    const dim3 grid(static_cast<unsigned>(tiles_r * tiles_c)), block(TNT);
    const int tc = static_cast<int>(tiles_c);
    if (vi == 4 && vo == 4) transpose_f32_kernel<4, 4><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols, tc);
    else if (vi == 4) transpose_f32_kernel<4, 1><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols, tc);
    else if (vo == 4) transpose_f32_kernel<1, 4><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols, tc);
    else transpose_f32_kernel<1, 1><<<grid, block, 0, stream>>>(in, ld_in, out, ld_out, rows, cols, tc);
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
        if (warp >= TNT / 32 || step >= (kind == 0 ? 16 : 4)) return TRANSPOSE_ERR_INVALID_ARG;
        for (int lane = 0; lane < 32; ++lane) {
            const int tid = warp * 32 + lane;
            int r, c;
            if (kind == 0) {  // 32-bit stores of component step % 4 of float4 step / 4
                tt_load_coord(tid, step >> 2, r, c);
                byte_offset[lane] = 4 * static_cast<int64_t>(tt_word(r, c + (step & 3)));
            } else {  // 128-bit reads
                tt_store_coord(tid, step, c, r);
                byte_offset[lane] = 4 * static_cast<int64_t>(tt_word(r, c));
            }
        }
        if (width_bytes) *width_bytes = kind == 0 ? 4 : 16;
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

/*
 * transpose_f32.h -- C ABI of the GB300 (sm_103a) FP32 matrix transpose, the
 * second workload of the shared-memory pages (libsgemm_f32.so).
 *
 * Operation (page "Memory Bank 机制与加速计算", section "放进矩阵转置里看"):
 *
 *     out[j*ld_out + i] = in[i*ld_in + j]   for 0 <= i < rows, 0 <= j < cols,
 *
 * i.e. a rows x cols row-major input becomes a cols x rows row-major output.
 * Pure data movement: results are bit-exact (NaN payloads and signed zeros
 * included).  Input and output must not overlap.
 *
 * All functions are thread-safe, allocate nothing, and check their arguments
 * on the host before any launch: an invalid call returns its error code
 * without touching the GPU.  Launches are asynchronous on `stream`; faults
 * surface at the caller's next synchronisation.
 */
#ifndef TRANSPOSE_F32_H
#define TRANSPOSE_F32_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TRANSPOSE_OK = 0,
    TRANSPOSE_ERR_INVALID_DIM = -1,  /* rows or cols negative, or the grid too large */
    TRANSPOSE_ERR_INVALID_LD = -2,   /* ld_in < max(1,cols) or ld_out < max(1,rows) */
    TRANSPOSE_ERR_NULL_PTR = -3,     /* NULL pointer for a non-empty matrix */
    TRANSPOSE_ERR_ALIAS = -4,        /* input and output address ranges overlap */
    TRANSPOSE_ERR_LAUNCH = -5,       /* the kernel launch was rejected */
    TRANSPOSE_ERR_INVALID_ARG = -7   /* misaligned pointer (not 4-byte) or unknown layout */
} transpose_status;

/* Shared-memory layouts of the pages' 32 x 32 tile kernel, and the tile of
 * the bandwidth-oriented kernel (for transpose_f32_smem_request). */
typedef enum {
    TRANSPOSE_LAYOUT_PADDED = 0,    /* tile[32][33]: +1 padding ("多一列") */
    TRANSPOSE_LAYOUT_UNPADDED = 1,  /* tile[32][32]: the control, 32-way column conflicts */
    TRANSPOSE_LAYOUT_SWIZZLED = 2,  /* tile[r][c ^ r] ("Padding 之外的选择") */
    TRANSPOSE_LAYOUT_FAST = 3,      /* transpose_f32's scalar path: 64 x 64 tile padded to [64][65] */
    TRANSPOSE_LAYOUT_FAST_VEC = 4   /* transpose_f32's 16-byte path: 64 x 64 tile, 16-byte chunks
                                       of row r XOR-swizzled by (r / 4) % 8 */
} transpose_layout;

/*
 * transpose_f32 -- out = in^T, the fast path.
 *   rows, cols : input sizes (>= 0); rows == 0 or cols == 0 is a no-op.
 *   in, ld_in  : DEVICE pointer, row-major rows x cols, row i at in + i*ld_in,
 *                ld_in >= max(1, cols).
 *   out, ld_out: DEVICE pointer, row-major cols x rows, row j at out + j*ld_out,
 *                ld_out >= max(1, rows); elements past `rows` in each row are
 *                not touched.
 * Any 4-byte alignment is accepted.  The kernel is the pages' shape scaled up
 * for bandwidth: 64 x 64 tiles, block (32, 8).  When in and out are 16-byte
 * aligned and ld_in, ld_out, rows and cols are multiples of 4, every global
 * access is a 16-byte vector and the tile's 16-byte chunks are XOR-swizzled
 * (TRANSPOSE_LAYOUT_FAST_VEC); otherwise accesses are 4-byte and the tile is
 * padded to [64][65] (TRANSPOSE_LAYOUT_FAST).
 */
int transpose_f32(int rows, int cols, const float *in, int ld_in, float *out, int ld_out,
                  cudaStream_t stream);

/*
 * transpose_f32_layout -- the pages' kernel shape (block (32, 8), one 32 x 32
 * tile per block, a barrier between the row-wise tile writes and the
 * column-wise tile reads) with shared layout `layout` (PADDED, UNPADDED or
 * SWIZZLED), for measuring what the layout alone changes.  Same arguments,
 * results and errors as transpose_f32.
 */
int transpose_f32_layout(int rows, int cols, const float *in, int ld_in, float *out, int ld_out,
                         int layout, cudaStream_t stream);

/*
 * transpose_f32_smem_request -- host-only description of one warp-wide
 * shared-memory access of a transpose kernel, from the same index functions
 * the kernel uses, for checking the layout against the bank rule
 * bank = (byte_address / 4) % 32.  Touches no GPU.
 *   layout : PADDED, UNPADDED or SWIZZLED (32 x 32 kernel: warp 0..7, step
 *            0..3), FAST (64 x 64 scalar kernel: warp 0..7, step 0..15) or
 *            FAST_VEC (64 x 64 vector kernel: warp 0..7, step 0..3 for
 *            kind 0, 0..15 for kind 1).
 *   kind   : 0 = the tile write that follows the global read,
 *            1 = the tile read that precedes the global write.
 *   byte_offset[32] (out): byte offset each lane touches in the tile.
 *   width_bytes (out): bytes per lane access (16 for FAST_VEC writes, else 4).
 * Returns TRANSPOSE_OK or TRANSPOSE_ERR_INVALID_ARG.
 */
int transpose_f32_smem_request(int layout, int kind, int warp, int step, int64_t byte_offset[32],
                               int *width_bytes);

/* Static English description of a status code (never NULL). */
const char *transpose_f32_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* TRANSPOSE_F32_H */

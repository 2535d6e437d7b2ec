/*
 * sgemm_f32.h -- C ABI of the GB300 (sm_103a) tiled FP32 matrix multiply.
 *
 * Operation (the textbook product the tiled kernel computes; page
 * "CUDA 深入浅出（五）: Vectorized Load 和 Shared Memory Layout", section
 * "这一篇放进 GEMM 路径里看"):
 *
 *     C[i*ldc + j] = sum_{k<K} A[i*lda + k] * B[k*ldb + j]
 *                    for 0 <= i < M, 0 <= j < N,
 *
 * with FP32 inputs, FP32 fused multiply-adds and an FP32 result.  lda, ldb
 * and ldc are row strides in elements (same page, section
 * "对齐也要从数据分配开始": the leading dimension fixes where each row starts,
 * and with it which rows allow 16-byte vector access).  C is overwritten;
 * there is no alpha/beta scaling and no transposed-operand mode.  Rounding:
 * IEEE round-to-nearest FMA, denormals kept; the summation order over k is
 * unspecified, so results agree with an exact dot product to FP32 rounding,
 * not bit for bit with another order.
 *
 * All functions are thread-safe (calls of sgemm_f32_static_scratch that
 * overlap on the GPU share its scratch: see there).  No product entry point
 * allocates device memory; only the two wait self-tests allocate (and free)
 * a few bytes.  The first call on a device sets up that device's kernel
 * attributes (once, under a lock).  That set-up belongs to the CUDA context
 * current at the time: after cudaDeviceReset the next call sets up again.
 */
#ifndef SGEMM_F32_H
#define SGEMM_F32_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_DIM = -1,  /* M, N or K negative, or the tile grid too large */
    SGEMM_ERR_INVALID_LD = -2,   /* lda < max(1,K), ldb < max(1,N) or ldc < max(1,N) */
    SGEMM_ERR_NULL_PTR = -3,     /* a pointer is NULL although its matrix is not empty */
    SGEMM_ERR_ALIAS = -4,        /* C's address range overlaps A's or B's */
    SGEMM_ERR_LAUNCH = -5,       /* the kernel launch was rejected by the runtime */
    SGEMM_ERR_DEVICE = -6,       /* current device is not sm_103 or its set-up failed */
    SGEMM_ERR_INVALID_ARG = -7,  /* any other out-of-range argument */
    SGEMM_ERR_SCRATCH_LIMIT = -8 /* sgemm_f32_static_scratch: more tiles than its fixed scratch holds */
} sgemm_status;

/*
 * sgemm_f32 -- enqueue C = A.B on `stream`.
 *
 *   M, N, K : sizes; A is M x K, B is K x N, C is M x N.  Each >= 0.
 *   A, lda  : DEVICE pointer to row-major A, row i at A + i*lda; lda >= max(1,K).
 *   B, ldb  : DEVICE pointer to row-major B, row k at B + k*ldb; ldb >= max(1,N).
 *   C, ldc  : DEVICE pointer to row-major C, row i at C + i*ldc; ldc >= max(1,N).
 *             Elements between N and ldc in each row are not touched.
 *   stream  : CUDA stream of the current device (0 = legacy default stream).
 *
 * Any pointer alignment (a multiple of 4 bytes) is accepted: the library
 * picks 16-, 8- or 4-byte copy widths from the alignment of each pointer and
 * its row stride.  The caller owns all memory; A and B are only read, C is
 * only written.  C must not overlap A or B (checked on address ranges).
 *
 * Schedule: one CTA per 128 x 128 output tile; or, for products with at
 * most G / 2 tiles (G = 2 CTAs per SM) and at least 4 K tiles of 16, the
 * cluster split of K: each tile runs on a thread-block cluster of S CTAs
 * (S = min(G / tiles, C, K tiles / 2), C = 8, the portable cluster size, or
 * 16 for at most 4 tiles where the GPU can schedule clusters of 16 of these
 * CTAs), CTA r summing K tiles
 * [KT r / S, KT (r+1) / S); the S partial tiles stay in shared memory and
 * are added in rank order over distributed shared memory, so the result does
 * not depend on timing.  Either way one kernel launch, no device memory.  If
 * the runtime refuses the cluster launch, the call runs one CTA per tile
 * instead (sgemm_f32_ws: the schedule it would run without the split).
 *
 * Edge cases: M == 0 or N == 0 returns SGEMM_OK without launching anything.
 * K == 0 sets C to zero (the empty sum); A and B may then be NULL.
 *
 * Errors: the arguments are checked on the host before anything is launched,
 * and an invalid call returns its error code without touching the GPU.  A
 * rejected launch returns SGEMM_ERR_LAUNCH.  The call is asynchronous:
 * faults during execution surface at the caller's next synchronisation.
 */
int sgemm_f32(int M, int N, int K,
              const float *A, int lda,
              const float *B, int ldb,
              float *C, int ldc,
              cudaStream_t stream);

/*
 * sgemm_f32_ws -- the same product, allowed to use a caller-provided device
 * workspace for a better-balanced schedule.
 *
 *   workspace       : DEVICE pointer, 16-byte aligned, or NULL (then
 *                     workspace_bytes must be 0); must not overlap A, B or C.
 *   workspace_bytes : its size.  sgemm_f32_workspace_size(M, N, K) is enough
 *                     for every schedule below;
 *                     sgemm_f32_workspace_size_for(M, N, K, A, lda, B, ldb)
 *                     also makes room for the operand copies below where
 *                     they pay.
 *
 * When the workspace is large enough, the call balances the work over the
 * CTAs the GPU holds at once (G = 2 per SM).  Every output tile (128 x 128)
 * cut into K parts is summed in a fixed order, so results are deterministic.
 * The schedules (sgemm_f32_ws_schedule reports which one a call uses):
 *   1  more tiles than G, not a whole number of waves, rows not 16-byte
 *      aligned: a persistent grid splits the last wave and a bit, with partial
 *      sums handed over through C (the workspace holds one flag per tile plus
 *      an error word);
 *   2  fewer tiles than G: a persistent grid splits every tile into several K
 *      parts (at least 4 K slices per CTA), with partial sums handed over
 *      through 64 KiB slots in the workspace (one flag and one slot per CTA,
 *      plus an error word);
 *   3  more tiles than G, not a whole number of waves, rows 16-byte aligned:
 *      one CTA per tile for the whole waves, and the R = T mod G leftover
 *      tiles cut into S K parts each (S = 4 to 8) in a second grid that starts
 *      as SMs free up; the part that finishes a tile last adds all parts
 *      (one count per leftover tile, then S * R slots of 64 KiB).
 *   0  otherwise, or with a smaller workspace: exactly as sgemm_f32.
 * The cluster split of K (see sgemm_f32) takes precedence where it applies,
 * except over schedule 2 where a cost model fitted to GB300 timings expects
 * schedule 2 to be faster: the split costs its CTAs' K tiles plus about 4.7
 * K tiles of fixed cost; schedule 2 its CTAs' (fewer) K tiles plus about 7.5
 * and 0.3 K tile per part of a tile (flag reset, hand-over waits, the serial
 * sum of the parts); a grid that fills at most half the SMs runs its K tiles
 * about twice as fast per CTA.  The split uses no workspace.
 * sgemm_f32_workspace_size reports the bytes for the current device.  The
 * call zero-fills the words it uses at the start of the workspace on
 * `stream` before the kernels, so the workspace needs no preparation and its
 * contents are not preserved; calls that share one workspace must not overlap
 * in time.  After a successful call those words are zero again.  In
 * schedules 1 and 2 the last of them is an error word, nonzero only if a CTA
 * gave up waiting for a partner (about a second; the result is then wrong,
 * nothing hangs); in schedule 3 no CTA waits for another.
 * Operand copies (K > 0 and 2*M*N*K >= 2e9: smaller products run faster on
 * the narrower copies of the kernels themselves, measured on GB300; each copy
 * is one kernel, HBM-bound, placed after the schedule's words in the
 * workspace):
 *   k-major A: when the k-major copy pays (large N, see
 *      sgemm_f32_workspace_size_for) or A's rows are not 16-byte aligned
 *      (pointer or lda), and the workspace has room for the schedule plus
 *      At = A^T (K rows of M floats, row stride M rounded up to 4) plus the
 *      repacked B below if B needs it, the call first transposes A into At
 *      (the transpose_f32 kernel) and runs kernels that load k-major A tiles
 *      straight into the layout the FMA loop reads (128-thread CTAs, 8 x 16
 *      register tiles, K tiles 32 deep): no transpose in shared memory and
 *      no shared store in the K loop.  With one CTA per tile the summation
 *      order is unchanged, so the result equals the call without the copy
 *      bit for bit; the split schedules cut K at multiples of 32 instead of
 *      16, so there the two agree within FP32 rounding.
 *   repacked rows: otherwise, when A's or B's rows are not 16-byte aligned
 *      and the workspace has room for the schedule plus a copy of that
 *      operand with 16-byte aligned rows (leading dimension rounded up to 4),
 *      the call first copies it there and runs the 16-byte-aligned kernels and
 *      schedules on the copy.
 *   Without the room it runs the narrower-copy kernels on the operands
 *   themselves.
 * Other argument checks and errors are those of sgemm_f32, plus
 * SGEMM_ERR_ALIAS for a workspace overlapping A, B or C and
 * SGEMM_ERR_INVALID_ARG for a misaligned workspace.
 */
int sgemm_f32_ws(int M, int N, int K,
                 const float *A, int lda,
                 const float *B, int ldb,
                 float *C, int ldc,
                 void *workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/* What sgemm_f32_ws would run for these arguments on the current device
 * with a workspace of workspace_bytes bytes (host-only; launches nothing):
 * *kind = the schedule (0 to 3, as listed above) in bits 0-1, plus 4 if A is
 * repacked, 8 if B is repacked, 16 if A is transposed into its k-major copy
 * and 32 for the cluster split of K (then bits 0-1 are 0, bits 8-12 hold
 * the cluster size S and *words is 0);
 * with workspace_bytes = 0 it reports what sgemm_f32 runs.
 * *words = the 32-bit words at the start of
 * the workspace that the call zero-fills and leaves zero on success (flags
 * and error word, or tile counts).  Returns the argument-check status of
 * sgemm_f32_ws, or SGEMM_ERR_DEVICE without a usable device. */
int sgemm_f32_ws_schedule(int M, int N, int K,
                          const float *A, int lda,
                          const float *B, int ldb,
                          const float *C, int ldc,
                          size_t workspace_bytes,
                          int *kind, long long *words);

/* Workspace bytes sgemm_f32_ws can use for this shape on the current device
 * (0 for an empty or invalid shape), not counting the operand copies.  Reads
 * device attributes only; with no usable device it returns the size of the
 * flags-only schedule. */
size_t sgemm_f32_workspace_size(int M, int N, int K);

/* Workspace bytes for these operands: sgemm_f32_workspace_size(M, N, K), or
 * more, enough for the operand copies of sgemm_f32_ws, in two cases:
 *   - A's or B's rows are not 16-byte aligned and the product has at least
 *     2 GFLOP (2*M*N*K): room for the k-major copy of an unaligned A and the
 *     repacked copy of an unaligned B (smaller products copy nothing);
 *   - the k-major copy of A pays: its expected saving, 6 % of the
 *     product's time at 68 TFLOP/s, exceeds 1.2 times the transpose's time
 *     (8*M*K bytes at 5.5 TB/s plus 4 us).  This holds for large N (4096^3:
 *     69.3 -> 73.0 TFLOP/s measured on GB300; 2048^3: 62.1 -> 64.4), not for
 *     16384 x 256 x 4096 or 1024^3.
 * The pointers are only inspected for alignment. */
size_t sgemm_f32_workspace_size_for(int M, int N, int K,
                                    const float *A, int lda,
                                    const float *B, int ldb);

/*
 * sgemm_f32_host -- the same product for operands in HOST memory: copies A
 * and B to the device, multiplies with sgemm_f32_ws, and copies C back.
 * A goes in row panels: for wide products (N >= 2048, M >= 3072) a first
 * panel of 1024 rows, one panel up to the last 512 rows and a last panel of
 * 512 rows; otherwise panels of about 1024 rows (at most 4, the last one cut
 * in two when it has at least 512 rows).  B goes after the first panel, and
 * each panel's product starts as soon as that panel and B have landed; with
 * several panels and N >= 512 the first panel's product runs in column
 * blocks of B (4 when N >= 1024, else 2), each while the next block of B is
 * still copying.
 * Each finished panel of C is copied back while the next one computes.  The
 * copies run on two internal non-blocking streams (created once per device),
 * the products on `stream`.  The pages have no counterpart: this entry point
 * is the path's public interface for host-resident data.
 *   A, B, C, M, N, K, lda, ldb, ldc : as for sgemm_f32, but HOST pointers.
 *                     Page-locked memory gives asynchronous copies at full
 *                     speed; pageable memory works, staged by the runtime.
 *   workspace       : DEVICE pointer, 256-byte aligned, at least
 *                     sgemm_f32_host_workspace_size(M,N,K) bytes.  It holds
 *                     device copies of B, A and C, their rows padded to a
 *                     multiple of 4 floats (16-byte aligned), and the products'
 *                     own workspace (with room for the k-major copy of a panel
 *                     of A where that pays, see sgemm_f32_workspace_size_for).
 *                     Its contents are not preserved, and calls sharing a
 *                     workspace are ordered by `stream`.
 *   stream          : work queued on `stream` before the call completes
 *                     before the workspace is touched; work queued after
 *                     the call sees C complete in host memory.  The host
 *                     buffers must stay valid and unchanged until then
 *                     (e.g. cudaStreamSynchronize(stream)).
 * Returns the status codes of sgemm_f32_ws, plus SGEMM_ERR_INVALID_ARG for a
 * missing, misaligned or too small workspace, and SGEMM_ERR_LAUNCH when a copy
 * cannot be queued.
 */
int sgemm_f32_host(int M, int N, int K,
                   const float *A, int lda,
                   const float *B, int ldb,
                   float *C, int ldc,
                   void *workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/* Device workspace bytes sgemm_f32_host needs (0 for an empty or invalid
 * shape).  Reads device attributes only. */
size_t sgemm_f32_host_workspace_size(int M, int N, int K);

/*
 * sgemm_f32_static_scratch -- the sgemm_f32_ws product for callers that
 * cannot allocate device memory.
 *
 * This call has no counterpart on the pages; it exists for callers that are
 * not allowed to allocate.  Examples are code whose device memory is wholly
 * owned by another allocator (a framework's caching pool or a fixed budget
 * set up at start-up), and latency-critical paths that must not risk the
 * implicit device-wide synchronisation a cudaFree can bring.  It allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.  The
 * caller still passes A, B and C exactly as for sgemm_f32, with the same
 * meaning, checks and error codes.
 *
 * The scratch that sgemm_f32_ws takes from the caller (one flag per 128 x 128
 * output tile plus an error word) lives here in a fixed array inside the
 * library, of 16384 32-bit words (64 KiB).  Every GPU that loads the library
 * holds it until the process exits.  Problems with more than 16383 output
 * tiles (ceil(M/128) * ceil(N/128); e.g. M = N = 16256 fits, 16384 does not)
 * are rejected with SGEMM_ERR_SCRATCH_LIMIT before anything is launched.
 *
 * Small products that take the cluster split of K (see sgemm_f32) use none
 * of it.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it, so it costs more than later calls.  The
 * address belongs to the CUDA context it was looked up in: a call made in a
 * new context of the device (after cudaDeviceReset, for instance) looks it up
 * again.  Every call shares the one array, which keeps whatever the last call
 * left there: each call zero-fills the words it uses on `stream` before its
 * kernel, and calls that overlap on the GPU (different streams, or different
 * host threads) race on the array and must not be issued.
 */
int sgemm_f32_static_scratch(int M, int N, int K,
                             const float *A, int lda,
                             const float *B, int ldb,
                             float *C, int ldc,
                             cudaStream_t stream);

/*
 * sgemm_f32_3xtf32 -- the same product on the tensor cores (tcgen05.mma,
 * TF32 inputs, FP32 accumulation in tensor memory), by the 3xTF32 split:
 * each FP32 operand x becomes hi = round_to_nearest_tf32(x) and
 * lo = round_to_nearest_tf32(x - hi), and C = Ahi.Bhi + Ahi.Blo + Alo.Bhi.
 * The tensor cores accumulate each 128-deep K block from zero; the blocks are
 * added in FP32 with round-to-nearest.  The pages describe only the CUDA-core
 * path; this variant of the same product meets the same FP32 acceptance bound
 * as sgemm_f32 but is not bit-identical to it (different rounding of the
 * partial sums).
 *
 *   A, B, C, M, N, K, lda, ldb, ldc : as for sgemm_f32 (any 4-byte alignment).
 *   workspace       : DEVICE pointer, 256-byte aligned, not overlapping A, B
 *                     or C, at least sgemm_f32_3xtf32_workspace_size(M,N,K)
 *                     bytes: it receives the split operands A_hi, A_lo (M x Kp)
 *                     and the transposed B_hi, B_lo (N x Kp), Kp = K rounded
 *                     up to 4.  Its contents are not preserved.
 *   stream          : CUDA stream; two kernels are enqueued (split, MMA).
 *
 * Errors are those of sgemm_f32, plus SGEMM_ERR_INVALID_ARG for a missing,
 * misaligned or too small workspace and SGEMM_ERR_DEVICE when no tensor map
 * can be encoded.  K == 0 writes C = 0 as sgemm_f32 does.  Every wait inside
 * the kernel is bounded: a wait that runs out (about a second) leaves C wrong
 * and sets the flag sgemm_f32_3xtf32_timeouts reports; nothing hangs.
 */
int sgemm_f32_3xtf32(int M, int N, int K,
                     const float *A, int lda,
                     const float *B, int ldb,
                     float *C, int ldc,
                     void *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* Workspace bytes sgemm_f32_3xtf32 needs (0 for an empty shape).  Host-only. */
size_t sgemm_f32_3xtf32_workspace_size(int M, int N, int K);

/* Copies into *count whether any tensor-core kernel on the current device gave
 * up a wait since the library was loaded (0 = never).  Synchronous. */
int sgemm_f32_3xtf32_timeouts(unsigned *count);

/* Copies into *count whether any CUDA-core kernel on the current device gave
 * up waiting for a tensor copy of its ring since the library was loaded
 * (0 = never; the product of that call is then wrong, nothing hangs).  The
 * wait allows about a second.  Synchronous. */
int sgemm_f32_timeouts(unsigned *count);

/* Failure-detection self-tests (the pages have no counterpart).  Each runs, in
 * a one-CTA kernel, one of the library's bounded waits with a limit of
 * `polls` polls (1 .. 65536) and stores into *timed_out 1 if the wait gave up,
 * else 0.  The target is either one that nothing ever completes (the wait must
 * give up and return; the kernel exits normally and the context stays usable)
 * or one already complete (the wait must not give up):
 *   sgemm_f32_wait_selftest, which = 0: a copy-ring mbarrier phase with no
 *     arrival and no copy; 1: a stream-K partner flag nobody raises;
 *     2: the phase after an arrival; 3: a raised flag.
 *   sgemm_f32_3xtf32_wait_selftest, which = 0: a tensor-core pipeline
 *     mbarrier phase with no arrival; 1: the phase after an arrival.
 * They leave the flags of sgemm_f32_timeouts and sgemm_f32_3xtf32_timeouts
 * alone.  Synchronous (they allocate and free 12 bytes of device memory).
 * SGEMM_ERR_INVALID_ARG for another `which` or a limit out of range. */
int sgemm_f32_wait_selftest(int which, unsigned polls, unsigned *timed_out);
int sgemm_f32_3xtf32_wait_selftest(int which, unsigned polls, unsigned *timed_out);

/* Static English description of a status code (never NULL). */
const char *sgemm_f32_status_string(int status);

/*
 * sgemm_f32_smem_request -- host-only description of the kernel's
 * shared-memory accesses, for checking its layout against the bank rule
 * bank = (byte_address / 4) % 32 (page "Memory Bank 机制与加速计算",
 * sections "地址怎样落到 bank" and "为什么 double 和 float4 要另算").
 * Touches no GPU.
 *
 *   kind : 0 = A tile copy into the raw staging tile (16-byte copies),
 *          6 = the same, 4-byte copies (misaligned A rows),
 *          1 = B tile copy (16-byte copies), 4 = 8-byte, 5 = 4-byte class,
 *          7 = A transpose read (raw tile -> registers, 16-byte),
 *          8 = A transpose store (registers -> k-major tile, 4-byte),
 *          2 = A fragment read (16-byte), 3 = B fragment read (16-byte);
 *          with the k-major copy of A (no transpose, a 3-deep ring, 8 x 16
 *          register tiles, 4 warps): 11 = A fragment read from the ring
 *          stage, 12 = B fragment read;
 *          the cluster split of K (one stage): 13 = a CTA's store of its
 *          partial 128 x 128 tile, 14 = the read of one row of a partial
 *          tile when the cluster sums them (the rows from 0 on; a CTA's
 *          range starts at another row, which shifts every lane alike).
 *   warp : warp index in the CTA, 0 <= warp < *n_warps.
 *   step : which instruction of that warp, 0 <= step < *n_steps (copies,
 *          transpose reads and stores: index within one tile; fragment
 *          reads: 2*k + half, k < BK; kind 12: 4*k + quarter; kind 13:
 *          2*i + half, row i of the thread's 8 x 8 tile; kind 14: the j-th
 *          row of the warp, row 8*j + warp).
 *   stage: ring stage (copies, transpose reads, B reads, kinds 11 and 12)
 *          or k-major buffer (A reads, transpose stores) the access targets,
 *          0 <= stage < *n_stages.
 *   byte_offset[32] (out): shared-memory byte offset each lane touches,
 *          relative to the start of the dynamic shared-memory block.
 *   width_bytes (out): bytes each lane moves (4, 8 or 16).
 *
 * sgemm_f32_smem_shape reports the valid ranges for a kind.  Both return
 * SGEMM_OK or SGEMM_ERR_INVALID_ARG.
 */
int sgemm_f32_smem_shape(int kind, int *n_warps, int *n_steps, int *n_stages);
int sgemm_f32_smem_request(int kind, int warp, int step, int stage,
                           int64_t byte_offset[32], int *width_bytes);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_F32_H */

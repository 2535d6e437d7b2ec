/*
 * smem_bank_probe.h -- C ABI of the shared-memory stride sweep (libsgemm_f32.so).
 *
 * The bank page ("Memory Bank 机制与加速计算") states how a warp's 32-bit
 * shared-memory accesses fall on the 32 banks: word w sits in bank w % 32
 * ("地址怎样落到 bank"), and a warp whose lane l touches word l * stride
 * reaches 32 / gcd(stride, 32) distinct banks, each gcd(stride, 32) times, so
 * the access is served in gcd(stride, 32) passes ("四种访问，四种结果").  Its
 * section "把推导变成测量" asks for that derivation to be checked by
 * measurement.  This probe measures it on the running GPU: one CTA of
 * `warps` warps repeats the access `iters` times per warp, and the SM's own
 * cycle counter times the whole loop.
 *
 *   int smem_bank_stride_probe(int stride, int op, int warps, int iters,
 *                              double *cycles_per_access, long long *checksum);
 *
 *   stride : 1 .. 64, the word stride between consecutive lanes.
 *   op     : 0 = 32-bit loads, 1 = 32-bit stores.
 *   warps  : 1 .. 8 warps in the CTA (8, two per scheduler, keep the
 *            shared-memory pipe busy even at stride 1).
 *   iters  : 64 .. 65536 accesses per warp (a multiple of 64).
 *   Access j of every warp's lane l touches word l * stride + 32 * (j % 64)
 *   (below 4096) of a 4096-word int array s[] that holds s[i] = i before the
 *   loop (loads), or -1 (stores, which write the word's own index).  The
 *   accesses are volatile: each one is issued, none merged or moved.
 *   *cycles_per_access (out): SM clock cycles from the barrier before the
 *       loop to the barrier after it, divided by warps * iters: about the
 *       passes one warp-wide access needs when the shared-memory pipe is the
 *       bottleneck.
 *   *checksum (out): loads: the sum over all threads of the values read;
 *       stores: the sum of s[] after the loop.  Both follow from the index
 *       formula alone, so the caller can check that every access touched the
 *       word it should.
 * Synchronous (it allocates and frees 16 bytes of device memory, and runs on
 * the legacy default stream of the current device).  Returns 0, -7 for an
 * argument out of range, -3 for a NULL output pointer, -5 when the launch or
 * a copy fails.
 */
#ifndef SMEM_BANK_PROBE_H
#define SMEM_BANK_PROBE_H

#ifdef __cplusplus
extern "C" {
#endif

int smem_bank_stride_probe(int stride, int op, int warps, int iters, double *cycles_per_access,
                           long long *checksum);

/*
 * smem_bank_pattern_probe -- the same measurement for any warp-wide load
 * pattern and width.  For 64- and 128-bit accesses the bank page says only
 * that the lanes each transaction serves must be analysed
 * ("为什么 double 和 float4 要另算"); this probe lets that be measured per
 * pattern (passes per instruction with ncu, or cycles with the SM clock).
 *
 *   width_bytes : 4, 8 or 16 bytes per lane.
 *   lane_word   : HOST array of 32 word offsets, 0 <= lane_word[l] < 2048,
 *                 each a multiple of width_bytes / 4: lane l reads
 *                 width_bytes bytes at word lane_word[l] + 32 * (j % 64) in
 *                 access j (a shift by 32 words keeps every bank).
 *   warps, iters, cycles_per_access : as for smem_bank_stride_probe (loads).
 *   *checksum (out): the sum over all threads of the first word of each
 *                 vector read, with s[i] = i before the loop.
 * Synchronous; the same status codes as smem_bank_stride_probe.
 */
int smem_bank_pattern_probe(int width_bytes, const int *lane_word, int warps, int iters,
                            double *cycles_per_access, long long *checksum);

#ifdef __cplusplus
}
#endif

#endif /* SMEM_BANK_PROBE_H */

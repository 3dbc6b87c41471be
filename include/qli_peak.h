/*
 * qli_peak.h -- measurement library (libqli_peak.so), not part of the indexer's ABI.
 *
 * Measures the rate of the tensor-core contraction the indexer's score kernel issues:
 * tcgen05.mma.cta_group::1.kind::f16 (fp16 operands, fp32 accumulator in tensor memory), M = 128
 * (or 64) rows, K = 16 per instruction, N columns, with the A operand read from tensor memory (the
 * score kernel's form: A is the converted key tile) or from shared memory, issued into one
 * accumulator (each MMA depends on the one before) or cycled over several independent ones.  The
 * README has no counterpart; the figures are the denominators the score kernel's tensor
 * utilisation is measured against.
 */
#ifndef QLI_PEAK_H
#define QLI_PEAK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launch `ctas` CTAs of 128 threads, `ctas_per_sm` (1 or 2) resident per SM (pass that many times
 * the SM count); each allocates 512 / ctas_per_sm tensor-memory columns.  In each CTA one warp
 * issues `iters` (a multiple of 8) back-to-back MMAs of shape m x n x 16 in groups of eight (the K
 * steps of one 128-dim key tile), the i-th group into accumulator i mod `chains`, then waits
 * (bounded) for their completion.
 * Shapes: m = 128 with n a multiple of 16 in [16, 256], A from tensor memory (a_from_tmem = 1) or
 * shared memory (0); m = 64 with n a multiple of 8 in [8, 256], A from shared memory only.  The
 * accumulators and A must fit the columns: 64 + chains * n <= 512 / ctas_per_sm.  Per CTA it
 * writes the elapsed SM cycles to cycles[c] and the elapsed nanoseconds (globaltimer) to nanos[c];
 * *err (device, zeroed by the caller) receives 1 if a wait gave up.  All pointers are device
 * memory owned by the caller.  Enqueued on `stream`.  Returns 0, or a CUDA error code (non-zero)
 * for a launch failure or bad arguments.
 */
int qli_peak_mma_f16(int a_from_tmem, int m, int n, int chains, int ctas_per_sm, int iters, int ctas,
                     unsigned long long* cycles, unsigned long long* nanos, unsigned int* err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QLI_PEAK_H */

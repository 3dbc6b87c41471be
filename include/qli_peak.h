/*
 * qli_peak.h -- measurement library (libqli_peak.so), not part of the indexer's ABI.
 *
 * Measures the rate of the tensor-core contraction the indexer's score kernel issues:
 * tcgen05.mma.cta_group::1.kind::f16 (fp16 operands, fp32 accumulator in tensor memory), M = 128
 * rows, K = 16 per instruction, N columns, with the A operand read from tensor memory (the score
 * kernel's form: A is the converted key tile) or from shared memory.  The README has no
 * counterpart; the figure is the denominator the score kernel's tensor utilisation is judged
 * against.
 */
#ifndef QLI_PEAK_H
#define QLI_PEAK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launch `ctas` CTAs (one per SM: pass the SM count) of 128 threads; in each, one thread issues
 * `iters` back-to-back MMAs of shape 128 x n x 16 into one accumulator (n a multiple of 16 in
 * [16, 256]; a_from_tmem: 1 A from tensor memory, 0 from shared memory), then waits (bounded) for
 * their completion.  Per CTA it writes the elapsed SM cycles to cycles[c] and the elapsed
 * nanoseconds (globaltimer) to nanos[c]; *err (device, zeroed by the caller) receives 1 if a wait
 * gave up.  All pointers are device memory owned by the caller.  Enqueued on `stream`.
 * Returns 0, or a CUDA error code (non-zero) for a launch failure or bad arguments.
 */
int qli_peak_mma_f16(int a_from_tmem, int n, int iters, int ctas, unsigned long long* cycles,
                     unsigned long long* nanos, unsigned int* err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QLI_PEAK_H */

/*
 * qli_testing.h -- entry points of the TESTING build of the library (libqli_testing.so) only.
 *
 * The product library (libqli.so) does not export these symbols and has no switch of any kind
 * that changes what its kernels do.  The testing build is the same library compiled with
 * QLI_TESTING; the failure-detection tests load it to make the score kernel's bounded waits run
 * out without faulting the GPU, and a top-k test to give its CTAs many rows each.  The README
 * has no counterpart.
 */
#ifndef QLI_TESTING_H
#define QLI_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Select a stall for the score kernels launched after this call (process-wide, host memory):
 *   0  normal operation;
 *   1  the producer warp issues no copies, so every consumer's bounded wait runs out;
 *   2  the converter warps consume nothing, so the producer's key copies land and wait in the
 *      ring until the producer's own bounded wait runs out.
 * Either stall ends the launch with QLI_ERR_DEVICE_TIMEOUT in the workspace's device error word
 * (qli_get_device_error); the kernel lets its in-flight copies land and releases its tensor
 * memory before it exits, so the CUDA context stays usable.  Other values select 0.
 */
void qli_testing_set_stall(int mode);

/*
 * Cap the grid of the persistent two-per-SM top-k (problems whose rows hold at most 8192 keys and
 * outnumber the SMs) at `ctas` CTAs for the launches after this call (process-wide, host memory),
 * so that a small problem gives each CTA hundreds of rows: the CTAs work their rows' places out
 * in chunks of 512 rows, and the tests reach the chunk boundaries this way.  0 or less: no cap.
 * The results are the same whatever the cap.
 */
void qli_testing_set_topk_ctas(int ctas);

#ifdef __cplusplus
}
#endif

#endif /* QLI_TESTING_H */

/*
 * qli_testing.h -- entry point of the TESTING build of the library (libqli_testing.so) only.
 *
 * The product library (libqli.so) does not export this symbol and has no switch of any kind
 * that changes what its kernels do.  The testing build is the same library compiled with
 * QLI_TESTING; the failure-detection tests load it to make the score kernel's bounded waits run
 * out without faulting the GPU.  The README has no counterpart.
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

#ifdef __cplusplus
}
#endif

#endif /* QLI_TESTING_H */

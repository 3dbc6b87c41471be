// qli_topk.cu -- the per-row top-k for rows of up to 32768 keys in shared memory: one 1024-thread
// CTA per SM.  The kernel itself is in qli_topk.cuh.
#define QLI_TOPK_THREADS 1024
#define QLI_TOPK_CACHE_KEYS 32768
#define QLI_TOPK_BINS 8192
#define QLI_TOPK_LAUNCHER launch_topk
#include "qli_topk.cuh"

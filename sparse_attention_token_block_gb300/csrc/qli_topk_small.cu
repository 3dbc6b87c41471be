// qli_topk_small.cu -- the per-row top-k for problems whose rows hold at most 8192 keys: 512-thread
// CTAs with about 100 KB of shared memory, two per SM.  The kernel itself is in qli_topk.cuh.
#define QLI_TOPK_THREADS 512
#define QLI_TOPK_CACHE_KEYS 8192
#define QLI_TOPK_BINS 4096
#define QLI_TOPK_LAUNCHER launch_topk_small
#include "qli_topk.cuh"

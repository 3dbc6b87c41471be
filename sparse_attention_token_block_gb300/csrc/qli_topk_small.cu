// qli_topk_small.cu -- the per-row top-k for problems whose rows hold at most 8192 keys: 512-thread
// CTAs with about 90 KB of shared memory, two per SM.  2048 ordering bins (the fewest the bins'
// 16-byte loads allow at 512 threads): the prefill's top-k took 539 us with 4096 and 515 us with
// 2048 (8192: 853 us).  The kernel itself is in qli_topk.cuh.
#define QLI_TOPK_THREADS 512
#define QLI_TOPK_CACHE_KEYS 8192
#define QLI_TOPK_BINS 2048
#define QLI_TOPK_LAUNCHER launch_topk_small
#include "qli_topk.cuh"

// qli_score_split.cu -- the scoring kernel for groups of one query token with the split-local
// selection in its epilogue (each CTA keeps the top k of every chunk of its range; the top-k
// kernel then merges the chunks' candidates): two CTAs per SM.  The kernel is in qli_score.cuh.
#define QLI_SCORE_GT 1
#define QLI_SCORE_SPLIT 1
#define QLI_SCORE_LAUNCHER launch_score_split
#include "qli_score.cuh"

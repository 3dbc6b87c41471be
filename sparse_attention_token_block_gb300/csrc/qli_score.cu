// qli_score.cu -- the scoring kernel for groups of one query token (decode with one token per
// sequence): two CTAs per SM.  The kernel itself is in qli_score.cuh.
#define QLI_SCORE_GT 1
#define QLI_SCORE_LAUNCHER launch_score
#include "qli_score.cuh"

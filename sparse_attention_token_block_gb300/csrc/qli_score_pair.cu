// qli_score_pair.cu -- the scoring kernel for groups of two query tokens (decodes with two or four
// tokens per sequence): one CTA per SM, MMA N = 128 and three accumulator buffers in tensor memory.
// The kernel itself is in qli_score.cuh.
#define QLI_SCORE_GT 2
#define QLI_SCORE_LAUNCHER launch_score_pair
#include "qli_score.cuh"

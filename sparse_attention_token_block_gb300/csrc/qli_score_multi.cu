// qli_score_multi.cu -- the scoring kernel for groups of up to three query tokens (TND prefill,
// decodes with several tokens per sequence other than two or four): one CTA per SM, each converted
// key tile multiplied against up to three tokens' 64 heads at once.  The kernel itself is in
// qli_score.cuh.
#define QLI_SCORE_GT 3
#define QLI_SCORE_LAUNCHER launch_score_multi
#include "qli_score.cuh"

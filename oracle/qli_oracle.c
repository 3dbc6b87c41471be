/*
 * qli_oracle.c -- plain, slow, obviously-correct CPU oracle for the quantized lightning indexer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load this library.  It shares no code, header, table or constant with the CUDA library: it
 * restates the method from the Ascend "VllmQuantLightningIndexer" README on its own.
 *
 * What it computes (README, "功能说明" / function section, the out = Top-k{...} formula and its three
 * numbered steps), for one query token with g = 64 heads and one shared key head:
 *
 *   step 1   dot[h][j]   = Q[h] . K[j]                      (int8: exact int32; e4m3: exact, then fp32)
 *   step 2   v[h][j]     = ReLU( (ScaleQ[h] * ScaleK[j]) * dot[h][j] )
 *   step 3   score[j]    = sum_h W[h] * v[h][j]  (the 1_{1 x g} @ [...] reduction over the heads)
 *            out         = indices of the sparse_count largest scores
 *
 * Arithmetic is fp32 in the formula's own order: the outer product ScaleQ @ ScaleK^T first, then
 * the element-wise product with the dot, ReLU, the weight, and the head sum in ascending head order,
 * each step rounded to fp32 (build with -ffp-contract=off so no FMA fuses two roundings).
 *
 * Readings of points the README leaves open (each also listed with the design notes):
 *   - actual_seq_lengths_key counts original tokens; batch b holds Lc = ceil(Sk / cmp_ratio)
 *     compressed keys (the fp8 compressed-key workload states this length).
 *   - sparse_mode 3 (rightDownCausal): the query at original position p = Sk - Sq + r sees compressed
 *     key j iff j * cmp_ratio <= p, so it sees n = clamp(ceil((p + 1) / cmp_ratio), 0, Lc) keys.  The
 *     alternative "only complete compressed blocks" reading, n = floor((p + 1) / cmp_ratio), is
 *     available through complete_blocks_only.
 *   - sparse_mode 0 (defaultMask): every live row sees all Lc keys.
 *   - Output order: score descending, ties by index ascending; fewer than sparse_count visible keys
 *     are padded with -1; BSND rows r >= actual_seq_lengths_query[b] are all -1.
 *   - Indices are the logical compressed-key positions 0..Lc-1 of the row's own batch.
 *   - Invalid inputs that only the data can reveal (a length out of range, a block_table entry
 *     outside the pool) make every row of that batch -1 and set a bit in the returned error mask;
 *     invalid TND prefix sums make every row of the call -1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t batch;              /* B */
    int32_t s1;                 /* BSND: query rows per batch; ignored for TND */
    int32_t total_q;            /* TND: T rows; ignored for BSND */
    int32_t layout_tnd;         /* 0 = BSND, 1 = TND */
    int32_t qk_fp8;             /* 0 = int8 codes, 1 = float8_e4m3fn codes */
    int32_t scale_f32;          /* 0 = float16 weights/scales, 1 = float32 */
    int32_t num_heads;          /* g (64) */
    int32_t head_dim;           /* d (128) */
    int32_t num_blocks;         /* pages in the key pool */
    int32_t block_size;         /* keys per page */
    int32_t max_blocks_per_seq; /* block_table row length */
    int32_t sparse_count;       /* k */
    int32_t sparse_mode;        /* 0 or 3 */
    int32_t cmp_ratio;          /* key compression multiple */
    int32_t complete_blocks_only;
    int32_t key_stride;         /* elements between consecutive pages of the key pool (the README's
                                   `stride` of key's first axis); 0 = block_size * head_dim */
} qlio_problem;

enum { QLIO_ERR_LENGTH = 1, QLIO_ERR_PAGE = 2 };

/* ---------------------------------------------------------------------------------------------
 * Number formats
 * ------------------------------------------------------------------------------------------- */

/* IEEE 754 binary16 -> value, from the format's definition (1 sign, 5 exponent bits with bias 15,
 * 10 fraction bits; exponent 0 = subnormal, exponent 31 = inf/NaN).  Every binary16 value is exact
 * in binary32, so returning float loses nothing. */
float qlio_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + m, e - 25);
    return (float)(sign ? -v : v);
}

/* OCP 8-bit floating point E4M3 -> value: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 is subnormal (m * 2^-9); there are no infinities and S.1111.111 is NaN. */
double qlio_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xf;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + m, e - 10);
    return sign ? -v : v;
}

/* decode table for the 256 e4m3 codes, filled from qlio_e4m3_value on first use */
static double e4m3_table[256];
static pthread_once_t e4m3_once = PTHREAD_ONCE_INIT;

static void fill_e4m3_table(void)
{
    for (int c = 0; c < 256; ++c)
        e4m3_table[c] = qlio_e4m3_value((uint8_t)c);
}

static float load_scale(const qlio_problem* p, const void* base, int64_t i)
{
    if (p->scale_f32)
        return ((const float*)base)[i];
    return qlio_half_to_float(((const uint16_t*)base)[i]);
}

/* ---------------------------------------------------------------------------------------------
 * Lengths and the mask
 * ------------------------------------------------------------------------------------------- */

/* Rows of batch b: first global row and the live row count Sq_b (README "约束说明": for TND
 * actual_seq_lengths_query holds prefix sums; for BSND it is the per-batch token count, S1 when
 * absent).  Returns 0 when the lengths are invalid. */
static int batch_rows(const qlio_problem* p, const int32_t* seq_lens_q, int b, int64_t* first_row,
                      int64_t* rows_alloc, int32_t* sq)
{
    if (!p->layout_tnd) {
        *first_row = (int64_t)b * p->s1;
        *rows_alloc = p->s1;
        int32_t v = seq_lens_q ? seq_lens_q[b] : p->s1;
        if (v < 0 || v > p->s1) {
            *sq = 0;
            return 0;
        }
        *sq = v;
        return 1;
    }
    int32_t lo = b > 0 ? seq_lens_q[b - 1] : 0;
    int32_t hi = seq_lens_q[b];
    if (lo < 0 || hi < lo || hi > p->total_q) {
        *first_row = lo < 0 ? 0 : lo;
        *rows_alloc = 0;
        *sq = 0;
        return 0;
    }
    *first_row = lo;
    *rows_alloc = hi - lo;
    *sq = hi - lo;
    return 1;
}

/* Compressed key count Lc = ceil(Sk / cmp_ratio). */
static int64_t compressed_len(const qlio_problem* p, int32_t sk)
{
    return ((int64_t)sk + p->cmp_ratio - 1) / p->cmp_ratio;
}

/* Visible compressed keys for live row r of a batch with Sq live rows and Sk original keys
 * (README parameter table, sparse_mode: 0 = defaultMask, 3 = rightDownCausal). */
int64_t qlio_visible(const qlio_problem* p, int32_t sq, int32_t sk, int64_t r)
{
    int64_t lc = compressed_len(p, sk);
    if (r < 0 || r >= sq)
        return 0;
    if (p->sparse_mode == 0)
        return lc;
    int64_t pos = (int64_t)sk - sq + r;    /* original position of the query, right-aligned */
    int64_t n;
    if (pos < 0)
        return 0;
    if (p->complete_blocks_only)
        n = (pos + 1) / p->cmp_ratio;
    else
        n = (pos + 1 + p->cmp_ratio - 1) / p->cmp_ratio;
    if (n > lc)
        n = lc;
    return n;
}

/* ---------------------------------------------------------------------------------------------
 * One row
 * ------------------------------------------------------------------------------------------- */

typedef struct {
    float score;
    int32_t idx;
} scored_key;

/* score descending, then index ascending: a total order, so qsort's instability cannot show */
static int cmp_scored(const void* a, const void* b)
{
    const scored_key* x = (const scored_key*)a;
    const scored_key* y = (const scored_key*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

typedef struct {
    const qlio_problem* p;
    const void* query;
    const void* key;
    const void* weights;
    const void* q_scale;
    const void* k_scale;
    const int32_t* seq_lens_q;
    const int32_t* seq_lens_k;
    const int32_t* block_table;
    int32_t* out;
    float* scores;       /* optional [rows, ld] */
    int64_t ld;
    const uint8_t* row_mask; /* optional: only rows with a non-zero entry are computed */
    int64_t rows;
    int64_t* row_batch;  /* batch of each global row, -1 if none */
    int32_t* batch_ok;   /* per batch: lengths and pages valid */
    int32_t* batch_sq;
    volatile int64_t next_row;
} job;

/* dot product of query head h of global row `row` with compressed key (page, slot) */
static double dot_qk(const job* J, int64_t row, int h, int64_t page, int64_t slot)
{
    const qlio_problem* p = J->p;
    int64_t qoff = (row * p->num_heads + h) * (int64_t)p->head_dim;
    const int64_t page_stride = p->key_stride ? (int64_t)p->key_stride : (int64_t)p->block_size * p->head_dim;
    int64_t koff = page * page_stride + slot * (int64_t)p->head_dim; /* one key head */
    if (!p->qk_fp8) {
        const int8_t* q = (const int8_t*)J->query + qoff;
        const int8_t* k = (const int8_t*)J->key + koff;
        int32_t acc = 0; /* |sum| <= 128 * 128 * 128 = 2^21: exact in int32 */
        for (int d = 0; d < p->head_dim; ++d)
            acc += (int32_t)q[d] * (int32_t)k[d];
        return (double)acc;
    }
    const uint8_t* q = (const uint8_t*)J->query + qoff;
    const uint8_t* k = (const uint8_t*)J->key + koff;
    /* Each e4m3 value is m * 2^e with |m| < 16; a product has an 8-bit significand and an exponent
     * in [-18, 16], so 128 products and their partial sums fit in double's 53 bits: exact. */
    double acc = 0.0;
    for (int d = 0; d < p->head_dim; ++d)
        acc += e4m3_table[q[d]] * e4m3_table[k[d]];
    return acc;
}

static void run_row(job* J, int64_t row, scored_key* buf)
{
    const qlio_problem* p = J->p;
    int32_t k = p->sparse_count;
    int32_t* out = J->out + row * (int64_t)k;
    for (int32_t i = 0; i < k; ++i)
        out[i] = -1;
    int64_t b = J->row_batch[row];
    if (b < 0 || !J->batch_ok[b])
        return;
    if (J->row_mask && !J->row_mask[row])
        return;
    int64_t first_row, rows_alloc;
    int32_t sq;
    batch_rows(p, J->seq_lens_q, (int)b, &first_row, &rows_alloc, &sq);
    int64_t r = row - first_row;
    int32_t sk = J->seq_lens_k[b];
    int64_t n = qlio_visible(p, sq, sk, r);
    if (n <= 0)
        return;
    const int32_t* table = J->block_table + b * (int64_t)p->max_blocks_per_seq;
    for (int64_t j = 0; j < n; ++j) {
        int64_t page = table[j / p->block_size];
        int64_t slot = j % p->block_size;
        float sK = load_scale(p, J->k_scale, page * p->block_size + slot);
        float score = 0.0f;
        for (int h = 0; h < p->num_heads; ++h) {
            float sQ = load_scale(p, J->q_scale, row * p->num_heads + h);
            float w = load_scale(p, J->weights, row * p->num_heads + h);
            float dot = (float)dot_qk(J, row, h, page, slot); /* int8: exact; e4m3: one rounding */
            float a = sQ * sK;          /* ScaleQ @ ScaleK^T */
            float v = a * dot;          /* (...) (.) (Q @ K^T) */
            v = v > 0.0f ? v : 0.0f;    /* ReLU */
            float t = w * v;            /* (W @ 1) (.) ReLU(...) */
            score = score + t;          /* 1_{1 x g} @ [...] in head order */
        }
        buf[j].score = score;
        buf[j].idx = (int32_t)j;
        if (J->scores)
            J->scores[row * J->ld + j] = score;
    }
    qsort(buf, (size_t)n, sizeof(scored_key), cmp_scored);
    int64_t m = n < k ? n : k;
    for (int64_t i = 0; i < m; ++i)
        out[i] = buf[i].idx;
}

static void* worker(void* arg)
{
    job* J = (job*)arg;
    int64_t max_lc = 0;
    for (int b = 0; b < J->p->batch; ++b) {
        int64_t lc = compressed_len(J->p, J->seq_lens_k[b] > 0 ? J->seq_lens_k[b] : 0);
        if (lc > max_lc) max_lc = lc;
    }
    scored_key* buf = (scored_key*)malloc(sizeof(scored_key) * (size_t)(max_lc > 0 ? max_lc : 1));
    for (;;) {
        int64_t row = __atomic_fetch_add(&J->next_row, 1, __ATOMIC_RELAXED);
        if (row >= J->rows)
            break;
        run_row(J, row, buf);
    }
    free(buf);
    return NULL;
}

/* Total query rows in the output: B * S1 (BSND) or T (TND). */
int64_t qlio_rows(const qlio_problem* p)
{
    return p->layout_tnd ? p->total_q : (int64_t)p->batch * p->s1;
}

/*
 * The whole operator.  Inputs are host arrays in the README's layouts (see the module header);
 * `out` is int32 [rows, sparse_count].  `scores` (optional, may be NULL) receives the fp32 score of
 * every visible key at [row * ld + j]; other entries are left untouched.  `row_mask` (optional)
 * restricts the work to the rows whose entry is non-zero; the others are written as -1.  Returns
 * the error mask (0 when every batch was valid).  `nthreads` worker threads split the rows.
 */
int qlio_score_topk(const qlio_problem* p, const void* query, const void* key, const void* weights,
                    const void* q_scale, const void* k_scale, const int32_t* seq_lens_q,
                    const int32_t* seq_lens_k, const int32_t* block_table, int32_t* out,
                    float* scores, int64_t ld, const uint8_t* row_mask, int nthreads)
{
    job J;
    pthread_once(&e4m3_once, fill_e4m3_table);
    memset(&J, 0, sizeof(J));
    J.p = p;
    J.query = query;
    J.key = key;
    J.weights = weights;
    J.q_scale = q_scale;
    J.k_scale = k_scale;
    J.seq_lens_q = seq_lens_q;
    J.seq_lens_k = seq_lens_k;
    J.block_table = block_table;
    J.out = out;
    J.scores = scores;
    J.ld = ld;
    J.row_mask = row_mask;
    J.rows = qlio_rows(p);
    J.next_row = 0;
    int err = 0;
    J.row_batch = (int64_t*)malloc(sizeof(int64_t) * (size_t)(J.rows > 0 ? J.rows : 1));
    J.batch_ok = (int32_t*)malloc(sizeof(int32_t) * (size_t)(p->batch > 0 ? p->batch : 1));
    J.batch_sq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(p->batch > 0 ? p->batch : 1));
    for (int64_t i = 0; i < J.rows; ++i)
        J.row_batch[i] = -1;
    /* TND prefix sums that are negative, decreasing or beyond T leave no consistent row ranges:
     * then every batch counts as invalid */
    int tnd_bad = 0;
    if (p->layout_tnd) {
        for (int b = 0; b < p->batch; ++b) {
            int64_t fr, ra;
            int32_t sq;
            if (!batch_rows(p, seq_lens_q, b, &fr, &ra, &sq))
                tnd_bad = 1;
        }
    }
    for (int b = 0; b < p->batch; ++b) {
        int64_t first_row, rows_alloc;
        int32_t sq;
        int ok = batch_rows(p, seq_lens_q, b, &first_row, &rows_alloc, &sq) && !tnd_bad;
        int32_t sk = seq_lens_k[b];
        if (sk < 0)
            ok = 0;
        int64_t lc = ok ? compressed_len(p, sk) : 0;
        if (lc > (int64_t)p->max_blocks_per_seq * p->block_size)
            ok = 0;
        if (!ok)
            err |= QLIO_ERR_LENGTH;
        /* every page the batch's live rows can see: a live row exists only if sq > 0, and the last
         * live row then sees all Lc keys */
        if (ok && sq > 0) {
            int64_t pages = (lc + p->block_size - 1) / p->block_size;
            for (int64_t i = 0; i < pages; ++i) {
                int32_t pg = block_table[(int64_t)b * p->max_blocks_per_seq + i];
                if (pg < 0 || pg >= p->num_blocks) {
                    ok = 0;
                    err |= QLIO_ERR_PAGE;
                    break;
                }
            }
        }
        J.batch_ok[b] = ok;
        J.batch_sq[b] = sq;
        for (int64_t r = 0; r < rows_alloc; ++r)
            if (first_row + r < J.rows)
                J.row_batch[first_row + r] = b;
    }
    if (nthreads < 1)
        nthreads = 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i)
        pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(th);
    free(J.row_batch);
    free(J.batch_ok);
    free(J.batch_sq);
    return err;
}

/* ---------------------------------------------------------------------------------------------
 * Upstream quantizer (README: query and key are quantized per token and head -- quant mode 0 --
 * "store 8-bit, compute 8-bit"; the dequant scales are the ScaleQ / ScaleK of the formula).  The
 * README names the mode only; the reading used: symmetric absmax per 128-element (token, head)
 * vector,
 *     amax  = max_d |x_d|                      (x: bfloat16 widened exactly to fp32)
 *     s     = amax / Qmax   (fp32 division)    Qmax = 127 (int8) or 448 (e4m3, its largest finite)
 *     s     = the scale's storage value: fp16 rounds to nearest (ties to even), saturating at 65504
 *     code  = int8:  rint(x_d / s) clamped to [-127, 127]   (fp32 division; ties to even)
 *             e4m3:  the nearest e4m3 value to x_d / s (ties to the even code), saturating at 448
 *     s = 0 (an all-zero vector): every code is 0.
 * Nearest-value searches below run over the formats' own code tables, so no conversion of the C
 * library or the hardware is involved.
 * ------------------------------------------------------------------------------------------- */

/* binary16 code nearest to v in [0, 65504] (ties: the even code) */
static uint16_t nearest_half_code(double v)
{
    uint16_t lo = 0, hi = 0x7BFF; /* largest finite */
    if (v >= (double)qlio_half_to_float(hi)) return hi;
    while (hi - lo > 1) { /* invariant: value(lo) <= v < value(hi) */
        uint16_t mid = (uint16_t)((lo + hi) / 2);
        if ((double)qlio_half_to_float(mid) <= v) lo = mid; else hi = mid;
    }
    double dl = v - (double)qlio_half_to_float(lo), dh = (double)qlio_half_to_float(hi) - v;
    if (dl < dh) return lo;
    if (dh < dl) return hi;
    return (lo & 1) ? hi : lo;
}

/* e4m3 code (sign bit clear) nearest to v in [0, 448] (ties: the even code) */
static uint8_t nearest_e4m3_code(double v)
{
    uint8_t lo = 0, hi = 0x7E; /* 0x7E = 448, the largest finite */
    if (v >= qlio_e4m3_value(hi)) return hi;
    while (hi - lo > 1) {
        uint8_t mid = (uint8_t)((lo + hi) / 2);
        if (qlio_e4m3_value(mid) <= v) lo = mid; else hi = mid;
    }
    double dl = v - qlio_e4m3_value(lo), dh = qlio_e4m3_value(hi) - v;
    if (dl < dh) return lo;
    if (dh < dl) return hi;
    return (lo & 1) ? hi : lo;
}

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof(f));
    return f;
}

/* one 128-element vector: codes (int8 or e4m3) and its scale as stored (fp16 or fp32) */
static void quantize_vector(int qk_fp8, int scale_f32, const uint16_t* x_bf16, void* codes, void* scale_out)
{
    float x[128];
    float amax = 0.0f;
    for (int d = 0; d < 128; ++d) {
        x[d] = bf16_to_float(x_bf16[d]);
        amax = fmaxf(amax, fabsf(x[d]));
    }
    const float qmax = qk_fp8 ? 448.0f : 127.0f;
    float s = amax / qmax;
    uint16_t s_half = 0;
    if (!scale_f32) {
        s_half = nearest_half_code(s < 65504.0f ? (double)s : 65504.0);
        s = qlio_half_to_float(s_half);
    }
    if (scale_f32) memcpy(scale_out, &s, sizeof(float));
    else memcpy(scale_out, &s_half, sizeof(uint16_t));
    for (int d = 0; d < 128; ++d) {
        if (s == 0.0f) {
            ((uint8_t*)codes)[d] = 0;
            continue;
        }
        const float y = x[d] / s;
        if (!qk_fp8) {
            float r = rintf(y);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            ((int8_t*)codes)[d] = (int8_t)r;
        } else {
            const double a = fabs((double)y);
            ((uint8_t*)codes)[d] = (uint8_t)((signbit(y) ? 0x80 : 0) | nearest_e4m3_code(a > 448.0 ? 448.0 : a));
        }
    }
}

/* Quantize n_vec vectors of 128 bfloat16 (a query [rows, 64, 128] is rows * 64 vectors) into
 * codes [n_vec, 128] and scales [n_vec]. */
void qlio_quantize_vectors(int qk_fp8, int scale_f32, const uint16_t* x_bf16, int64_t n_vec, void* codes,
                           void* scales)
{
    const size_t ssz = scale_f32 ? 4 : 2;
    for (int64_t v = 0; v < n_vec; ++v)
        quantize_vector(qk_fp8, scale_f32, x_bf16 + v * 128, (uint8_t*)codes + v * 128,
                        (uint8_t*)scales + v * ssz);
}

/* The paged key-cache write: token t's key (one head, 128 bfloat16) goes to compressed position
 * token_pos[t] of batch token_batch[t], i.e. page block_table[b][pos / bs], slot pos % bs, of the
 * pool (pages p->key_stride elements apart, 0 = contiguous) and of k_scale [num_blocks, bs].  A
 * batch or position out of range skips the token (QLIO_ERR_LENGTH), a page outside the pool too
 * (QLIO_ERR_PAGE).  Returns the error mask. */
int qlio_quantize_keys(const qlio_problem* p, const uint16_t* key_bf16, int64_t tokens, const int32_t* token_batch,
                       const int32_t* token_pos, const int32_t* block_table, void* key_pool, void* k_scale)
{
    int err = 0;
    const int64_t bs = p->block_size;
    const int64_t stride = p->key_stride ? (int64_t)p->key_stride : bs * 128;
    const size_t ssz = p->scale_f32 ? 4 : 2;
    for (int64_t t = 0; t < tokens; ++t) {
        const int64_t b = token_batch[t], pos = token_pos[t];
        if (b < 0 || b >= p->batch || pos < 0 || pos >= (int64_t)p->max_blocks_per_seq * bs) {
            err |= QLIO_ERR_LENGTH;
            continue;
        }
        const int64_t page = block_table[b * p->max_blocks_per_seq + pos / bs], slot = pos % bs;
        if (page < 0 || page >= p->num_blocks) {
            err |= QLIO_ERR_PAGE;
            continue;
        }
        quantize_vector(p->qk_fp8, p->scale_f32, key_bf16 + t * 128, (uint8_t*)key_pool + page * stride + slot * 128,
                        (uint8_t*)k_scale + (page * bs + slot) * ssz);
    }
    return err;
}

/* ---------------------------------------------------------------------------------------------
 * Downstream sparse-attention gather (README: sparse_indices are the token indices that take part
 * in the sparse attention, the output "as the input of Attention"; block_table is the PageAttention
 * KV storage block map).  Reading used: the attention reads, for every output row and every
 * selected compressed position j of the row's batch b, the KV entry stored at that position through
 * the same block map:
 *     out[r][i] = kv[ block_table[b][j / block_size] ][ j % block_size ]     (entry_bytes bytes)
 * where j = sparse_indices[r][i]; j = -1 (padding) gives an all-zero entry.  The KV pool holds
 * num_blocks pages of block_size entries, pages kv_stride bytes apart (0 = contiguous).
 * Row r belongs to batch r / S1 (BSND) or to the b with seq_lens_q[b-1] <= r < seq_lens_q[b]
 * (TND prefix sums, seq_lens_q[-1] = 0, within T).  An index other than -1 that is negative, not
 * below the block_table's capacity max_blocks_per_seq * block_size, not below the batch's
 * Lc = ceil(seq_lens_k[b] / cmp_ratio) (when seq_lens_k is given), or in a row with no batch, gives
 * a zero entry and QLIO_ERR_LENGTH; a page outside the pool gives a zero entry and QLIO_ERR_PAGE.
 * counts[r] (optional) = the entries of row r copied from the pool.  Returns the error mask.
 * ------------------------------------------------------------------------------------------- */

/* batch of global row r, or -1 */
static int64_t gather_row_batch(const qlio_problem* p, const int32_t* seq_lens_q, int64_t r)
{
    if (!p->layout_tnd)
        return p->s1 > 0 ? r / p->s1 : -1;
    for (int b = 0; b < p->batch; ++b) {
        int64_t lo = b > 0 ? seq_lens_q[b - 1] : 0, hi = seq_lens_q[b];
        if (r < hi)
            return (lo <= r && hi <= p->total_q) ? b : -1;
    }
    return -1;
}

int qlio_gather_kv(const qlio_problem* p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                   const int32_t* block_table, const int32_t* sparse_indices, const void* kv, int64_t entry_bytes,
                   int64_t kv_stride, void* out, int32_t* counts)
{
    int err = 0;
    const int64_t rows = qlio_rows(p), k = p->sparse_count, bs = p->block_size;
    const int64_t stride = kv_stride ? kv_stride : bs * entry_bytes;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t b = gather_row_batch(p, seq_lens_q, r);
        int64_t limit = -1;
        if (b >= 0) {
            limit = (int64_t)p->max_blocks_per_seq * bs;
            if (seq_lens_k) {
                const int64_t lc = seq_lens_k[b] < 0 ? -1 : compressed_len(p, seq_lens_k[b]);
                if (lc < limit)
                    limit = lc;
            }
        }
        int32_t copied = 0;
        for (int64_t i = 0; i < k; ++i) {
            const int64_t j = sparse_indices[r * k + i];
            uint8_t* dst = (uint8_t*)out + (r * k + i) * entry_bytes;
            memset(dst, 0, (size_t)entry_bytes);
            if (j == -1)
                continue;
            if (j < 0 || j >= limit) {
                err |= QLIO_ERR_LENGTH;
                continue;
            }
            const int64_t page = block_table[b * p->max_blocks_per_seq + j / bs];
            if (page < 0 || page >= p->num_blocks) {
                err |= QLIO_ERR_PAGE;
                continue;
            }
            memcpy(dst, (const uint8_t*)kv + page * stride + (j % bs) * entry_bytes, (size_t)entry_bytes);
            ++copied;
        }
        if (counts)
            counts[r] = copied;
    }
    return err;
}

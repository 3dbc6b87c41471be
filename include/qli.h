/*
 * qli.h -- C ABI of the GB300 (sm_103a) quantized lightning indexer.
 *
 * The operation (Ascend "VllmQuantLightningIndexer" README, function section, the formula
 * out = Top-k{ 1_{1 x g} @ [ (W @ 1_{1 x Sk}) (.) ReLU( (Scale_Q @ Scale_K^T) (.) (Q @ K^T) ) ] }):
 * for every query token with g = 64 quantized heads of dim 128 and one shared quantized key head,
 *
 *     score[j] = sum_h W[h] * ReLU( ScaleQ[h] * ScaleK[j] * (Q_h . K_j) )
 *
 * over the token's visible compressed keys j, and the int32 indices of the sparse_count largest
 * scores (score descending, ties by index ascending), padded with -1.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library never allocates,
 *     frees or retains them past the call.  Host structs are read during the call only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Calls only
 *     enqueue work; none synchronises except qli_get_device_error.  No call reads device data on
 *     the host, so the enqueueing calls can be captured into a CUDA graph.
 *   - Arguments that are wrong on their face (shape, dtype, attribute, size, alignment, null) are
 *     rejected synchronously with a status and nothing is enqueued.
 *   - Faults only the device data can reveal (a length beyond the declared maxima or the
 *     block_table's capacity, non-monotone TND prefix sums, a block_table entry outside the pool)
 *     never trap: every output row of the affected batch (all rows, for bad TND prefix sums) is
 *     written as -1 and a bit is set in the workspace's sticky device error word, which
 *     qli_get_device_error reports.
 *
 * Layouts (README parameter table and layout constraints):
 *   query        BSND [B, S1, 64, 128] or TND [T, 64, 128]; int8 or float8_e4m3fn codes
 *   key          PA_BSND pool [num_blocks, block_size, 1, 128], same dtype as query, contiguous
 *   weights      [B, S1, 64] / [T, 64]     float16 or float32 (one dtype shared by the three
 *   q_scale      [B, S1, 64] / [T, 64]       float inputs), contiguous
 *   k_scale      [num_blocks, block_size, 1]
 *   seq_lens_q   int32 [B]: BSND query tokens per batch (optional, default S1);
 *                TND prefix sums (required)
 *   seq_lens_k   int32 [B]: original key tokens per batch (required); the batch holds
 *                ceil(seq_lens_k / cmp_ratio) compressed keys, key j at
 *                key[block_table[b][j / block_size]][j % block_size]
 *   block_table  int32 [B, max_blocks_per_seq]
 *   sparse_indices int32 [B, S1, 1, sparse_count] / [T, 1, sparse_count]: compressed-key indices
 *                within the row's batch
 */
#ifndef QLI_H
#define QLI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QLI_OK = 0,
    QLI_ERR_INVALID_ARG = 1,          /* argument wrong on its face; nothing enqueued */
    QLI_ERR_UNSUPPORTED = 2,          /* valid per the README but not implemented */
    QLI_ERR_WORKSPACE_TOO_SMALL = 3,  /* metadata or workspace buffer below the required size */
    QLI_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
    QLI_ERR_DEVICE_BAD_INPUT = 5,     /* (qli_get_device_error) device data was invalid */
    QLI_ERR_DEVICE_TIMEOUT = 6,       /* (qli_get_device_error) a bounded device wait gave up */
    QLI_ERR_NO_DEVICE = 7             /* no sm_100-family GPU with tensor memory is current */
} qli_status;

typedef enum { QLI_INT8 = 0, QLI_FP8_E4M3 = 1 } qli_qk_dtype;    /* README: INT8, FLOAT8_e4m3fn */
typedef enum { QLI_F16 = 0, QLI_F32 = 1 } qli_scale_dtype;       /* README: FLOAT16, FLOAT32 */
typedef enum { QLI_BSND = 0, QLI_TND = 1 } qli_q_layout;         /* README layout_query */

/*
 * Every attribute of one call (README parameter table).  Fields are plain ints so the struct has
 * the same layout for every caller.
 */
typedef struct {
    int32_t batch;              /* B; for TND the number of entries of seq_lens_q */
    int32_t max_q_tokens;       /* BSND: S1 (rows per batch in query/output); ignored for TND */
    int32_t total_q_tokens;     /* TND: T (rows of query/output); ignored for BSND */
    int32_t num_heads_q;        /* must be 64 (README constraint on query's N axis) */
    int32_t num_heads_k;        /* must be 1 (README constraint on key's N axis) */
    int32_t head_dim;           /* must be 128 (README constraint on the D axis) */
    int32_t qk_dtype;           /* qli_qk_dtype of query and key */
    int32_t scale_dtype;        /* qli_scale_dtype of weights, q_scale and k_scale */
    int32_t layout_q;           /* qli_q_layout; the key layout is always PA_BSND */
    int32_t num_blocks;         /* pages in the key pool */
    int32_t block_size;         /* keys per page: a multiple of 16, at most 1024 */
    int32_t max_blocks_per_seq; /* block_table row length: >= ceil(ceil(max_seqlen_k/cmp)/bs) */
    int32_t sparse_count;       /* k, in [1, 2048] */
    int32_t sparse_mode;        /* 0 = defaultMask, 3 = rightDownCausal */
    int32_t cmp_ratio;          /* key compression multiple: 1, 2, 4, ..., 128 */
    int32_t query_quant_mode;   /* must be 0 (per-token-head) */
    int32_t key_quant_mode;     /* must be 0 (per-token-head) */
    int32_t return_value;       /* 1: also write sparse_values (the scores of the indices); 0: not */
    int64_t pre_tokens;         /* reserved by the README: must be INT64_MAX */
    int64_t next_tokens;        /* reserved by the README: must be INT64_MAX */
    int32_t max_seqlen_q;       /* host-known bound on per-batch query tokens (>= every one) */
    int32_t max_seqlen_k;       /* host-known bound on seq_lens_k (>= every entry) */
    int32_t key_stride;         /* README `stride`: elements between consecutive pages of the key
                                   pool, >= block_size * 128 and a multiple of 16; 0 = contiguous */
    int32_t mask_complete_blocks; /* sparse_mode 3 with cmp_ratio > 1: 0 = a compressed key is
                                   visible once its block has started, n = ceil((p + 1) / cmp);
                                   1 = only complete blocks, n = floor((p + 1) / cmp) */
    int32_t split_topk;         /* qli_split_topk: how the top-k runs for one query token per
                                   sequence (BSND, S1 = 1); the result is the same either way */
} qli_problem;

/*
 * The top-k in two stages (README function section, step 3, done as a per-split selection and a
 * cross-split merge).  ON: every score CTA keeps, for each part of its key range that lies in one
 * aligned block of 4096 keys of a row, the exact top sparse_count keys of that part (by score
 * descending, index ascending), and the top-k merges those candidates per row; OFF: the top-k
 * reads each row's whole score line.  AUTO is OFF: on a GB300 the two-stage form measured slower
 * at every size tried.  Problems with more than one query token per sequence always run OFF.  ON
 * makes the workspace larger (qli_workspace_size).  The indices are the same either way.
 */
typedef enum { QLI_SPLIT_AUTO = 0, QLI_SPLIT_ON = 1, QLI_SPLIT_OFF = 2 } qli_split_topk;

/* Fill `p` with the README's defaults (BSND, int8, fp16, mode 0, cmp 1, k 2048, reserved fields
 * at their only accepted values).  The caller then sets the sizes. */
void qli_problem_init(qli_problem* p);

/* Check `p` on the host without touching the device.  QLI_OK or QLI_ERR_INVALID_ARG /
 * QLI_ERR_UNSUPPORTED; `why` (optional, may be NULL) receives a static message. */
qli_status qli_validate(const qli_problem* p, const char** why);

/* Number of int32 words the metadata buffer needs for `p` (at least 1024, the README's size).
 * 0 if `p` is invalid. */
size_t qli_metadata_words(const qli_problem* p);

/* Bytes of device scratch qli_score_topk needs for `p` (256-byte aligned start required).
 * 0 if `p` is invalid. */
size_t qli_workspace_size(const qli_problem* p);

/*
 * Work-split scheduler (README: metadata parameter of the indexer and its companion
 * VllmQuantLightningIndexerMetadata call: cores used, block size and each core's start points).
 * Reads the device lengths and writes, into `metadata` (int32[metadata_words], device, caller-
 * owned, 16-byte aligned), the per-batch row/key extents and a balanced split of every live query
 * group's key tiles over the GPU's SMs.  One kernel, enqueued on `stream`.  The result depends
 * only on the lengths and `p`, so one metadata buffer serves every call that shares them (e.g. all
 * layers of a step).  seq_lens_q may be NULL for BSND.
 */
qli_status qli_metadata(const qli_problem* p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                        int32_t* metadata, size_t metadata_words, void* stream);

/*
 * The indexer (README: the indexer call and its formula).  Scores every visible (query token,
 * compressed key) pair on the tensor cores and writes the top-sparse_count indices per row into
 * sparse_indices.  `metadata` must come from qli_metadata with the same `p` and lengths.
 * `workspace` is caller-owned device scratch of at least qli_workspace_size(p) bytes, 256-byte
 * aligned, zeroed once after allocation (qli_workspace_init); calls sharing a workspace must be
 * ordered on one stream.  sparse_values (README return_value, which the README lists as not yet
 * supported there): with p->return_value = 1, float32 [rows, sparse_count], device, caller-owned,
 * receives the score of each index written (as the kernel computed it, fp32) and -infinity where
 * the index is -1; with return_value = 0 it must be NULL.  A mismatch is QLI_ERR_INVALID_ARG.
 * query, key, weights, q_scale, k_scale and metadata must be 16-byte aligned.
 */
qli_status qli_score_topk(const qli_problem* p, const void* query, const void* key,
                          const void* weights, const void* q_scale, const void* k_scale,
                          const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                          const int32_t* block_table, const int32_t* metadata,
                          size_t metadata_words, void* workspace, size_t workspace_bytes,
                          int32_t* sparse_indices, float* sparse_values, void* stream);

/*
 * The two stages of qli_score_topk, for callers that time or reuse them separately.  Same
 * arguments, rules and errors as qli_score_topk; calling qli_score then qli_topk on one stream with
 * one workspace gives exactly what qli_score_topk gives.
 *   qli_score: README steps 1-2 and the weighted head sum -- every visible key's score, kept in the
 *              workspace (one line per query row);
 *   qli_topk:  README step 3 -- the top-sparse_count indices of each row's score line, padded
 *              with -1, into sparse_indices (and their scores into sparse_values).
 */
qli_status qli_score(const qli_problem* p, const void* query, const void* key, const void* weights,
                     const void* q_scale, const void* k_scale, const int32_t* seq_lens_q,
                     const int32_t* seq_lens_k, const int32_t* block_table, const int32_t* metadata,
                     size_t metadata_words, void* workspace, size_t workspace_bytes, void* stream);
qli_status qli_topk(const qli_problem* p, const int32_t* block_table, const int32_t* metadata,
                    size_t metadata_words, void* workspace, size_t workspace_bytes,
                    int32_t* sparse_indices, float* sparse_values, void* stream);

/*
 * qli_score_topk without a caller-provided workspace.  The README has no counterpart: this entry
 * point exists for callers that cannot allocate device memory -- a plugin whose host framework
 * owns every allocation and forbids cudaMalloc, a runtime with a fixed memory budget set aside at
 * start-up, or latency-critical code that must not call cudaMalloc because it can synchronise
 * the device.  The scratch lives in one 16 MiB array inside the library, reserved on every GPU
 * that loads the library until the process exits; a problem whose qli_workspace_size exceeds
 * 16 MiB is rejected with QLI_ERR_WORKSPACE_TOO_SMALL.  Inputs, metadata and sparse_indices are
 * as for qli_score_topk (return_value must be 0: no sparse_values here); `device_error` (optional device pointer to one uint32) receives this
 * call's device error word (bits as for qli_get_device_error).  The first call on a device looks
 * up the array's address with that device current; make it before any stream capture.  All
 * calls share the array: calls that overlap on the GPU race, so order them on one stream.  No
 * allocating call is made.
 */
qli_status qli_score_topk_static(const qli_problem* p, const void* query, const void* key,
                                 const void* weights, const void* q_scale, const void* k_scale,
                                 const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                                 const int32_t* block_table, const int32_t* metadata,
                                 size_t metadata_words, int32_t* sparse_indices,
                                 uint32_t* device_error, void* stream);

/*
 * Execution plans: one indexer call (optionally preceded by its metadata call) captured once into
 * a CUDA graph and replayed.  The README has no counterpart; a plan removes the per-call launch
 * path (about 4.6 us per call on GB300 for the decode workloads) for callers whose buffers stay
 * at fixed addresses from call to call -- a serving loop that refreshes the same input buffers in
 * place before each launch.  A plan captures the pointers and problem given here: every launch
 * reads the inputs, lengths and block_table at those addresses as they are when it runs and
 * writes metadata (if captured), workspace and sparse_indices there.  All arguments are as for
 * qli_metadata and qli_score_topk; with_metadata = 0 captures the indexer alone (the metadata
 * buffer must then hold the metadata of the lengths each launch sees).  The capture runs on a
 * private stream of the current device and enqueues no work; `*plan` (host object, owned by the
 * caller, released with qli_plan_destroy) is NULL on failure.  Errors: the argument checks of the
 * captured calls, QLI_ERR_CUDA if capture or instantiation fails.
 */
typedef struct qli_plan qli_plan;
qli_status qli_plan_create(const qli_problem* p, int with_metadata, const void* query, const void* key,
                           const void* weights, const void* q_scale, const void* k_scale,
                           const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                           const int32_t* block_table, int32_t* metadata, size_t metadata_words,
                           void* workspace, size_t workspace_bytes, int32_t* sparse_indices,
                           float* sparse_values, qli_plan** plan);
/* Enqueue one replay of the plan on `stream` (any stream of the plan's device). */
qli_status qli_plan_launch(const qli_plan* plan, void* stream);
/* Release a plan (NULL is ignored).  Launches already enqueued still run. */
void qli_plan_destroy(qli_plan* plan);

/*
 * Upstream quantizer (README parameter table: query_quant_mode / key_quant_mode 0, the
 * per-token-head mode; the README names the mode but gives no formula, so this is the plain
 * symmetric absmax reading).  Each vector of 128 bfloat16 values x (one token of one head) becomes
 *
 *     amax = max_d |x_d|,   s = amax / Qmax   (Qmax = 127 for int8, 448 for float8_e4m3fn)
 *
 * computed in fp32 and then rounded to the scale dtype (fp16: to nearest, ties to even, values
 * above 65504 saturate to 65504), and codes  c_d = x_d / s  (fp32 division by the stored s)
 * rounded to nearest with ties to even: int8 saturates to [-127, 127], e4m3 to +-448.  A vector
 * whose stored s is 0 gets zero codes.  So x_d ~= s * c_d, which is how the indexer reads them.
 * Non-finite inputs are outside the definition.
 *
 * qli_quantize: `x` bfloat16 [n_vec][128] (16-byte aligned) -> `codes` [n_vec][128] of qk_dtype
 * (8-byte aligned) and `scales` [n_vec] of scale_dtype (aligned to its element).  For the query of
 * the indexer, n_vec = rows * 64 and the outputs are exactly its query / q_scale arguments.  All
 * device pointers, caller-owned; one kernel on `stream`.  n_vec = 0 enqueues nothing; n_vec is
 * at most 2^36.
 * QLI_ERR_INVALID_ARG for a bad dtype, a negative count, a NULL or misaligned pointer.
 */
qli_status qli_quantize(int32_t qk_dtype, int32_t scale_dtype, const void* x, int64_t n_vec, void* codes,
                        void* scales, void* stream);

/*
 * The paged key-cache write of new keys (README layout: key is the PA_BSND pool addressed by
 * block_table, k_scale is [num_blocks, block_size, 1]).  Token t's key `key_bf16[t]` (128
 * bfloat16, 16-byte aligned rows) is quantized as in qli_quantize (qk_dtype and scale_dtype of `p`)
 * and written to compressed position `token_pos[t]` of batch `token_batch[t]`: page
 * block_table[b][pos / block_size], slot pos % block_size, of `key` (pages p->key_stride elements
 * apart as in qli_score_topk -- bytes, since a code is one byte -- 0 = contiguous; 16-byte
 * aligned) and of `k_scale`.  Nothing else of the pool changes.  Positions
 * must be distinct (two tokens writing one slot leave either).  Lengths are not consulted: the
 * caller raises seq_lens_k afterwards.  A batch outside [0, batch) or a position outside
 * [0, max_blocks_per_seq * block_size) skips the token and sets error bit 1 (length), a page
 * outside the pool skips it and sets bit 2 (page), in `workspace`'s device error word when
 * `workspace` is given (NULL: not reported); qli_get_device_error reads it.  One kernel on
 * `stream`; tokens = 0 enqueues nothing.
 */
qli_status qli_quantize_keys(const qli_problem* p, const void* key_bf16, int64_t tokens, const int32_t* token_batch,
                             const int32_t* token_pos, const int32_t* block_table, void* key, void* k_scale,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Downstream sparse-attention gather (README function section: the selected indices are the token
 * indices that take part in the sparse attention, the output is the attention's input; parameter
 * table: block_table is the PageAttention KV block map).  Reading: the attention reads, for each
 * output row r (batch b = r / max_q_tokens for BSND; for TND the b with seq_lens_q[b-1] <= r <
 * seq_lens_q[b]) and each i < sparse_count, the KV entry at compressed position
 * j = sparse_indices[r][i] of its batch through the same block map:
 *
 *     out[r][i][0 .. entry_bytes) = kv page block_table[b][j / block_size], entry j % block_size
 *
 * `kv` is the attention's paged KV cache: num_blocks pages of block_size entries of `entry_bytes`
 * bytes (a multiple of 16, at most 65536), pages `kv_stride` bytes apart (0 = contiguous
 * block_size * entry_bytes; else a multiple of 16 of at least that), 16-byte aligned; its content
 * is opaque bytes.  `out` [rows, sparse_count, entry_bytes] (16-byte aligned).  j = -1 (padding)
 * gives an all-zero entry.  An index that is otherwise negative, not below the block_table's
 * capacity max_blocks_per_seq * block_size, not below the batch's ceil(seq_lens_k[b] / cmp_ratio)
 * (when seq_lens_k is given; NULL skips that bound), or in a row that belongs to no batch, gives a
 * zero entry and error bit 1; a page outside the pool gives a zero entry and bit 2 (in
 * `workspace`'s device error word when `workspace` is given).  `counts` (optional, int32 [rows])
 * receives the number of entries of each row copied from the pool.  seq_lens_q: TND prefix sums
 * (required for TND, unused for BSND); prefix sums that are not non-decreasing are invalid input
 * (then rows may be zero-filled; nothing is read or written outside the buffers).  One kernel on
 * `stream`; it may begin while the previous kernel on the stream finishes and waits for it before
 * reading the indices.
 */
qli_status qli_gather_kv(const qli_problem* p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                         const int32_t* block_table, const int32_t* sparse_indices, const void* kv,
                         int64_t entry_bytes, int64_t kv_stride, void* out, int32_t* counts, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Zero the workspace's device error word (enqueued on `stream`).  Call once after allocating a
 * workspace, before its first qli_score_topk. */
qli_status qli_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronise `stream`, read and clear the workspace's sticky device error word.  QLI_OK,
 * QLI_ERR_DEVICE_BAD_INPUT (a length or block_table entry was invalid; the affected rows are -1),
 * QLI_ERR_DEVICE_TIMEOUT (a bounded wait inside a kernel gave up), or QLI_ERR_CUDA.
 * `bits` (optional) receives the raw word: 1 length, 2 page, 4 timeout, 8 metadata mismatch.
 */
qli_status qli_get_device_error(void* workspace, void* stream, uint32_t* bits);

/* Static, human-readable name of a status. */
const char* qli_status_string(qli_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int qli_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QLI_H */

// qli_api.cu -- host side of the C ABI: argument validation (README parameter table and
// constraints), buffer sizing, the key pool's TMA descriptor, and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>

#include "qli_internal.cuh"

namespace qli {

MetaLayout meta_layout(int64_t batch, int64_t max_groups)
{
    MetaLayout m;
    m.batch_off = kMhWords;
    m.cta_off = m.batch_off + batch * kBatchWords;
    m.group_off = (m.cta_off + kCtaWords * (int64_t)kMaxCtas + 3) & ~int64_t(3);   // 16-byte aligned records
    m.max_groups = max_groups;
    m.total_words = m.group_off + max_groups * kGroupWords;
    if (m.total_words < 1024) m.total_words = 1024;
    return m;
}

namespace {

#ifdef QLI_TESTING
std::atomic<int> g_test_stall{0};
std::atomic<int> g_test_topk_ctas{0};
#endif

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

qli_status check(const qli_problem* p, const char** why)
{
#define QLI_REJECT(cond, msg, st)       \
    do {                                \
        if (cond) {                     \
            if (why) *why = msg;        \
            return st;                  \
        }                               \
    } while (0)
    QLI_REJECT(p == nullptr, "problem is NULL", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->num_heads_q != kHeads, "num_heads_q must be 64", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->num_heads_k != 1, "num_heads_k must be 1", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->head_dim != kDim, "head_dim must be 128", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->qk_dtype != QLI_INT8 && p->qk_dtype != QLI_FP8_E4M3, "qk_dtype must be int8 or fp8 e4m3", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->scale_dtype != QLI_F16 && p->scale_dtype != QLI_F32, "scale_dtype must be f16 or f32", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->layout_q != QLI_BSND && p->layout_q != QLI_TND, "layout_q must be BSND or TND", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->batch < 0, "batch must be >= 0", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->layout_q == QLI_BSND && p->max_q_tokens < 0, "max_q_tokens must be >= 0", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->layout_q == QLI_TND && p->total_q_tokens < 0, "total_q_tokens must be >= 0", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->block_size < 16 || p->block_size > 1024 || p->block_size % 16 != 0,
               "block_size must be a multiple of 16 in [16, 1024]", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->num_blocks < 1, "num_blocks must be >= 1", QLI_ERR_INVALID_ARG);
    QLI_REJECT((int64_t)p->num_blocks * p->block_size >= INT32_MAX, "key pool too large", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->sparse_count < 1 || p->sparse_count > kMaxSparse, "sparse_count must be in [1, 2048]", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->sparse_mode != 0 && p->sparse_mode != 3, "sparse_mode must be 0 or 3", QLI_ERR_INVALID_ARG);
    QLI_REJECT(!is_pow2(p->cmp_ratio) || p->cmp_ratio > 128, "cmp_ratio must be 1, 2, 4, ..., 128", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->query_quant_mode != 0 || p->key_quant_mode != 0, "quant modes must be 0 (per-token-head)", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->pre_tokens != INT64_MAX || p->next_tokens != INT64_MAX, "pre_tokens/next_tokens must be 2^63-1", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->max_seqlen_k < 0 || p->max_seqlen_q < 0, "max_seqlen_q/k must be >= 0", QLI_ERR_INVALID_ARG);
    const int64_t max_lc = compressed_keys(p->max_seqlen_k, p->cmp_ratio);
    QLI_REJECT(p->max_blocks_per_seq < 0 || (int64_t)p->max_blocks_per_seq * p->block_size < max_lc,
               "max_blocks_per_seq too small for max_seqlen_k", QLI_ERR_INVALID_ARG);
    const int64_t rows = p->layout_q == QLI_BSND ? (int64_t)p->batch * p->max_q_tokens : p->total_q_tokens;
    QLI_REJECT(rows >= INT32_MAX, "too many query rows", QLI_ERR_INVALID_ARG);
    QLI_REJECT(rows * ceil_div64(max_lc, kTileKeys) >= INT32_MAX, "problem too large for one call", QLI_ERR_UNSUPPORTED);
    QLI_REJECT(p->return_value != 0 && p->return_value != 1, "return_value must be 0 or 1", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->mask_complete_blocks != 0 && p->mask_complete_blocks != 1, "mask_complete_blocks must be 0 or 1",
               QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->key_stride != 0 && ((int64_t)p->key_stride < (int64_t)p->block_size * 128 || p->key_stride % 16 != 0),
               "key_stride must be 0 or a multiple of 16 of at least block_size * 128", QLI_ERR_INVALID_ARG);
    QLI_REJECT(p->split_topk < QLI_SPLIT_AUTO || p->split_topk > QLI_SPLIT_OFF, "split_topk must be 0, 1 or 2",
               QLI_ERR_INVALID_ARG);
#undef QLI_REJECT
    if (why) *why = "ok";
    return QLI_OK;
}

// Query tokens scored together by one MMA (N = 64 per token): one for one query token per
// sequence; two for two or four (the build with a third accumulator buffer: the fp8 decode's call
// measured 37.4 -> 35.3 us, the page-shaped decode's 28.2 -> 27.2 us); else up to kMultiTokens
// (the TND prefill measured 777 us with groups of three against 897 us with groups of two)
int group_tokens_of(const qli_problem* p)
{
    if (p->layout_q == QLI_BSND) {
        const int s1 = p->max_q_tokens;
        if (s1 <= 1) return 1;
        if (s1 == 2 || s1 == 4) return 2;
        return s1 < kMultiTokens ? s1 : kMultiTokens;
    }
    return kMultiTokens;
}

// Whether the indexer's top-k runs in two stages (split-local selection in the one-token score
// kernel, then the merge): only on request.  Measured on GB300 it is slower than the one-stage
// top-k at every size tried (32 rows of 8k-32k and of 64k-128k keys, k = 64 ... 2048): each chunk's
// selection stalls its CTA's key stream for ~18k cycles (four warps that run alone on their
// sub-partitions), more than the merge saves, so AUTO keeps one stage.
bool split_topk_of(const qli_problem* p, int group_tokens)
{
    return group_tokens == 1 && p->split_topk == QLI_SPLIT_ON;
}

int64_t max_groups_of(const qli_problem* p)
{
    const int gt = group_tokens_of(p);
    if (p->layout_q == QLI_BSND) return (int64_t)p->batch * ceil_div64(p->max_q_tokens, gt);
    return ceil_div64(p->total_q_tokens, gt) + p->batch;
}

Params params_of(const qli_problem* q)
{
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.batch = q->batch;
    p.s1 = q->layout_q == QLI_BSND ? q->max_q_tokens : 0;
    p.total_q = q->layout_q == QLI_TND ? q->total_q_tokens : 0;
    p.layout_tnd = q->layout_q == QLI_TND;
    p.qk_fp8 = q->qk_dtype == QLI_FP8_E4M3;
    p.scale_f32 = q->scale_dtype == QLI_F32;
    p.num_blocks = q->num_blocks;
    p.block_size = q->block_size;
    p.max_blocks_per_seq = q->max_blocks_per_seq;
    p.sparse_count = q->sparse_count;
    p.sparse_mode = q->sparse_mode;
    p.cmp_ratio = q->cmp_ratio;
    p.max_seqlen_q = q->max_seqlen_q;
    p.max_seqlen_k = q->max_seqlen_k;
    int box = 128;
    while (q->block_size % box != 0) box >>= 1;
    p.box_rows = box;
    p.rows = (int32_t)(p.layout_tnd ? (int64_t)p.total_q : (int64_t)p.batch * p.s1);
    const int64_t max_lc = compressed_keys(q->max_seqlen_k, q->cmp_ratio);
    int64_t ld = ceil_div64(max_lc, kTileKeys) * kTileKeys;
    p.ld = ld > 0 ? ld : kTileKeys;
    p.group_tokens = group_tokens_of(q);
    p.meta = meta_layout(p.batch, max_groups_of(q));
    p.hash = problem_hash(p);
    p.complete_blocks = q->mask_complete_blocks;
    p.key_stride = q->key_stride ? q->key_stride : q->block_size * kDim;
    p.split_topk = split_topk_of(q, p.group_tokens) ? 1 : 0;
#ifdef QLI_TESTING
    // failure-detection test switch of the testing build only (no device fault involved): the
    // score kernel's producer issues no copies (1), or its converters consume nothing (2) so the
    // producer's key copies land and wait in the ring; either way the waits run out and report a
    // timeout
    p.test_stall = g_test_stall.load();
#else
    p.test_stall = 0;
#endif
    return p;
}

WsLayout ws_layout(const Params& p)
{
    WsLayout w;
    w.scores_off = kWsHeaderBytes;
    w.ld = p.ld;
    const size_t line = (size_t)p.rows * (size_t)p.ld * sizeof(uint32_t);
    w.cand_code_off = w.scores_off + line;
    w.cand_idx_off = w.cand_code_off;
    w.info_off = w.cand_code_off;
    w.total = w.scores_off + line;
    if (p.split_topk) {
        w.cand_idx_off = w.cand_code_off + line;
        w.info_off = w.cand_idx_off + line;
        w.total = w.info_off + line / kTileKeys;
    }
    return w;
}

// SM count of the current device, cached per device
int device_sms(int* dev_out)
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev_out) *dev_out = dev;
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && cache[dev] > 0) return cache[dev];
    int sms = 0, major = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return -1;
    if (major != 10) return 0;  // tensor memory and tcgen05: sm_100 family only
    if (dev < 64) cache[dev] = sms;
    return sms;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link needed)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Key pool viewed as a 3-D byte tensor [num_blocks pages][block_size keys][128 B] with the page
// stride of the problem (README `stride`); the box is 128 B x box_rows keys x 1 page with the
// 128-byte swizzle the score kernel reads back.
bool encode_key_map(CUtensorMap* tm, const void* key, const Params& p)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)p.block_size, (cuuint64_t)p.num_blocks};
    cuuint64_t strides[2] = {(cuuint64_t)kDim, (cuuint64_t)p.key_stride};
    cuuint32_t box[3] = {(cuuint32_t)kDim, (cuuint32_t)p.box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(key), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


}  // namespace
}  // namespace qli

using namespace qli;

extern "C" {

void qli_problem_init(qli_problem* p)
{
    if (!p) return;
    std::memset(p, 0, sizeof(*p));
    p->num_heads_q = kHeads;
    p->num_heads_k = 1;
    p->head_dim = kDim;
    p->qk_dtype = QLI_INT8;
    p->scale_dtype = QLI_F16;
    p->layout_q = QLI_BSND;
    p->block_size = 128;
    p->num_blocks = 1;
    p->sparse_count = kMaxSparse;
    p->sparse_mode = 0;
    p->cmp_ratio = 1;
    p->pre_tokens = INT64_MAX;
    p->next_tokens = INT64_MAX;
}

qli_status qli_validate(const qli_problem* p, const char** why) { return check(p, why); }

size_t qli_metadata_words(const qli_problem* p)
{
    if (check(p, nullptr) != QLI_OK) return 0;
    return (size_t)params_of(p).meta.total_words;
}

size_t qli_workspace_size(const qli_problem* p)
{
    if (check(p, nullptr) != QLI_OK) return 0;
    return ws_layout(params_of(p)).total;
}

qli_status qli_metadata(const qli_problem* p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                        int32_t* metadata, size_t metadata_words, void* stream)
{
    qli_status s = check(p, nullptr);
    if (s != QLI_OK) return s;
    const Params P = params_of(p);
    if (!metadata || !aligned(metadata, 16)) return QLI_ERR_INVALID_ARG;
    if (metadata_words < (size_t)P.meta.total_words) return QLI_ERR_WORKSPACE_TOO_SMALL;
    if (P.batch > 0 && !seq_lens_k) return QLI_ERR_INVALID_ARG;     // PA_BSND needs key lengths
    if (P.batch > 0 && P.layout_tnd && !seq_lens_q) return QLI_ERR_INVALID_ARG;  // TND needs prefix sums
    int sms = device_sms(nullptr);
    if (sms < 0) return QLI_ERR_CUDA;
    if (sms == 0) return QLI_ERR_NO_DEVICE;
    cudaError_t e = launch_metadata(P, seq_lens_q, seq_lens_k, metadata, score_ctas(sms, P.group_tokens),
                                    score_first_ctas(sms, P.group_tokens), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

namespace {

// Shared argument checks of the score and top-k stages
qli_status check_call(const qli_problem* p, const int32_t* metadata, size_t metadata_words, void* workspace,
                      size_t workspace_bytes, Params* P, WsLayout* W, int* sms)
{
    qli_status s = check(p, nullptr);
    if (s != QLI_OK) return s;
    *P = params_of(p);
    *W = ws_layout(*P);
    if (metadata_words < (size_t)P->meta.total_words || workspace_bytes < W->total) return QLI_ERR_WORKSPACE_TOO_SMALL;
    if (!metadata || !aligned(metadata, 16) || !workspace || !aligned(workspace, 256)) return QLI_ERR_INVALID_ARG;
    *sms = device_sms(nullptr);
    if (*sms < 0) return QLI_ERR_CUDA;
    if (*sms == 0) return QLI_ERR_NO_DEVICE;
    return QLI_OK;
}

}  // namespace

}  // extern "C"

namespace {

// The split-local selection's buffers inside the workspace
SplitBufs split_bufs(uint8_t* ws, const WsLayout& W)
{
    return SplitBufs{reinterpret_cast<uint32_t*>(ws + W.cand_code_off), reinterpret_cast<uint32_t*>(ws + W.cand_idx_off),
                     reinterpret_cast<uint32_t*>(ws + W.info_off)};
}

// The score stage; *launched tells whether a kernel was enqueued
qli_status score_impl(const qli_problem* p, const void* query, const void* key, const void* weights,
                      const void* q_scale, const void* k_scale, const int32_t* seq_lens_q,
                      const int32_t* seq_lens_k, const int32_t* block_table, const int32_t* metadata,
                      size_t metadata_words, void* workspace, size_t workspace_bytes, void* stream,
                      bool* launched)
{
    *launched = false;
    Params P;
    WsLayout W;
    int sms = 0;
    qli_status s = check_call(p, metadata, metadata_words, workspace, workspace_bytes, &P, &W, &sms);
    if (s != QLI_OK) return s;
    if (P.rows == 0 || P.batch == 0) return QLI_OK;
    if (!query || !key || !weights || !q_scale || !k_scale || !seq_lens_k || !block_table) return QLI_ERR_INVALID_ARG;
    if (P.layout_tnd && !seq_lens_q) return QLI_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(key, 16) || !aligned(k_scale, 16) || !aligned(weights, 16) ||
        !aligned(q_scale, 16))
        return QLI_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    CUtensorMap tm;
    if (!encode_key_map(&tm, key, P)) return QLI_ERR_CUDA;
    auto launch = P.group_tokens == 1 ? (P.split_topk ? launch_score_split : launch_score)
                                      : (P.group_tokens == 2 ? launch_score_pair : launch_score_multi);
    cudaError_t e = launch(P, &tm, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table,
                           metadata, reinterpret_cast<uint32_t*>(ws + W.scores_off), split_bufs(ws, W),
                           reinterpret_cast<uint32_t*>(ws), score_ctas(sms, P.group_tokens),
                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return QLI_ERR_CUDA;
    *launched = true;
    return QLI_OK;
}

// The top-k stage; after_score: the launch directly follows this library's score kernel
qli_status topk_impl(const qli_problem* p, const int32_t* block_table, const int32_t* metadata,
                     size_t metadata_words, void* workspace, size_t workspace_bytes, int32_t* sparse_indices,
                     float* sparse_values, void* stream, bool after_score)
{
    Params P;
    WsLayout W;
    int sms = 0;
    qli_status s = check_call(p, metadata, metadata_words, workspace, workspace_bytes, &P, &W, &sms);
    if (s != QLI_OK) return s;
    if ((p->return_value != 0) != (sparse_values != nullptr)) return QLI_ERR_INVALID_ARG;
    if (P.rows == 0) return QLI_OK;
    if (!sparse_indices) return QLI_ERR_INVALID_ARG;
    if (P.batch > 0 && !block_table) return QLI_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // more rows than SMs, each of at most kTopkSmallRows keys (ld bounds every row's visible keys):
    // the two-per-SM form for throughput; few rows: the 1024-thread form for latency
    // (the two-per-SM form runs persistent: one CTA per resident slot, each striding over the rows,
    // which saves a CTA's launch and set-up per row and lets a CTA ask for its next row early)
    // rows longer than one CTA's row cache (and at most four times it), one stage: a cluster of
    // four CTAs per row, each holding a quarter of the row
    if (!P.split_topk && P.ld > kTopkCacheRows && P.ld <= (int64_t)kTopkClusterParts * kTopkCacheRows) {
        cudaError_t e = launch_topk_cluster(P, block_table, metadata, reinterpret_cast<const uint32_t*>(ws + W.scores_off),
                                            reinterpret_cast<uint32_t*>(ws), sparse_indices, sparse_values,
                                            static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
    }
    const bool small = P.ld <= kTopkSmallRows && P.rows > sms;
    auto launch = small ? launch_topk_small : launch_topk;
    int max_ctas = small ? 2 * sms : 0;
#ifdef QLI_TESTING
    const int test_ctas = g_test_topk_ctas.load();
    if (small && test_ctas > 0 && test_ctas < max_ctas) max_ctas = test_ctas;
#endif
    cudaError_t e = launch(P, block_table, metadata, reinterpret_cast<const uint32_t*>(ws + W.scores_off),
                           split_bufs(ws, W), reinterpret_cast<uint32_t*>(ws), sparse_indices, sparse_values,
                           after_score, max_ctas, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

}  // namespace

extern "C" {

qli_status qli_score(const qli_problem* p, const void* query, const void* key, const void* weights,
                     const void* q_scale, const void* k_scale, const int32_t* seq_lens_q,
                     const int32_t* seq_lens_k, const int32_t* block_table, const int32_t* metadata,
                     size_t metadata_words, void* workspace, size_t workspace_bytes, void* stream)
{
    bool launched = false;
    return score_impl(p, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table, metadata,
                      metadata_words, workspace, workspace_bytes, stream, &launched);
}

qli_status qli_topk(const qli_problem* p, const int32_t* block_table, const int32_t* metadata,
                    size_t metadata_words, void* workspace, size_t workspace_bytes, int32_t* sparse_indices,
                    float* sparse_values, void* stream)
{
    return topk_impl(p, block_table, metadata, metadata_words, workspace, workspace_bytes, sparse_indices,
                     sparse_values, stream, false);
}

qli_status qli_score_topk(const qli_problem* p, const void* query, const void* key, const void* weights,
                          const void* q_scale, const void* k_scale, const int32_t* seq_lens_q,
                          const int32_t* seq_lens_k, const int32_t* block_table, const int32_t* metadata,
                          size_t metadata_words, void* workspace, size_t workspace_bytes,
                          int32_t* sparse_indices, float* sparse_values, void* stream)
{
    qli_status s = check(p, nullptr);
    if (s != QLI_OK) return s;
    // validate everything the top-k stage checks before enqueueing the score stage
    if ((p->return_value != 0) != (sparse_values != nullptr)) return QLI_ERR_INVALID_ARG;
    {
        const Params P = params_of(p);
        if (P.rows > 0 && !sparse_indices &&
            metadata_words >= (size_t)P.meta.total_words && workspace_bytes >= ws_layout(P).total)
            return QLI_ERR_INVALID_ARG;
    }
    bool launched = false;
    s = score_impl(p, query, key, weights, q_scale, k_scale, seq_lens_q, seq_lens_k, block_table, metadata,
                   metadata_words, workspace, workspace_bytes, stream, &launched);
    if (s != QLI_OK) return s;
    // the top-k directly follows the score kernel, which let it start only after its own wait on
    // the metadata kernel returned: it may read the metadata before its own wait
    return topk_impl(p, block_table, metadata, metadata_words, workspace, workspace_bytes, sparse_indices,
                     sparse_values, stream, launched);
}

qli_status qli_quantize(int32_t qk_dtype, int32_t scale_dtype, const void* x, int64_t n_vec, void* codes,
                        void* scales, void* stream)
{
    if (qk_dtype != QLI_INT8 && qk_dtype != QLI_FP8_E4M3) return QLI_ERR_INVALID_ARG;
    if (scale_dtype != QLI_F16 && scale_dtype != QLI_F32) return QLI_ERR_INVALID_ARG;
    if (n_vec < 0 || n_vec > (INT64_C(1) << 36)) return QLI_ERR_INVALID_ARG;   // grid.x < 2^31
    if (n_vec == 0) return QLI_OK;
    if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 8) ||
        !aligned(scales, scale_dtype == QLI_F32 ? 4 : 2))
        return QLI_ERR_INVALID_ARG;
    int sms = device_sms(nullptr);
    if (sms < 0) return QLI_ERR_CUDA;
    if (sms == 0) return QLI_ERR_NO_DEVICE;
    cudaError_t e = launch_quantize_vectors(x, n_vec, codes, scales, qk_dtype == QLI_FP8_E4M3,
                                            scale_dtype == QLI_F32, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

qli_status qli_quantize_keys(const qli_problem* p, const void* key_bf16, int64_t tokens, const int32_t* token_batch,
                             const int32_t* token_pos, const int32_t* block_table, void* key, void* k_scale,
                             void* workspace, size_t workspace_bytes, void* stream)
{
    qli_status s = check(p, nullptr);
    if (s != QLI_OK) return s;
    if (tokens < 0 || tokens > (INT64_C(1) << 36)) return QLI_ERR_INVALID_ARG;
    if (workspace && (workspace_bytes < kWsHeaderBytes || !aligned(workspace, 256))) return QLI_ERR_INVALID_ARG;
    if (tokens == 0) return QLI_OK;
    if (!key_bf16 || !token_batch || !token_pos || !block_table || !key || !k_scale) return QLI_ERR_INVALID_ARG;
    if (!aligned(key_bf16, 16) || !aligned(key, 16) || !aligned(k_scale, p->scale_dtype == QLI_F32 ? 4 : 2))
        return QLI_ERR_INVALID_ARG;
    int sms = device_sms(nullptr);
    if (sms < 0) return QLI_ERR_CUDA;
    if (sms == 0) return QLI_ERR_NO_DEVICE;
    const Params P = params_of(p);
    cudaError_t e = launch_quantize_keys(P, key_bf16, tokens, token_batch, token_pos, block_table, key, k_scale,
                                         static_cast<uint32_t*>(workspace), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

qli_status qli_gather_kv(const qli_problem* p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                         const int32_t* block_table, const int32_t* sparse_indices, const void* kv,
                         int64_t entry_bytes, int64_t kv_stride, void* out, int32_t* counts, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    qli_status s = check(p, nullptr);
    if (s != QLI_OK) return s;
    if (entry_bytes < 16 || entry_bytes > 65536 || entry_bytes % 16 != 0) return QLI_ERR_INVALID_ARG;
    const int64_t page_bytes = (int64_t)p->block_size * entry_bytes;
    if (kv_stride != 0 && (kv_stride < page_bytes || kv_stride % 16 != 0)) return QLI_ERR_INVALID_ARG;
    if (workspace && (workspace_bytes < kWsHeaderBytes || !aligned(workspace, 256))) return QLI_ERR_INVALID_ARG;
    const Params P = params_of(p);
    if (P.rows == 0) return QLI_OK;
    if (!sparse_indices || !out || !aligned(out, 16) || (counts && !aligned(counts, 4))) return QLI_ERR_INVALID_ARG;
    if (P.batch > 0 && (!block_table || !kv || !aligned(kv, 16))) return QLI_ERR_INVALID_ARG;
    if (P.layout_tnd && P.batch > 0 && !seq_lens_q) return QLI_ERR_INVALID_ARG;
    if ((int64_t)P.rows * p->sparse_count * (entry_bytes / 16) >= (INT64_C(1) << 40)) return QLI_ERR_UNSUPPORTED;
    int sms = device_sms(nullptr);
    if (sms < 0) return QLI_ERR_CUDA;
    if (sms == 0) return QLI_ERR_NO_DEVICE;
    cudaError_t e = launch_gather(P, seq_lens_q, seq_lens_k, block_table, sparse_indices, kv, entry_bytes,
                                  kv_stride ? kv_stride : page_bytes, out, counts, static_cast<uint32_t*>(workspace),
                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

qli_status qli_workspace_init(void* workspace, size_t workspace_bytes, void* stream)
{
    if (!workspace || workspace_bytes < kWsHeaderBytes || !aligned(workspace, 256)) return QLI_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(workspace, 0, kWsHeaderBytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLI_OK : QLI_ERR_CUDA;
}

qli_status qli_get_device_error(void* workspace, void* stream, uint32_t* bits)
{
    if (!workspace) return QLI_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return QLI_ERR_CUDA;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return QLI_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), st) != cudaSuccess) return QLI_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return QLI_ERR_CUDA;
    if (bits) *bits = word;
    if (word & kErrTimeout) return QLI_ERR_DEVICE_TIMEOUT;
    if (word) return QLI_ERR_DEVICE_BAD_INPUT;
    return QLI_OK;
}

const char* qli_status_string(qli_status s)
{
    switch (s) {
    case QLI_OK: return "ok";
    case QLI_ERR_INVALID_ARG: return "invalid argument";
    case QLI_ERR_UNSUPPORTED: return "unsupported";
    case QLI_ERR_WORKSPACE_TOO_SMALL: return "metadata or workspace buffer too small";
    case QLI_ERR_CUDA: return "CUDA error";
    case QLI_ERR_DEVICE_BAD_INPUT: return "device data invalid (affected rows written as -1)";
    case QLI_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case QLI_ERR_NO_DEVICE: return "no sm_100-family device current";
    }
    return "unknown status";
}

int qli_version(void) { return 100; }

#ifdef QLI_TESTING
void qli_testing_set_stall(int mode) { g_test_stall.store(mode == 1 || mode == 2 ? mode : 0); }
void qli_testing_set_topk_ctas(int ctas) { g_test_topk_ctas.store(ctas > 0 ? ctas : 0); }
#endif

}  // extern "C"

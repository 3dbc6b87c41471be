// qli_internal.cuh -- layouts shared by the host code and the kernels of the CUDA library, plus
// thin wrappers over the sm_100-family PTX the kernels use (mbarrier, TMA, tcgen05).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

#include "qli.h"

namespace qli {

// ------------------------------------------------------------------------------------------------
// Fixed shape of the method (README constraints: N_q = 64, N_k = 1, D = 128)
// ------------------------------------------------------------------------------------------------
constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kMaxSparse = 2048;

// Score kernel tiling: a tile is 128 consecutive compressed keys of one batch (one TMEM lane per
// key); a query group is up to group_tokens consecutive query tokens of one batch scored together
// (MMA N = 64 * tokens).  One query token per sequence (decode): groups of one token, two score CTAs
// per SM (separate CTAs keep more key copies in flight than one CTA with twice the resources).
// Several tokens per sequence: groups of up to kMultiTokens tokens, one CTA per SM with all of the
// SM's tensor memory, each converted key tile serving every token of the group (groups of two for
// decodes of two or four tokens per sequence, which measured faster with a third accumulator
// buffer; groups of three otherwise).
constexpr int kTileKeys = 128;
constexpr int kMultiTokens = 3;
constexpr int kMaxCtas = 1024;            // bound on the split's CTA count (GB300 has 152 SMs)

// Score CTAs of the split on a device with `sms` SMs for groups of `gt` tokens: two per SM less two
// for single-token groups (so that a concurrently resident metadata CTA never delays one), one per
// SM otherwise (at most kMaxCtas)
inline int score_ctas(int sms, int gt)
{
    const int g = gt == 1 ? 2 * sms - 2 : sms;
    return g < 1 ? 1 : (g > kMaxCtas ? kMaxCtas : g);
}

// The CTAs of such a split that are the first to arrive on their SM
inline int score_first_ctas(int sms, int gt)
{
    const int g = score_ctas(sms, gt);
    return gt == 1 ? (sms < g ? sms : g) : g;
}

// Top-k: candidates held per row
constexpr int kTopkCap = 4096;

// Split-local selection (the indexer's top-k in two stages: per split of a row, then across the
// splits).  With it on, each one-token score CTA cuts its share of a row into chunks -- the parts of
// the row's aligned kChunkKeys-key blocks that fall in its range -- and, once a chunk's scores are
// all in its shared memory, keeps the chunk's exact top min(k, chunk keys) by (score descending,
// index ascending).  A chunk of more than k keys writes those k candidates, in index order, to the
// candidate lines at the chunk's own first key; a shorter chunk keeps its keys where the score line
// has them.  One word per 128-key tile of a row says how many candidates the tile's slots hold and
// where (kTileFromCandidates set: the candidate lines; clear: the score line); every tile that has
// visible keys is written on every call, so the top-k reads only current words.
constexpr int kChunkKeys = 4096;
constexpr uint32_t kTileFromCandidates = 0x80000000u;
struct SplitBufs {
    uint32_t* code;   // [rows, ld] candidate codes (ordered uint32 scores)
    uint32_t* idx;    // [rows, ld] candidate key indices
    uint32_t* info;   // [rows, ld / kTileKeys] tile words
};

// Device error bits (sticky word at the start of the workspace)
constexpr uint32_t kErrLength = 1u;       // a length beyond its bound / non-monotone prefix sums
constexpr uint32_t kErrPage = 2u;         // a block_table entry outside [0, num_blocks)
constexpr uint32_t kErrTimeout = 4u;      // a bounded wait gave up
constexpr uint32_t kErrMetadata = 8u;     // metadata buffer not written for this problem

// ------------------------------------------------------------------------------------------------
// Metadata buffer (int32 words), written by qli_metadata, read by qli_score_topk
// ------------------------------------------------------------------------------------------------
constexpr int32_t kMetaMagic = 0x514C4932;  // "QLI2"
enum MetaHeader {
    kMhMagic = 0,
    kMhCtas = 1,        // G: score CTAs the split was made for
    kMhLive = 2,        // live query groups (groups with at least one visible key), records written
    kMhTiles = 3,       // T: key tiles over all live groups
    kMhErr = 4,         // error bits found while reading the lengths
    kMhBatch = 5,
    kMhRows = 6,        // output rows (B * S1 or T)
    kMhGroups = 7,      // query groups, live or not
    kMhLayoutHash = 8,  // hash of the problem fields the split depends on
    kMhFirst = 9,       // G1: the first G1 CTAs are the first to arrive on their SM (see split_start)
    kMhUnitCost = 10,   // kUnitCost: virtual tiles charged to each live group in the split
    kMhWords = 16
};
constexpr int kBatchWords = 8;
enum BatchEntry {
    kBeSq = 0,          // live query rows Sq_b
    kBeSk = 1,          // original key tokens Sk_b
    kBeLc = 2,          // compressed keys Lc_b
    kBeFirstRow = 3,    // first output row of the batch
    kBeOk = 4,          // 1 when the lengths are valid
    kBeGroups = 5,      // query groups ceil(Sq_b / group_tokens) (0 if invalid)
    kBeGroupBase = 6,   // index of the batch's first group
};
// A live query group (group_tokens consecutive live rows of one batch whose last row sees at least
// one key), in batch and row order.  The split cuts a sequence in which every live group occupies
// kUnitCost virtual tiles (the cost of loading and converting its query, which a CTA pays per group
// it touches) followed by its key tiles; the record holds the position of its first key tile in
// that sequence.  The batch's fields travel with the group so that a reader needs one 32-byte load.
constexpr int kUnitCost = 2;
constexpr int kGroupWords = 8;
enum GroupRecord {
    kGrBatch = 0,
    kGrRow = 1,         // first row of the group within its batch
    kGrOutRow = 2,      // first output row of the group
    kGrSq = 3,          // Sq_b
    kGrSk = 4,          // Sk_b
    kGrLc = 5,          // Lc_b
    kGrTile = 6,        // position of the group's first key tile in the split's sequence
    kGrTiles = 7,       // tiles of the group: ceil(visible keys of its last row / kTileKeys)
};
// Per score CTA c (two words): the live groups [first, end) whose key tiles its range of the
// sequence overlaps (first = end when it overlaps none).
constexpr int kCtaWords = 2;

struct MetaLayout {
    int64_t batch_off, cta_off, group_off, total_words;
    int64_t max_groups;
};

// ------------------------------------------------------------------------------------------------
// Workspace (bytes): header (error word ...), then the per-row score lines
// ------------------------------------------------------------------------------------------------
constexpr size_t kWsHeaderBytes = 256;

struct WsLayout {
    size_t scores_off;     // uint32 ordered scores [rows, ld]
    int64_t ld;            // row stride in elements (max Lc rounded up to a tile)
    size_t cand_code_off;  // split-local selection only: candidate codes [rows, ld]
    size_t cand_idx_off;   //   candidate indices [rows, ld]
    size_t info_off;       //   tile words [rows, ld / kTileKeys]
    size_t total;
};

// ------------------------------------------------------------------------------------------------
// Kernel parameter block (host-validated problem plus derived sizes)
// ------------------------------------------------------------------------------------------------
struct Params {
    int32_t batch, s1, total_q, layout_tnd, qk_fp8, scale_f32;
    int32_t num_blocks, block_size, max_blocks_per_seq;
    int32_t sparse_count, sparse_mode, cmp_ratio;
    int32_t max_seqlen_q, max_seqlen_k;
    int32_t box_rows;      // TMA box height (largest power of two <= 128 dividing block_size)
    int32_t rows;          // output rows
    int32_t meta_ctas;     // G
    int32_t hash;
    int32_t test_stall;    // test switch: 1 the score kernel's producer, 2 its converters do nothing
    int32_t complete_blocks;   // mode 3 visibility: 0 ceil((p + 1) / cmp), 1 floor((p + 1) / cmp)
    int32_t key_stride;        // elements between key pages
    int32_t group_tokens;      // query tokens per group (1, or up to kMultiTokens)
    int32_t split_topk;        // 1: split-local selection (one-token groups only), then the merge
    int64_t ld;            // score line stride
    MetaLayout meta;
};

// ---------------------------------------------------------------------------- shared helpers
__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// log2 of a power-of-two cmp_ratio (validated on the host)
__host__ __device__ inline int log2_pow2(int v)
{
    int s = 0;
    while ((1 << s) < v) ++s;
    return s;
}

// Compressed keys of a batch with sk original tokens: ceil(sk / cmp)
__host__ __device__ inline int64_t compressed_keys(int64_t sk, int cmp)
{
    return (sk + cmp - 1) >> log2_pow2(cmp);
}

// Visible compressed keys of live row r (0 <= r < sq); mode 3 counts the compressed blocks that
// have started at or before the row's right-aligned original position, ceil((pos + 1) / cmp), or
// with `complete` only those that have ended, floor((pos + 1) / cmp).
__host__ __device__ inline int64_t visible_keys(int mode, int cmp, int64_t sq, int64_t sk, int64_t lc,
                                                int64_t r, int complete)
{
    if (r < 0 || r >= sq) return 0;
    if (mode == 0) return lc;
    const int64_t pos = sk - sq + r;
    if (pos < 0) return 0;
    const int64_t n = (pos + (complete ? 1 : cmp)) >> log2_pow2(cmp);
    return n < lc ? n : lc;
}

// Extents of batch b read from the device lengths (the metadata's definition, shared by every
// kernel that derives it): live query rows sq, key tokens sk (0 when invalid), compressed keys lc,
// first output row, validity, and whether b's TND prefix sums are themselves invalid (which
// invalidates every batch).  A batch is invalid when a length is negative or beyond its bound
// (BSND seq_lens_q above S1, TND prefix sums not non-decreasing or beyond T, seq_lens_k above
// max_seqlen_k, more compressed keys than the block_table row holds).
struct BatchExtent {
    int32_t sq, sk, lc, first;
    bool ok, tnd_bad;
};

__device__ __forceinline__ BatchExtent batch_extent(const Params& p, const int32_t* seq_lens_q,
                                                    const int32_t* seq_lens_k, int b)
{
    BatchExtent e{0, 0, 0, 0, true, false};
    int64_t sq = 0, first = 0;
    if (!p.layout_tnd) {
        first = (int64_t)b * p.s1;
        const int64_t v = seq_lens_q ? seq_lens_q[b] : p.s1;
        e.ok = v >= 0 && v <= p.s1;
        sq = e.ok ? v : 0;
    } else {
        const int64_t lo = b > 0 ? seq_lens_q[b - 1] : 0, hi = seq_lens_q[b];
        e.ok = lo >= 0 && hi >= lo && hi <= p.total_q;
        e.tnd_bad = !e.ok;
        first = lo < 0 ? 0 : lo;
        sq = e.ok ? hi - lo : 0;
    }
    const int64_t sk = seq_lens_k[b];
    e.ok = e.ok && sk >= 0 && sk <= p.max_seqlen_k;
    const int64_t lc = e.ok ? compressed_keys(sk, p.cmp_ratio) : 0;
    e.ok = e.ok && lc <= (int64_t)p.max_blocks_per_seq * p.block_size;
    e.sq = (int32_t)sq;
    e.sk = (int32_t)(e.ok ? sk : 0);
    e.lc = (int32_t)lc;
    e.first = (int32_t)first;
    return e;
}

// Key tiles of the query group of batch rows [r0, min(r0 + gt, sq)): ceil(n / kTileKeys), n the
// visible keys of its last row (the largest in the group under either mask)
__host__ __device__ inline int64_t group_tiles(const Params& p, int64_t sq, int64_t sk, int64_t lc, int64_t r0)
{
    const int64_t rl = (r0 + p.group_tokens < sq ? r0 + p.group_tokens : sq) - 1;
    const int64_t n = visible_keys(p.sparse_mode, p.cmp_ratio, sq, sk, lc, rl, p.complete_blocks);
    return (n + kTileKeys - 1) / kTileKeys;
}

// Problem fields the metadata depends on, folded into one word to catch mismatched buffers
__host__ __device__ inline int32_t problem_hash(const Params& p)
{
    uint32_t h = 2166136261u;
    const int32_t f[] = {p.batch, p.s1, p.total_q, p.layout_tnd, p.sparse_mode, p.cmp_ratio,
                         p.max_seqlen_q, p.max_seqlen_k, p.block_size, p.max_blocks_per_seq,
                         p.complete_blocks, p.group_tokens};
    for (int i = 0; i < 12; ++i) { h ^= (uint32_t)f[i]; h *= 16777619u; }
    return (int32_t)(h & 0x7fffffff);
}

MetaLayout meta_layout(int64_t batch, int64_t max_groups);

// The split of the T tiles over G score CTAs: W(c) is the weight of CTAs 0 .. c - 1, and CTA c owns
// tiles [T W(c) / W(G), T W(c + 1) / W(G)).  The CTAs that arrive first on their SM (0 .. G1 - 1)
// may weigh kSplitFirst against the others' kSplitSecond; they weigh the same: with a three-stage
// key ring the first and second CTA of an SM stream equally fast, and any skew (12 : 11, 13 : 11,
// 11 : 12, 10 : 11 tried) left the long decode's score kernel ~2 us longer than equal ranges.
// (T < 2^31 and W(G) < 2^14, so the product fits.)
constexpr int64_t kSplitFirst = 1, kSplitSecond = 1;

__host__ __device__ inline int64_t split_weight(int64_t G1, int64_t c)
{
    return c <= G1 ? c * kSplitFirst : G1 * kSplitFirst + (c - G1) * kSplitSecond;
}

// First tile of score CTA c's range
__host__ __device__ inline int64_t split_start(int64_t T, int64_t G, int64_t G1, int64_t c)
{
    return (T * split_weight(G1, c)) / split_weight(G1, G);
}

// Launch `kernel` with programmatic stream serialization: it may begin launching while the
// previous kernel in the stream finishes; every kernel of this library calls griddepcontrol.wait
// before touching memory another kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (defined in the kernel translation units)
cudaError_t launch_metadata(const Params& p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                            int32_t* meta, int num_ctas, int first_ctas, cudaStream_t st);
// (the score launchers share one signature; only launch_score_split writes `split`)
cudaError_t launch_score(const Params& p, const void* tmap_key, const void* query, const void* key,
                         const void* weights, const void* q_scale, const void* k_scale,
                         const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                         const int32_t* block_table, const int32_t* meta, uint32_t* scores,
                         const SplitBufs& split, uint32_t* err_word, int grid, cudaStream_t st);
cudaError_t launch_score_multi(const Params& p, const void* tmap_key, const void* query, const void* key,
                               const void* weights, const void* q_scale, const void* k_scale,
                               const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                               const int32_t* block_table, const int32_t* meta, uint32_t* scores,
                               const SplitBufs& split, uint32_t* err_word, int grid, cudaStream_t st);
cudaError_t launch_score_pair(const Params& p, const void* tmap_key, const void* query, const void* key,
                              const void* weights, const void* q_scale, const void* k_scale,
                              const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                              const int32_t* block_table, const int32_t* meta, uint32_t* scores,
                              const SplitBufs& split, uint32_t* err_word, int grid, cudaStream_t st);
cudaError_t launch_score_split(const Params& p, const void* tmap_key, const void* query, const void* key,
                               const void* weights, const void* q_scale, const void* k_scale,
                               const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                               const int32_t* block_table, const int32_t* meta, uint32_t* scores,
                               const SplitBufs& split, uint32_t* err_word, int grid, cudaStream_t st);
// (max_ctas > 0: at most that many CTAs, each striding over the rows; else one CTA per row;
// `split` is read when p.split_topk is set)
cudaError_t launch_topk(const Params& p, const int32_t* block_table, const int32_t* meta,
                        const uint32_t* scores, const SplitBufs& split, uint32_t* err_word, int32_t* out,
                        float* values, bool after_score, int max_ctas, cudaStream_t st);
// the one-stage top-k for rows longer than the 1024-thread form's row cache (kTopkCacheRows keys) and
// at most kTopkClusterParts times it: a cluster of that many CTAs per row
constexpr int kTopkCacheRows = 32768;
constexpr int kTopkClusterParts = 4;
cudaError_t launch_topk_cluster(const Params& p, const int32_t* block_table, const int32_t* meta,
                                const uint32_t* scores, uint32_t* err_word, int32_t* out, float* values,
                                cudaStream_t st);
// the same top-k with half the threads and a row cache of kTopkSmallRows keys (two CTAs per SM)
constexpr int kTopkSmallRows = 8192;
cudaError_t launch_topk_small(const Params& p, const int32_t* block_table, const int32_t* meta,
                              const uint32_t* scores, const SplitBufs& split, uint32_t* err_word, int32_t* out,
                              float* values, bool after_score, int max_ctas, cudaStream_t st);
cudaError_t launch_quantize_vectors(const void* x_bf16, int64_t nvec, void* codes, void* scales, bool fp8,
                                    bool scale_f32, cudaStream_t st);
cudaError_t launch_quantize_keys(const Params& p, const void* k_bf16, int64_t tokens, const int32_t* tok_batch,
                                 const int32_t* tok_pos, const int32_t* block_table, void* pool, void* k_scale,
                                 uint32_t* err, cudaStream_t st);
cudaError_t launch_gather(const Params& p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                          const int32_t* block_table, const int32_t* idx, const void* kv, int64_t entry_bytes,
                          int64_t kv_stride, void* out, int32_t* counts, uint32_t* err, cudaStream_t st);

}  // namespace qli

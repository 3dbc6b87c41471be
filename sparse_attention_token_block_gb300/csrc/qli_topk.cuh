// qli_topk.cuh -- per-row top-k over the score lines (README function section, step 3: select the
// top-k indices; parameter table: sparse_count, sparse_indices).  Included by the translation units
// that size the CTA:
//   qli_topk.cu         1024 threads, rows of up to 32768 keys cached, 8192 ordering bins: one CTA
//                       per SM (decode rows of up to 32k keys, latency first);
//   qli_topk_small.cu   512 threads, rows of up to 8192 keys cached, 2048 bins, about 90 KB of
//                       shared memory: two CTAs per SM (problems whose rows hold at most 8192 keys,
//                       such as a prefill's many rows: throughput first);
//   qli_topk_cluster.cu the helpers only, for its cluster kernel (rows of 32k to 128k keys).
//
// One CTA per output row.  Scores are held as order-preserving uint32 codes; a key's
// full sort key is (code << 32) | (0xFFFFFFFF - index): score descending, then index ascending.
//
// Rows of up to kCacheKeys keys are bulk-copied into shared memory and ordered by bins:
//   1. the code range [lo, hi] of the row is cut into kBins equal bins (bin 0 holds the highest
//      codes) and one pass counts the keys per bin;
//   2. a scan finds the bin where the running count reaches min(k, n); every key in it or in a
//      higher bin is a candidate, and the scan gives each bin its place in the candidate array;
//   3. one pass scatters the candidates into their bins;
//   4. each candidate's position is its bin's start plus the number of candidates of its bin with a
//      larger sort key.
// Longer rows first gather, in one pass over global memory, the keys at or above a threshold code:
// the rank-r largest of 2048 evenly spaced keys of the row (radix select over the samples), with
// r = 1.15 k S / n + 4 sqrt(k S / n) + 2, which leaves between k and kCap keys at or above it with
// overwhelming probability; the same bins then order them.  Whenever the candidates would exceed
// kCap (heavy ties) an exact radix select on the 64-bit sort keys finds the k-th key and exactly k
// keys are gathered; when a bin holds more than kBigBucket candidates, a block-wide bitonic sort
// orders them instead of step 4.
// With the split-local selection on, a row's candidates are the keys each chunk of the score
// CTAs kept (see SplitBufs): the row's tile words give each 128-key tile's count and source, a scan
// gives each tile its place, and the candidates are gathered into the row cache in index order;
// the same steps then order them by position, which follows index order, and each position is
// mapped back to its key index.  Rows whose candidates do not fit (more than kSplitKeys, or more
// than kSplitTiles tiles) are ordered from the whole score line, which the score kernel still
// writes.
// The first min(k, n) indices are written, then -1 up to sparse_count.  Rows with no visible key,
// rows of an invalid batch and rows whose batch's block_table names a page outside the pool are all
// -1.
#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

#if !defined(QLI_TOPK_THREADS) || !defined(QLI_TOPK_CACHE_KEYS) || !defined(QLI_TOPK_BINS) || !defined(QLI_TOPK_LAUNCHER)
#error "include through qli_topk.cu or qli_topk_small.cu"
#endif
// The phases every ordered row runs (sampling, compaction, bin counts and order, the short rows'
// ranking) are inlined in every build: out of line, each first call fetched its code from DRAM
// after an L2 flush (long decode top-k 18.3 -> 17.0 us inlined, fp8 decode 18.1 -> 16.3 us).  The
// rarer ones (the exact fallback, the bitonic network, the uncached rows' gather, the merge) stay
// out of line in the one-per-SM build, whose decode call measured faster so, and are inlined in
// the two-per-SM build, whose 64 registers a thread otherwise went through local memory at every
// call (prefill top-k 446 -> 430 us)
#if QLI_TOPK_THREADS == 512
#define QLI_TOPK_FN __forceinline__
#else
#define QLI_TOPK_FN __noinline__
#endif
constexpr int kThreads = QLI_TOPK_THREADS;
constexpr int kCtasPerSm = kThreads == 1024 ? 1 : 2;
constexpr int kWarps = kThreads / 32;
constexpr int kSampleKeys = 1024;             // keys sampled to bound the candidates' codes
constexpr int kCap = kTopkCap;                // candidates held in shared memory
constexpr int kSamples = 8192;               // samples of an uncached row (held in the row cache)
constexpr int kBins = QLI_TOPK_BINS;          // ordering bins
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kSampleBins = 2048;             // bins of the sample histogram
constexpr int kBigBucket = 256;
constexpr int kCacheKeys = QLI_TOPK_CACHE_KEYS;   // score lines up to this length are cached in smem
static_assert(kCacheKeys >= 2 * kTopkCap, "the row cache doubles as the uncached rows' scatter target");
static_assert(kCacheKeys >= kSamples, "the row cache holds an uncached row's samples");
constexpr int kMiscWords = 128;               // scratch: [0, 64) block reductions, [100, 111) single values,
                                              // [116, 124) the row places handed over
constexpr int kSmemBytes = (kCacheKeys + kBins + 3 * kCap + 256 + kMiscWords) * 4 + 16;
// Split-local candidates: gathered into the row cache from word kSplitBase on (the sampled path
// scatters into the first 2 kCap words), at most kSplitKeys of them; tile offsets for rows of up
// to kSplitTiles tiles follow the rest of shared memory
constexpr int kSplitBase = kCacheKeys >= 3 * kCap ? 2 * kCap : 0;
constexpr int kSplitKeys = kSplitBase > 0 ? kCacheKeys - kSplitBase : kCap;
constexpr int kSplitTiles = kThreads == 1024 ? 2048 : kCacheKeys / kTileKeys;
constexpr int kSmemSplitBytes = kSmemBytes + (kSplitTiles + 1) * 4;
static_assert(kSmemSplitBytes <= 227 * 1024, "shared memory");
// The two-per-SM build's CTAs take many rows each: their places are worked out ahead and each
// next line is copied as soon as the row cache is free
constexpr bool kPipe = kCtasPerSm == 2;

struct TopkArgs {
    Params p;
    const int32_t* block_table;
    const int32_t* meta;
    const uint32_t* scores;
    uint32_t* err;
    int32_t* out;
    float* values;     // optional: the score of each index written, -inf beside -1
    SplitBufs split;   // the split-local candidates (read by the merging build only)
    // 1 when this launch directly follows the library's score kernel in the stream: that kernel
    // lets its dependents start only after its own griddepcontrol.wait returned, i.e. after the
    // metadata kernel before it had completed, so the metadata and the (unchanged) block_table can
    // be read before this kernel's own wait; 0 for a standalone top-k launch
    int32_t early;
};

// Where output row `row` lives: its batch b, row r within the batch, visible keys n and the
// batch's compressed length lc (n = 0 for rows of no batch or an invalid one).  Loads bypass L1.
struct RowInfo {
    int64_t b, r, n, lc;
};

__device__ RowInfo row_info(const TopkArgs& a, bool meta_ok, int64_t row)
{
    const Params& p = a.p;
    const int32_t* be = a.meta + p.meta.batch_off;
    RowInfo ri{-1, 0, 0, 0};
    if (!meta_ok || p.batch <= 0) return ri;
    if (!p.layout_tnd) {
        ri.b = row / p.s1;
        ri.r = row % p.s1;
    } else {
        int64_t lo = 0, hi = p.batch - 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (__ldcg(be + mid * kBatchWords + kBeFirstRow) <= row) lo = mid; else hi = mid - 1;
        }
        ri.b = lo;
    }
    const int4 e0 = __ldcg(reinterpret_cast<const int4*>(be + ri.b * kBatchWords));       // sq, sk, lc, first
    const int ok = __ldcg(be + ri.b * kBatchWords + kBeOk);
    if (p.layout_tnd) ri.r = row - e0.w;
    ri.lc = e0.z;
    if (ok && ri.r >= 0) ri.n = visible_keys(p.sparse_mode, p.cmp_ratio, e0.x, e0.y, ri.lc, ri.r, p.complete_blocks);
    return ri;
}

struct Smem {
    uint32_t* cache;  // [kCacheKeys] one score line (uncached rows: scatter targets)
    uint32_t* bins;   // [kBins] bin counts, then bin ends / starts; bitonic scratch
    uint32_t* key;    // [kCap] candidate codes
    uint32_t* val;    // [kCap] candidate indices
    uint32_t* outv;   // [kCap] ordered indices
    uint32_t* hist;   // [256] radix-select digits
    uint32_t* misc;   // [kMiscWords] reduction scratch
    uint64_t* bar;    // bulk-copy barrier
    uint32_t* toff;   // merging build: [kSplitTiles + 1] tile offsets (kTileFromCandidates: source)
};

extern __shared__ __align__(16) uint8_t topk_smem[];

// The CTA's shared-memory carve-up, rebuilt from the dynamic shared memory symbol (cheaper than
// passing it to non-inlined functions through local memory)
__device__ __forceinline__ Smem smem_view()
{
    Smem S;
    S.cache = reinterpret_cast<uint32_t*>(topk_smem);
    S.bins = S.cache + kCacheKeys;
    S.key = S.bins + kBins;
    S.val = S.key + kCap;
    S.outv = S.val + kCap;
    S.hist = S.outv + kCap;
    S.misc = S.hist + 256;
    S.bar = reinterpret_cast<uint64_t*>(S.misc + kMiscWords);
    S.toff = reinterpret_cast<uint32_t*>(topk_smem + kSmemBytes);
    return S;
}

__device__ __forceinline__ uint64_t sort_key(uint32_t code, uint32_t idx)
{
    return (static_cast<uint64_t>(code) << 32) | (0xFFFFFFFFu - idx);
}

// Block-wide exclusive scan of one value per thread; also returns the total.  One barrier: every
// warp scans the 32 warp totals itself.  `sh` (kWarps words) must not be written again before a
// later barrier.
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t* total, uint32_t* sh)
{
    static_assert(kWarps <= 32, "one warp total per lane");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    const uint32_t wt = lane < kWarps ? sh[lane] : 0u;
    uint32_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
    }
    *total = __shfl_sync(0xffffffffu, wi, 31);
    return __shfl_sync(0xffffffffu, wi - wt, warp) + x - v;
}

// Radix select over 64-bit sort keys produced by `get(i)` for i < n: the k-th largest key
// (one shared 256-bin histogram per 8-bit digit, counts aggregated per warp before the atomic).
template <class Get>
__device__ uint64_t radix_select(const Smem& S, int64_t n, int k, Get get, int top_shift)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* s_digit = S.misc + 100;
    uint32_t* s_rem = S.misc + 101;
    uint32_t* s_done = S.misc + 102;
    uint64_t prefix = 0, mask = 0;
    uint32_t rem = (uint32_t)k;
    for (int shift = top_shift; shift >= 0; shift -= 8) {
        if (tid < 256) S.hist[tid] = 0;
        __syncthreads();
        for (int64_t i0 = 0; i0 < n; i0 += kThreads) {
            const int64_t i = i0 + tid;
            bool in = false;
            uint32_t digit = 0;
            if (i < n) {
                const uint64_t c = get(i);
                in = (c & mask) == prefix;
                digit = (uint32_t)(c >> shift) & 0xFFu;
            }
            const unsigned act = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned peers = __match_any_sync(act, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&S.hist[digit], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t c8[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c8[q] = S.hist[255 - 8 * lane - q];
                sum += c8[q];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - sum;
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
            if (lane == __ffs(hit) - 1) {
                uint32_t above = excl;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (above + c8[q] >= rem) {
                        *s_digit = 255 - 8 * lane - q;
                        *s_rem = rem - above;
                        *s_done = (c8[q] == rem - above) ? 1u : 0u;
                        break;
                    }
                    above += c8[q];
                }
            }
        }
        __syncthreads();
        prefix |= (uint64_t)*s_digit << shift;
        mask |= (uint64_t)0xFFu << shift;
        rem = *s_rem;
        const bool done = *s_done != 0;
        __syncthreads();
        if (done) break;
    }
    return prefix;
}

// Gather (unordered) into key/val the keys j < n of `line` (shared or global memory) whose sort
// key is >= t64; returns how many (only the first kCap are stored).  Each thread loads its kGatherU
// keys of a stretch before testing any: over a score line in global memory one load at a time
// left the loop waiting on each load's latency (a 2^17-key row: ~130 loads in a row per thread).
constexpr int kGatherU = 8;
__device__ int gather(const Smem& S, const uint32_t* line, int64_t n, uint64_t t64)
{
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t* s_cnt = S.misc + 104;
    if (tid == 0) *s_cnt = 0;
    __syncthreads();
    for (int64_t j0 = 0; j0 < n; j0 += (int64_t)kThreads * kGatherU) {
        uint32_t c[kGatherU];
#pragma unroll
        for (int u = 0; u < kGatherU; ++u) {
            const int64_t j = j0 + u * kThreads + tid;
            c[u] = j < n ? line[j] : 0u;
        }
#pragma unroll
        for (int u = 0; u < kGatherU; ++u) {
            const int64_t j = j0 + u * kThreads + tid;
            const bool take = j < n && sort_key(c[u], (uint32_t)j) >= t64;
            const unsigned bal = __ballot_sync(0xffffffffu, take);
            if (bal) {
                uint32_t base = 0;
                if (lane == 0) base = atomicAdd(s_cnt, (uint32_t)__popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (take) {
                    const uint32_t pos = base + __popc(bal & ((1u << lane) - 1u));
                    if (pos < (uint32_t)kCap) {
                        S.key[pos] = c[u];
                        S.val[pos] = (uint32_t)j;
                    }
                }
            }
        }
    }
    __syncthreads();
    return (int)*s_cnt;
}

// Descending bitonic sort of kThreads * E 64-bit keys, thread t holding positions t*E .. t*E+E-1.
template <int E>
__device__ void bitonic_desc(uint64_t (&v)[E], uint64_t* xbuf)
{
    constexpr int P = kThreads * E;
    const int tid = threadIdx.x;
#pragma unroll 1
    for (int k = 2; k <= P; k <<= 1) {
#pragma unroll 1
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j < E) {
#pragma unroll
                for (int jj = 1; jj < E; jj <<= 1) {
                    if (jj == j) {
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const int pe = e ^ jj;
                            if (pe > e) {
                                const bool desc = ((tid * E + e) & k) == 0;
                                const uint64_t x = v[e], y = v[pe];
                                if (desc ? (x < y) : (x > y)) {
                                    v[e] = y;
                                    v[pe] = x;
                                }
                            }
                        }
                    }
                }
            } else if (j < 32 * E) {
                const int lm = j / E;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = tid * E + e;
                    const uint64_t other = __shfl_xor_sync(0xffffffffu, v[e], lm);
                    const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
                    v[e] = keep_max ? (v[e] > other ? v[e] : other) : (v[e] < other ? v[e] : other);
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) xbuf[tid * E + e] = v[e];
                __syncthreads();
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = tid * E + e;
                    const uint64_t other = xbuf[i ^ j];
                    const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
                    v[e] = keep_max ? (v[e] > other ? v[e] : other) : (v[e] < other ? v[e] : other);
                }
                __syncthreads();
            }
        }
    }
}

// Order keys[0..c) / vals[0..c) descending by sort key with the bitonic network (c <= kThreads *
// E); the ordered indices end in vals.  `scratch` holds kThreads * E 64-bit words.
template <int E>
__device__ void bitonic_order(uint32_t* keys, uint32_t* vals, int c, uint64_t* scratch)
{
    uint64_t v[E];
    const int tid = threadIdx.x;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        v[e] = i < c ? sort_key(keys[i], vals[i]) : 0ull;   // 0 sorts below every real key
    }
    __syncthreads();
    bitonic_desc<E>(v, scratch);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        if (i < c) vals[i] = 0xFFFFFFFFu - (uint32_t)(v[e] & 0xFFFFFFFFu);
    }
    __syncthreads();
}

// Rarely taken: heavy ties in one bin (or the exact fallback)
__device__ QLI_TOPK_FN void bitonic_any(uint32_t* keys, uint32_t* vals, int c, uint64_t* scratch)
{
    constexpr int kMaxE = kCap / kThreads;          // c <= kCap
    static_assert(kMaxE * kThreads == kCap && kMaxE <= 16, "the network covers kCap keys");
    if (c <= kThreads) bitonic_order<1>(keys, vals, c, scratch);
    else if (c <= 2 * kThreads) bitonic_order<2>(keys, vals, c, scratch);
    else if (c <= 4 * kThreads || kMaxE <= 4) bitonic_order<(kMaxE < 4 ? kMaxE : 4)>(keys, vals, c, scratch);
    else if (c <= 8 * kThreads || kMaxE <= 8) bitonic_order<(kMaxE < 8 ? kMaxE : 8)>(keys, vals, c, scratch);
    else bitonic_order<(kMaxE < 16 ? kMaxE : 16)>(keys, vals, c, scratch);
}

// Largest of one value per thread and smallest of another, returned to every thread.  One
// barrier; `sh` (64 words) must not be written again before a later barrier.
__device__ void block_max_min(uint32_t* mx, uint32_t* mn, uint32_t* sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t a = *mx, b = *mn;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = min(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
        sh[warp] = a;
        sh[32 + warp] = b;
    }
    __syncthreads();
    a = lane < kWarps ? sh[lane] : 0u;
    b = lane < kWarps ? sh[32 + lane] : 0xFFFFFFFFu;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = min(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    *mx = a;
    *mn = b;
}

// The bins: codes in [L, top] fall in bin (top - code) >> shift (codes above top share bin 0);
// bin 0 holds the highest codes.
struct Binning {
    uint32_t L, top;
    int shift;
    __device__ uint32_t operator()(uint32_t x) const { return x >= top ? 0u : (top - x) >> shift; }
};

__device__ Binning make_binning(uint32_t L, uint32_t top)
{
    Binning g;
    g.L = L;
    g.top = top;
    g.shift = 0;
    while (g.shift < 32 && ((top - L) >> g.shift) >= (uint32_t)kBins) ++g.shift;
    return g;
}

// Steps 1-2 over src[0..c) (shared memory, 16-byte aligned, c <= kCacheKeys): each thread tests
// its keys (4 * kVecPerThread of them, four at a time) against g.L and keeps one bit per key; a
// scan of the per-thread counts gives each thread its offset, and each thread then visits only
// its set bits, appending those keys to S.key / S.val and counting them in their bins (if
// `count`).  Visiting set bits keeps the warp on the ~15 % of keys that pass instead of taking
// the append path for every key position.  Returns how many keys reached g.L (only the first
// kCap are stored or counted).
constexpr int kVecPerThread = kCacheKeys / (4 * kThreads);
static_assert(kVecPerThread * 4 <= 32, "one pass bit per key in a 32-bit mask");
__device__ __forceinline__ int compact_and_count(const uint32_t* src, int c, Binning g, bool count)
{
    const Smem S = smem_view();
    const int tid = threadIdx.x;
    if (count)
        for (int b = tid; b < kBins; b += kThreads) S.bins[b] = 0;
    const int c4 = c >> 2;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    const uint32_t L = g.L;
    uint32_t mask = 0;                 // bit 4q + e: key e of this thread's vector q passes
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
        const int i = tid + q * kThreads;
        if (i < c4) {
            const uint4 v = s4[i];
            mask |= ((v.x >= L ? 1u : 0u) | (v.y >= L ? 2u : 0u) | (v.z >= L ? 4u : 0u) | (v.w >= L ? 8u : 0u))
                    << (4 * q);
        }
    }
    // the c mod 4 keys past the last full vector: thread t < c - 4 c4 takes key 4 c4 + t
    const int tail = c - 4 * c4;
    const bool tail_in = tid < tail && src[4 * c4 + tid] >= L;
    uint32_t total;
    uint32_t pos = block_excl_scan(__popc(mask) + (tail_in ? 1u : 0u), &total, S.misc);
    auto put = [&](uint32_t x, int j) {
        if (pos < (uint32_t)kCap) {
            S.key[pos] = x;
            S.val[pos] = (uint32_t)j;
            if (count) atomicAdd(&S.bins[g(x)], 1u);
        }
        ++pos;
    };
    while (mask) {
        const int bit = __ffs(mask) - 1;
        mask &= mask - 1;
        const int j = 4 * (tid + (bit >> 2) * kThreads) + (bit & 3);
        put(src[j], j);
    }
    if (tail_in) put(src[4 * c4 + tid], 4 * c4 + tid);
    __syncthreads();
    return (int)total;
}

// Bin counts of the m listed candidates lkey[0..m) (shared memory)
__device__ __forceinline__ void count_bins(const uint32_t* lkey, int m, Binning g)
{
    const Smem S = smem_view();
    const int tid = threadIdx.x;
    for (int b = tid; b < kBins; b += kThreads) S.bins[b] = 0;
    __syncthreads();
    for (int i = tid; i < m; i += kThreads) atomicAdd(&S.bins[g(lkey[i])], 1u);
    __syncthreads();
}

enum BinResult { kBinOrdered = 0, kBinTooMany = 1 };

// Steps 3-4 over the m listed candidates lkey / lval (lval null: a candidate's index is its
// position; bins counted): the scan finds the bin where
// the running count reaches need; the candidates of that bin and above are scattered into
// tkey / tval (kCap words each, tval = tkey + kCap) and each takes its bin's start plus its rank
// among the bin's keys; the
// first min(need, m) indices of the order go to S.outv.  A bin of more than kBigBucket candidates
// sends them to the bitonic network instead.  kBinTooMany: fewer than `need` candidates or more
// than kCap up to the threshold bin (nothing ordered).
__device__ __forceinline__ int order_bins(const uint32_t* lkey, const uint32_t* lval, int m, int need, Binning g,
                                       uint32_t* tkey, uint32_t* tval)
{
    const Smem S = smem_view();
    const int tid = threadIdx.x;
    uint32_t* bins = S.bins;
    // thread t scans bins [8t, 8t + 8)
    static_assert(kBinsPerThread % 4 == 0, "16-byte loads");
    uint32_t cnt[kBinsPerThread], sum = 0;
    {
        const uint4* b4 = reinterpret_cast<const uint4*>(bins) + (kBinsPerThread / 4) * tid;
#pragma unroll
        for (int v = 0; v < kBinsPerThread / 4; ++v) {
            const uint4 c = b4[v];
            cnt[4 * v] = c.x;
            cnt[4 * v + 1] = c.y;
            cnt[4 * v + 2] = c.z;
            cnt[4 * v + 3] = c.w;
        }
    }
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) sum += cnt[q];
    uint32_t total;
    const uint32_t before = block_excl_scan(sum, &total, S.misc);
    uint32_t* s_thr = S.misc + 108;
    uint32_t* s_cc = S.misc + 109;
    if (before < (uint32_t)need && before + sum >= (uint32_t)need) {
        uint32_t run = before;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            if (run < (uint32_t)need && run + cnt[q] >= (uint32_t)need) {
                *s_thr = tid * kBinsPerThread + q;
                *s_cc = run + cnt[q];
            }
            run += cnt[q];
        }
    }
    __syncthreads();
    const uint32_t thr = *s_thr;
    const int cc = (int)*s_cc;
    if (total < (uint32_t)need || m > kCap || cc > kCap) {
        __syncthreads();
        return kBinTooMany;
    }
    // bin ends (inclusive prefix) for the scatter, which fills each bin from its end
    bool big = false;
    {
        uint32_t run = before, end[kBinsPerThread];
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            const uint32_t b = tid * kBinsPerThread + q;
            run += cnt[q];
            end[q] = run;
            big |= b <= thr && cnt[q] > (uint32_t)kBigBucket;
        }
        uint4* b4 = reinterpret_cast<uint4*>(bins) + (kBinsPerThread / 4) * tid;
#pragma unroll
        for (int v = 0; v < kBinsPerThread / 4; ++v)
            b4[v] = make_uint4(end[4 * v], end[4 * v + 1], end[4 * v + 2], end[4 * v + 3]);
    }
    big = __syncthreads_or(big);
    // 3. scatter the candidates up to the threshold bin
    constexpr int kPer = kCap / kThreads;           // m <= kCap: at most kPer per thread
    if (big || !kPipe) {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = tid + q * kThreads;
            if (i < m) {
                const uint32_t x = lkey[i];
                const uint32_t b = g(x);
                if (b <= thr) {
                    const uint32_t pos = atomicSub(&bins[b], 1u) - 1u;
                    tkey[pos] = x;
                    tval[pos] = lval ? lval[i] : (uint32_t)i;
                }
            }
        }
        __syncthreads();
        if (big) {
            bitonic_any(tkey, tval, cc, reinterpret_cast<uint64_t*>(S.bins));
            for (int i = tid; i < need; i += kThreads) S.outv[i] = tval[i];
            __syncthreads();
            return kBinOrdered;
        }
        // 4. rank inside the bin (bins[b] is now the bin's start)
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = tid + q * kThreads;
            if (i < cc) {
                const uint32_t kc = tkey[i], kv = tval[i];
                const uint64_t kk = sort_key(kc, kv);
                const uint32_t b = g(kc);
                const uint32_t s0 = bins[b];
                const uint32_t e0 = b < thr ? bins[b + 1] : (uint32_t)cc;
                uint32_t r = 0;
                for (uint32_t j = s0; j < e0; ++j) r += sort_key(tkey[j], tval[j]) > kk ? 1u : 0u;
                S.outv[s0 + r] = kv;
            }
        }
        __syncthreads();
        return kBinOrdered;
    }
    // The two-per-SM build scatters each candidate of small bins as its 64-bit sort key into the
    // 2 kCap words from tkey on (tval follows tkey), so that the ranking reads one word pair per
    // comparison (prefill top-k 428 -> 409 us; the one-per-SM build keeps two arrays: its long
    // decode call measured 0.25 us slower with one)
    uint64_t* tk = reinterpret_cast<uint64_t*>(tkey);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int i = tid + q * kThreads;
        if (i < m) {
            const uint32_t x = lkey[i];
            const uint32_t b = g(x);
            if (b <= thr) {
                const uint32_t pos = atomicSub(&bins[b], 1u) - 1u;
                tk[pos] = sort_key(x, lval ? lval[i] : (uint32_t)i);
            }
        }
    }
    __syncthreads();
    // 4. rank inside the bin (bins[b] is now the bin's start); the index is the key's low word
    // complemented
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int i = tid + q * kThreads;
        if (i < cc) {
            const uint64_t kk = tk[i];
            const uint32_t b = g((uint32_t)(kk >> 32));
            const uint32_t s0 = bins[b];
            const uint32_t e0 = b < thr ? bins[b + 1] : (uint32_t)cc;
            uint32_t r = 0;
            for (uint32_t j = s0; j < e0; ++j) r += tk[j] > kk ? 1u : 0u;
            S.outv[s0 + r] = ~(uint32_t)kk;
        }
    }
    __syncthreads();
    return kBinOrdered;
}

// Rows longer than kCap (src: the line in the row cache or in global memory, c keys): a lower
// bound L for the candidates' codes from a sample of kSampleKeys evenly spaced keys -- the code of the rank-r largest sample,
// r = 1.15 l + 4 sqrt(l) + 2 with l = need * kSampleKeys / c the samples expected above the
// need-th key -- and the largest sample, the top of the bins.
__device__ __forceinline__ Binning sample_bound(const uint32_t* src, int c, int need)
{
    const Smem S = smem_view();
    const int tid = threadIdx.x;
    constexpr int per = kSampleKeys / kThreads;     // samples per thread
    uint32_t x[per];
    uint32_t smx = 0, smn = 0xFFFFFFFFu;
#pragma unroll
    for (int q = 0; q < per; ++q) {
        x[q] = src[((int64_t)(tid + q * kThreads) * c) / kSampleKeys];
        smx = max(smx, x[q]);
        smn = min(smn, x[q]);
    }
    block_max_min(&smx, &smn, S.misc);
    // the sample's rank-r largest code, to the resolution of kSampleBins bins over its range
    int s1 = 0;
    while (s1 < 32 && ((smx - smn) >> s1) >= (uint32_t)kSampleBins) ++s1;
    uint32_t* sb = S.bins;
    for (int b = tid; b < kSampleBins; b += kThreads) sb[b] = 0;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < per; ++q) atomicAdd(&sb[(smx - x[q]) >> s1], 1u);
    __syncthreads();
    const float lam = (float)need * (float)kSampleKeys / (float)c;   // single precision: FP64 is slow here
    int r = (int)(1.15f * lam + 4.0f * sqrtf(lam) + 2.0f);
    r = r < 1 ? 1 : (r > kSampleKeys ? kSampleKeys : r);
    constexpr int bpt = kSampleBins / kThreads;     // sample bins per thread
    static_assert(bpt % 2 == 0, "8-byte loads");
    uint32_t cnt[bpt], sum = 0;
#pragma unroll
    for (int v = 0; v < bpt / 2; ++v) {
        const uint2 cv = reinterpret_cast<const uint2*>(sb)[(bpt / 2) * tid + v];
        cnt[2 * v] = cv.x;
        cnt[2 * v + 1] = cv.y;
        sum += cv.x + cv.y;
    }
    uint32_t total;
    const uint32_t before = block_excl_scan(sum, &total, S.misc);
    uint32_t* s_b = S.misc + 110;
    if (before < (uint32_t)r && before + sum >= (uint32_t)r) {
        uint32_t run = before;
#pragma unroll
        for (int q = 0; q < bpt; ++q) {
            if (run < (uint32_t)r && run + cnt[q] >= (uint32_t)r) *s_b = bpt * tid + q;
            run += cnt[q];
        }
    }
    __syncthreads();
    const uint32_t b1 = *s_b;
    __syncthreads();
    // L: the lowest code of bin b1
    const uint64_t span = ((uint64_t)b1 + 1) << s1;
    const uint32_t L = span > (uint64_t)(smx - smn) ? smn : (uint32_t)(smx - span + 1);
    return make_binning(L, smx);
}

// Rows of at most kRankKeys keys: each key's place in the order is the number of keys of the row
// that sort before it (a higher code, or the same code and a lower index), counted against every
// key of the row cache; the first `need` places receive their indices in S.outv.  One pass and
// one barrier instead of the bins' passes, which cost more than this count on short rows.
constexpr int kRankKeys = 256;   // n^2 comparisons: measured faster than the bins up to ~256 keys
__device__ __forceinline__ void rank_order(const uint32_t* src, int n, int need)
{
    const Smem S = smem_view();
    for (int t = threadIdx.x; t < n; t += kThreads) {
        const uint32_t ct = src[t];
        uint32_t r = 0;
#pragma unroll 8
        for (int j = 0; j < t; ++j) r += src[j] >= ct ? 1u : 0u;       // lower index: ties sort first
#pragma unroll 8
        for (int j = t + 1; j < n; ++j) r += src[j] > ct ? 1u : 0u;
        if (r < (uint32_t)need) S.outv[r] = (uint32_t)t;
    }
    __syncthreads();
}

// Exact fallback: the k-th largest sort key of the row (radix select), then exactly k keys at or
// above it, ordered by the bitonic network; the ordered indices end in S.val.
__device__ QLI_TOPK_FN void exact_topk(const uint32_t* line, int64_t n, int k)
{
    const Smem S = smem_view();
    const uint64_t T = radix_select(S, n, k, [&](int64_t j) { return sort_key(line[j], (uint32_t)j); }, 56);
    const int c = min(gather(S, line, n, T), kCap);
    bitonic_any(S.key, S.val, c, reinterpret_cast<uint64_t*>(S.bins));
}

// Uncached rows (longer than kCacheKeys): the keys at or above the rank-r largest of kSamples
// evenly spaced keys of the line, r = 1.15 k S / n + 4 sqrt(k S / n) + 2, gathered from global
// memory into S.key / S.val; returns their count.  The samples go to the row cache, which such a
// row does not use: with S = 8192 the count expected at k = 2048 stays near 1.5 k up to 2^17 keys
// (about 4.4 standard deviations below kCap), where 2048 samples left it near kCap and the exact
// fallback often ran.
__device__ QLI_TOPK_FN int gather_sampled(const uint32_t* line, int64_t n, int k)
{
    const Smem S = smem_view();
    const int tid = threadIdx.x;
    for (int i = tid; i < kSamples; i += kThreads) {
        const int64_t j = ((int64_t)i * n) / kSamples;
        S.cache[i] = __ldg(line + j);
    }
    __syncthreads();
    const float lam = (float)k * (float)kSamples / (float)n;   // samples expected above the k-th
    int rank = (int)(1.15f * lam + 4.0f * sqrtf(lam) + 2.0f);
    rank = rank < 1 ? 1 : (rank > kSamples ? kSamples : rank);
    // the bound: the lowest code of the histogram bin (kSampleBins over the samples' range) that
    // holds the rank-th largest sample -- one counting pass instead of a radix select's four
    constexpr int kPer = kSamples / kThreads;
    static_assert(kPer * kThreads == kSamples, "whole samples per thread");
    uint32_t x[kPer], smx = 0, smn = 0xFFFFFFFFu;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        x[q] = S.cache[tid + q * kThreads];
        smx = max(smx, x[q]);
        smn = min(smn, x[q]);
    }
    block_max_min(&smx, &smn, S.misc);
    int s1 = 0;
    while (s1 < 32 && ((smx - smn) >> s1) >= (uint32_t)kSampleBins) ++s1;
    uint32_t* sb = S.bins;
    for (int b = tid; b < kSampleBins; b += kThreads) sb[b] = 0;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kPer; ++q) atomicAdd(&sb[(smx - x[q]) >> s1], 1u);
    __syncthreads();
    constexpr int bpt = kSampleBins / kThreads;     // sample bins per thread
    uint32_t cnt[bpt], sum = 0;
#pragma unroll
    for (int q = 0; q < bpt; ++q) {
        cnt[q] = sb[bpt * tid + q];
        sum += cnt[q];
    }
    uint32_t total;
    const uint32_t before = block_excl_scan(sum, &total, S.misc);
    uint32_t* s_b = S.misc + 110;
    if (before < (uint32_t)rank && before + sum >= (uint32_t)rank) {
        uint32_t run = before;
#pragma unroll
        for (int q = 0; q < bpt; ++q) {
            if (run < (uint32_t)rank && run + cnt[q] >= (uint32_t)rank) *s_b = bpt * tid + q;
            run += cnt[q];
        }
    }
    __syncthreads();
    const uint32_t b1 = *s_b;
    __syncthreads();
    const uint64_t span = ((uint64_t)b1 + 1) << s1;
    const uint32_t L = span > (uint64_t)(smx - smn) ? smn : (uint32_t)(smx - span + 1);
    return gather(S, line, n, (uint64_t)L << 32);
}

// Merging build: the row's tile words -> exclusive offsets (with the source bit) in S.toff[0,
// ntile) and the total in S.toff[ntile]; returns the candidate count, or -1 when the row is to be
// ordered from its score line instead (too many tiles or candidates, or fewer candidates than the
// row needs, which only a failed score launch leaves).  Block-wide.
__device__ QLI_TOPK_FN int split_offsets(const TopkArgs& a, int64_t row, int64_t n, int need)
{
    const Smem S = smem_view();
    const int tid = threadIdx.x;
    const int64_t ntile = (n + kTileKeys - 1) / kTileKeys;
    if (ntile > kSplitTiles) return -1;
    const uint32_t* info = a.split.info + row * (a.p.ld / kTileKeys);
    constexpr int kPer = (kSplitTiles + kThreads - 1) / kThreads;   // tiles per thread, contiguous
    uint32_t w[kPer], sum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int64_t t = (int64_t)tid * kPer + q;
        w[q] = t < ntile ? __ldcg(info + t) : 0u;
        sum += min(w[q] & ~kTileFromCandidates, (uint32_t)kTileKeys);
    }
    uint32_t total;
    uint32_t off = block_excl_scan(sum, &total, S.misc);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int64_t t = (int64_t)tid * kPer + q;
        if (t < ntile) S.toff[t] = off | (w[q] & kTileFromCandidates);
        off += min(w[q] & ~kTileFromCandidates, (uint32_t)kTileKeys);
    }
    if (tid == 0) S.toff[ntile] = total;
    __syncthreads();
    return (total > (uint32_t)kSplitKeys || total < (uint32_t)need) ? -1 : (int)total;
}

// Merging build: the candidates of the row's tiles, in tile order, into dst[0, total) (a warp per
// tile, four 32-key loads per lane)
__device__ QLI_TOPK_FN void split_gather(const TopkArgs& a, int64_t row, int64_t ntile, uint32_t* dst)
{
    const Smem S = smem_view();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = row * a.p.ld;
    for (int64_t t = warp; t < ntile; t += kWarps) {
        const uint32_t o0 = S.toff[t], o1 = S.toff[t + 1] & ~kTileFromCandidates;
        const uint32_t off = o0 & ~kTileFromCandidates, c = o1 - off;
        if (c == 0) continue;
        const uint32_t* src = ((o0 & kTileFromCandidates) ? a.split.code : a.scores) + base + t * kTileKeys;
        uint32_t v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = (uint32_t)(lane + 32 * m) < c ? __ldcg(src + lane + 32 * m) : 0u;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if ((uint32_t)(lane + 32 * m) < c) dst[off + lane + 32 * m] = v[m];
    }
    __syncthreads();
}

// Merging build: the key index of candidate position q (the last tile whose offset is <= q holds it)
__device__ __forceinline__ uint32_t split_key(const TopkArgs& a, int64_t row, int64_t ntile, uint32_t q)
{
    const Smem S = smem_view();
    int64_t lo = 0, hi = ntile - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if ((S.toff[mid] & ~kTileFromCandidates) <= q) lo = mid; else hi = mid - 1;
    }
    const uint32_t o = S.toff[lo], r = q - (o & ~kTileFromCandidates);
    return (o & kTileFromCandidates) ? __ldcg(a.split.idx + row * a.p.ld + lo * kTileKeys + r)
                                     : (uint32_t)(lo * kTileKeys + r);
}

// Bounded wait for the row cache's bulk copy (false: it did not land within about 2 s)
__device__ bool wait_copy(uint64_t* bar, uint32_t& parity)
{
    bool ok = true;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > 2000000000ull) {
            ok = false;
            break;
        }
    }
    parity ^= 1u;
    return __syncthreads_and(ok);
}

#ifndef QLI_TOPK_HELPERS_ONLY
// One CTA per row (the grid strides over rows).  kMerge: the rows' candidates come from the
// split-local selection.
template <bool kMerge>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) topk_kernel(const __grid_constant__ TopkArgs a)
{
    const Smem S = smem_view();
    if (threadIdx.x == 0) {
        ptx::mbar_init(S.bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    uint32_t bar_parity = 0;
    __shared__ int s_bad;

    const Params& p = a.p;
    const int tid = threadIdx.x;
    const int k = p.sparse_count;
    bool meta_ok = false;
    RowInfo ri{};
    int64_t pages = 0;
    int32_t pg_first = 0;
    bool bad = false;
    auto read_header = [&]() {
        meta_ok = __ldcg(a.meta + kMhMagic) == kMetaMagic && __ldcg(a.meta + kMhLayoutHash) == p.hash;
    };
    auto locate = [&](int64_t row) {
        ri = row_info(a, meta_ok, row);
        pages = ri.n > 0 ? ceil_div64(ri.lc, p.block_size) : 0;
    };
    // every page the batch's rows can see must lie in the pool: the first entry per thread is
    // loaded here and checked after the selection, the rest (rows of more than kThreads pages) at
    // once
    auto load_pages = [&]() {
        const int32_t* table = a.block_table + (ri.b < 0 ? 0 : ri.b) * p.max_blocks_per_seq;
        pg_first = tid < pages ? __ldcg(table + tid) : 0;
        bad = false;
        for (int64_t i = tid + kThreads; i < pages; i += kThreads) {
            const int32_t pg = __ldcg(table + i);
            bad |= pg < 0 || pg >= p.num_blocks;
        }
    };
    // The two-per-SM build's CTAs take many rows each (a prefill's: ~50).  There the place of each
    // row is worked out ahead -- thread t finds that of the CTA's (c kThreads + t)-th row when
    // chunk c of its rows begins, one round of dependent loads instead of one per row -- and handed
    // over through shared memory when the row comes up.  (Copying the next row's line earlier --
    // while the current row is written, during its ranking, or into a second line buffer during
    // its selection -- measured slower: a copy landing in shared memory slows the selection.)
    RowInfo mine{-1, 0, 0, 0};
    auto fill = [&](int64_t it0) {
        const int64_t r = blockIdx.x + (it0 + tid) * (int64_t)gridDim.x;
        if (r < p.rows) mine = row_info(a, meta_ok, r);
    };
    int32_t* hand = reinterpret_cast<int32_t*>(S.misc + 116);   // [0, 4) this row, [4, 8) the next
    auto publish = [&](int32_t* dst) {
        dst[0] = (int32_t)mine.b;
        dst[1] = (int32_t)mine.r;
        dst[2] = (int32_t)mine.n;
        dst[3] = (int32_t)mine.lc;
    };
    auto start_copy = [&](uint32_t* dst, const uint32_t* src, int64_t keys) {
        ptx::fence_proxy_async_smem();
        const uint32_t bytes = (uint32_t)(((keys * 4) + 15) & ~(int64_t)15);
        ptx::mbar_arrive_expect_tx(S.bar, bytes);
        ptx::bulk_load(dst, src, bytes, S.bar);
    };
    // row r's line into L2: its first `keys` codes (at most kCacheKeys)
    auto prefetch_line = [&](int64_t r, int64_t keys) {
        const int64_t nb = ((min(keys, (int64_t)kCacheKeys) * 4) + 15) & ~(int64_t)15;
        if (nb > 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.scores + r * p.ld), "r"((uint32_t)nb)
                         : "memory");
    };
    // after the score kernel the first row's place and pages are read before the wait; a
    // standalone launch reads them after it and loads the pages once the row's copy is issued
    const bool early = a.early && blockIdx.x < p.rows;
    if (early) {
        read_header();
        locate(blockIdx.x);
        load_pages();
        if constexpr (kPipe) fill(0);
    }
    // the score lines (and, for a standalone launch, the metadata) come from earlier kernels; the
    // next call may overwrite them only after this grid completes (it waits too)
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    if (!a.early) {
        read_header();
        if constexpr (kPipe) fill(0);
    }

    int64_t it = 0;
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
        int32_t* out = a.out + row * k;
        const bool loaded = early && it == 0;
        const bool ahead = kPipe && !kMerge && (it + 1) % kThreads != 0 && row + gridDim.x < p.rows;
        if constexpr (kPipe) {
            const int slot = (int)(it % kThreads);
            if (slot == 0 && it > 0) fill(it);
            if (tid == slot) publish(hand);
            if (ahead && tid == slot + 1) publish(hand + 4);
        } else if (!loaded) {
            locate(row);
        }
        __syncthreads();                           // the previous row is done with shared memory
        if (kPipe && !loaded) {
            ri = RowInfo{hand[0], hand[1], hand[2], hand[3]};
            pages = ri.n > 0 ? ceil_div64(ri.lc, p.block_size) : 0;
        }
        const int64_t nn = ahead ? hand[6] : 0;   // the next row's keys
        const int64_t n = ri.n;
        const uint32_t* line = a.scores + row * p.ld;
        const int need = (int)(n < k ? n : k);
        int M = -1;                                // merging build: the row's candidates
        if constexpr (kMerge) {
            if (n > 0) M = split_offsets(a, row, n, need);
        }
        const bool cached = n > 0 && n <= kCacheKeys && M < 0;
        if (tid == 0) {
            s_bad = 0;
            if (cached) start_copy(S.cache, line, n);
            // the CTA's next row comes from DRAM: ask for its line now, so that its copy finds it
            // in L2 (its keys where known, else the line's first kCacheKeys codes; asking two rows
            // ahead measured slower)
            if (!kMerge && row + gridDim.x < p.rows) prefetch_line(row + gridDim.x, ahead ? nn : p.ld);
        }
        __syncthreads();
        if (!loaded) load_pages();
        bool copy_ok = true;
        if (cached) {
            copy_ok = wait_copy(S.bar, bar_parity);   // bounded wait for the line
            if (!copy_ok && tid == 0) atomicOr(a.err, kErrTimeout);
        }
        const uint32_t* result = S.outv;           // ordered indices of this row
        const uint32_t* msrc = S.cache + kSplitBase;   // merging: the gathered candidates
        if (n > 0 && copy_ok) {
            int st = kBinTooMany;
            if (kMerge && M >= 0) {
                // the same orders over the candidates' positions (index order)
                split_gather(a, row, (n + kTileKeys - 1) / kTileKeys, S.cache + kSplitBase);
                if (M <= kRankKeys) {
                    rank_order(msrc, M, need);
                    st = kBinOrdered;
                } else if (M <= kCap) {
                    uint32_t hi = 0, lo = 0xFFFFFFFFu;
                    for (int i = tid; i < M; i += kThreads) {
                        hi = max(hi, msrc[i]);
                        lo = min(lo, msrc[i]);
                    }
                    block_max_min(&hi, &lo, S.misc);
                    const Binning g = make_binning(lo, hi);
                    count_bins(msrc, M, g);
                    st = order_bins(msrc, nullptr, M, need, g, S.key, S.val);
                } else if (kSplitBase > 0) {
                    const Binning g = sample_bound(msrc, M, need);
                    const int m = compact_and_count(msrc, M, g, true);
                    st = order_bins(S.key, S.val, m, need, g, S.cache, S.cache + kCap);
                }
                if (st == kBinTooMany) {
                    exact_topk(msrc, M, need);
                    result = S.val;
                }
            } else if (cached) {
                // bins over the whole range (short rows: every key is a candidate) or from a sample
                if (n <= kRankKeys) {
                    rank_order(S.cache, (int)n, need);
                    st = kBinOrdered;
                } else if (n <= kCap) {
                    // every key is a candidate: bins over the row's whole code range, counted and
                    // scattered straight from the row cache
                    uint32_t hi = 0, lo = 0xFFFFFFFFu;
                    for (int i = tid; i < (int)n; i += kThreads) {
                        const uint32_t x = S.cache[i];
                        hi = max(hi, x);
                        lo = min(lo, x);
                    }
                    block_max_min(&hi, &lo, S.misc);
                    const Binning g = make_binning(lo, hi);
                    count_bins(S.cache, (int)n, g);
                    st = order_bins(S.cache, nullptr, (int)n, need, g, S.key, S.val);
                } else {
                    const Binning g = sample_bound(S.cache, (int)n, need);
                    const int m = compact_and_count(S.cache, (int)n, g, true);
                    st = order_bins(S.key, S.val, m, need, g, S.cache, S.cache + kCap);
                }
                if (st == kBinTooMany) {
                    exact_topk(S.cache, n, k);
                    result = S.val;
                }
            } else {
                const int c = gather_sampled(line, n, k);
                if (c >= k && c <= kCap) {
                    uint32_t hi = 0, lo = 0xFFFFFFFFu;
                    for (int i = tid; i < c; i += kThreads) {
                        hi = max(hi, S.key[i]);
                        lo = min(lo, S.key[i]);
                    }
                    block_max_min(&hi, &lo, S.misc);
                    const Binning g = make_binning(lo, hi);
                    count_bins(S.key, c, g);
                    st = order_bins(S.key, S.val, c, need, g, S.cache, S.cache + kCap);
                }
                if (st == kBinTooMany) {
                    exact_topk(line, n, k);
                    result = S.val;
                }
            }
        }
        // ---- the page check, then the row
        bad |= tid < pages && (pg_first < 0 || pg_first >= p.num_blocks);
        if (bad) s_bad = 1;
        __syncthreads();
        const bool blank = n <= 0 || !copy_ok || s_bad;
        if (tid == 0 && s_bad) atomicOr(a.err, kErrPage);
        const bool merged = kMerge && M >= 0;
        const int64_t ntile = (n + kTileKeys - 1) / kTileKeys;
        for (int i = tid; i < k; i += kThreads) {
            int32_t v = -1;
            if (!blank && i < need) v = merged ? (int32_t)split_key(a, row, ntile, result[i]) : (int32_t)result[i];
            out[i] = v;
        }
        if (a.values) {
            // the written indices' scores, decoded from the row's score line (in L2) or, merging,
            // from the gathered candidates
            float* val = a.values + row * k;
            for (int i = tid; i < k; i += kThreads) {
                float v = -__int_as_float(0x7F800000);
                if (!blank && i < need) {
                    const uint32_t c = merged ? msrc[result[i]] : __ldg(line + result[i]);
                    v = __uint_as_float((c & 0x80000000u) ? (c & 0x7FFFFFFFu) : ~c);
                }
                val[i] = v;
            }
        }
    }
}

#endif  // QLI_TOPK_HELPERS_ONLY

}  // namespace

#ifndef QLI_TOPK_HELPERS_ONLY
cudaError_t QLI_TOPK_LAUNCHER(const Params& p, const int32_t* block_table, const int32_t* meta,
                        const uint32_t* scores, const SplitBufs& split, uint32_t* err_word, int32_t* out,
                        float* values, bool after_score, int max_ctas, cudaStream_t st)
{
    if (p.rows == 0) return cudaSuccess;
    TopkArgs a{p, block_table, meta, scores, err_word, out, values, split, after_score ? 1 : 0};
    auto kernel = p.split_topk ? topk_kernel<true> : topk_kernel<false>;
    const int smem = p.split_topk ? kSmemSplitBytes : kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // one CTA per row, or (max_ctas > 0) at most max_ctas CTAs that stride over the rows
    int grid = p.rows < (1 << 30) ? p.rows : (1 << 30);
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, st, a);
}
#endif  // QLI_TOPK_HELPERS_ONLY

}  // namespace qli

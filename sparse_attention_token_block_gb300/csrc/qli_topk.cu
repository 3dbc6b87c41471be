// qli_topk.cu -- per-row top-k over the score lines (README function section, step 3: select the
// top-k indices; parameter table: sparse_count, sparse_indices).
//
// One 1024-thread CTA per output row.  Scores are held as order-preserving uint32 codes; a key's
// full sort key is (code << 32) | (0xFFFFFFFF - index): score descending, then index ascending.
//
// 1. Candidates.  n <= kCap: every visible key.  n <= 32768: the row is held in registers and a
//    two-level 2048-bin histogram over its code range narrows the k-th largest code to a sub-bin;
//    every key in that sub-bin or above is a candidate.  Longer rows: a threshold code is the rank-r largest
//    of 2048 evenly spaced keys of the row (radix select over the samples), with
//    r = 1.15 k S / n + 4 sqrt(k S / n) + 2, which leaves between k and kCap keys at or above it
//    with overwhelming probability; one pass gathers them.  Outside [k, kCap], an exact radix
//    select on the 64-bit sort keys finds the k-th key and exactly k keys are gathered.
// 2. Order.  The candidates are distributed into 8192 buckets by code (bucket 0 = highest codes;
//    the code range is scaled to the bucket count), and each bucket is insertion-sorted by its
//    owner thread on the full sort key.  If any bucket holds more than kBigBucket keys (heavy ties),
//    a block-wide bitonic sort on the 64-bit sort keys is used instead.
// 3. The first min(k, n) indices are written, then -1 up to sparse_count.  Rows with no visible
//    key, rows of an invalid batch and rows whose batch's block_table names a page outside the pool
//    are all -1.
#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 4096;                    // candidates held in shared memory
constexpr int kSamples = 2048;
constexpr int kBuckets = 2048;
constexpr int kBigBucket = 256;
constexpr int kOrderBuckets = 8192;           // ordering buckets (counters kept in the row cache)
constexpr int kCacheKeys = 32768;             // score lines up to this length are cached in smem
constexpr int kSmemBytes = kCacheKeys * 4 + 4 * kCap * 4 + 2 * kBuckets * 4 + 256 * 4 + 64 * 4 + 16;

struct TopkArgs {
    Params p;
    const int32_t* block_table;
    const int32_t* meta;
    const uint32_t* scores;
    uint32_t* err;
    int32_t* out;
};

struct Smem {
    uint32_t* key;    // [kCap] candidate codes (gather order)
    uint32_t* val;    // [kCap] candidate indices
    uint32_t* okey;   // [kCap] ordered codes
    uint32_t* oval;   // [kCap] ordered indices
    uint32_t* cnt;    // [kBuckets]
    uint32_t* off;    // [kBuckets]
    uint32_t* hist;   // [256]
    uint32_t* misc;   // [64]
    uint32_t* cache;  // [kCacheKeys] one score line
    uint64_t* bar;    // bulk-copy barrier
};

__device__ __forceinline__ uint64_t sort_key(uint32_t code, uint32_t idx)
{
    return (static_cast<uint64_t>(code) << 32) | (0xFFFFFFFFu - idx);
}

// Block-wide exclusive scan of one value per thread; also returns the total.
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t* total, uint32_t* sh /* >= kWarps */)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kWarps ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kWarps) sh[lane] = w;
    }
    __syncthreads();
    const uint32_t before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
    *total = sh[kWarps - 1];
    __syncthreads();
    return before;
}

__device__ uint32_t block_max(uint32_t v, uint32_t* sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kWarps ? sh[lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = max(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (lane == 0) sh[32] = w;
    }
    __syncthreads();
    const uint32_t r = sh[32];
    __syncthreads();
    return r;
}

// Radix select over 64-bit sort keys produced by `get(i)` for i < n: the k-th largest key
// (one shared 256-bin histogram per 8-bit digit, counts aggregated per warp before the atomic).
template <class Get>
__device__ uint64_t radix_select(const Smem& S, int64_t n, int k, Get get, int top_shift)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* s_digit = S.misc + 40;
    uint32_t* s_rem = S.misc + 41;
    uint32_t* s_done = S.misc + 42;
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

// Gather (unordered) the keys j < n whose sort key is >= t64; returns how many (only the first
// kCap are stored).
__device__ int gather(const Smem& S, const uint32_t* line, int64_t n, uint64_t t64)
{
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t* s_cnt = S.misc + 48;
    if (tid == 0) *s_cnt = 0;
    __syncthreads();
    for (int64_t j0 = 0; j0 < n; j0 += kThreads) {
        const int64_t j = j0 + tid;
        uint32_t c = 0;
        bool take = false;
        if (j < n) {
            c = __ldg(line + j);
            take = sort_key(c, (uint32_t)j) >= t64;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(s_cnt, (uint32_t)__popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (take) {
                const uint32_t pos = base + __popc(bal & ((1u << lane) - 1u));
                if (pos < (uint32_t)kCap) {
                    S.key[pos] = c;
                    S.val[pos] = (uint32_t)j;
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

// Slow path: order key/val[0..c) with the bitonic network; the ordered indices end in val.
template <int E>
__device__ void bitonic_order(const Smem& S, int c)
{
    uint64_t v[E];
    const int tid = threadIdx.x;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        v[e] = i < c ? sort_key(S.key[i], S.val[i]) : 0ull;   // 0 sorts below every real key
    }
    __syncthreads();
    bitonic_desc<E>(v, reinterpret_cast<uint64_t*>(S.okey));   // okey/oval double as 64-bit scratch
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = tid * E + e;
        if (i < c) S.val[i] = 0xFFFFFFFFu - (uint32_t)(v[e] & 0xFFFFFFFFu);
    }
    __syncthreads();
}

// Order the c candidates (key/val) descending by sort key; the ordered indices end in val.
// lo = lower bound of codes.  The buckets' counters live in the row cache, idle by now.
__device__ void order_candidates(const Smem& S, int c, uint32_t lo)
{
    const int tid = threadIdx.x;
    uint32_t* cnt = S.cache;                       // [kOrderBuckets]
    uint32_t* off = S.cache + kOrderBuckets;       // [kOrderBuckets]
    constexpr int per = kOrderBuckets / kThreads;
    uint32_t hi_local = 0;
    for (int i = tid; i < c; i += kThreads) hi_local = max(hi_local, S.key[i]);
    const uint32_t hi = block_max(hi_local, S.misc);
    const uint32_t range = hi - lo;
    int shift = 0;
    while (shift < 32 && (range >> shift) >= (uint32_t)kOrderBuckets) ++shift;
    for (int b = tid; b < kOrderBuckets; b += kThreads) cnt[b] = 0;
    __syncthreads();
    for (int i = tid; i < c; i += kThreads) atomicAdd(&cnt[(hi - S.key[i]) >> shift], 1u);
    __syncthreads();
    // exclusive scan of the bucket counts, `per` consecutive buckets per thread
    uint32_t mine[per], sum = 0;
    bool big = false;
#pragma unroll
    for (int q = 0; q < per; ++q) {
        mine[q] = cnt[tid * per + q];
        sum += mine[q];
        big |= mine[q] > (uint32_t)kBigBucket;
    }
    uint32_t total;
    uint32_t base = block_excl_scan(sum, &total, S.misc);
#pragma unroll
    for (int q = 0; q < per; ++q) {
        off[tid * per + q] = base;
        base += mine[q];
    }
    if (__syncthreads_or(big)) {
        if (c <= kThreads) bitonic_order<1>(S, c);
        else if (c <= 2 * kThreads) bitonic_order<2>(S, c);
        else bitonic_order<4>(S, c);
        return;
    }
    // scatter (filling each bucket from its end), then place every candidate at its bucket's start
    // plus its rank among the bucket's keys (one thread per candidate)
    for (int i = tid; i < c; i += kThreads) {
        const uint32_t b = (hi - S.key[i]) >> shift;
        const uint32_t pos = off[b] + atomicSub(&cnt[b], 1u) - 1u;
        S.okey[pos] = S.key[i];
        S.oval[pos] = S.val[i];
    }
    __syncthreads();
    for (int i = tid; i < c; i += kThreads) {
        const uint32_t kc = S.okey[i], kv = S.oval[i];
        const uint64_t kk = sort_key(kc, kv);
        const uint32_t b = (hi - kc) >> shift;
        const uint32_t s0 = off[b];
        const uint32_t e0 = (b + 1 < (uint32_t)kOrderBuckets) ? off[b + 1] : (uint32_t)c;
        uint32_t r = 0;
        for (uint32_t j = s0; j < e0; ++j) r += sort_key(S.okey[j], S.oval[j]) > kk ? 1u : 0u;
        S.val[s0 + r] = kv;
    }
    __syncthreads();
}

// Find, from per-bin counts in S.cnt (bin 0 = highest codes), the bin where the running count
// reaches `need`; returns it and stores the count of the bins before it in *above.
__device__ uint32_t locate_bin(const Smem& S, uint32_t need, uint32_t* above)
{
    const int tid = threadIdx.x;
    const uint32_t c0 = S.cnt[2 * tid], c1 = S.cnt[2 * tid + 1];
    uint32_t total;
    const uint32_t before = block_excl_scan(c0 + c1, &total, S.misc);
    uint32_t* s_bin = S.misc + 56;
    uint32_t* s_above = S.misc + 57;
    if (before < need && before + c0 >= need) {
        *s_bin = 2 * tid;
        *s_above = before;
    } else if (before + c0 < need && before + c0 + c1 >= need) {
        *s_bin = 2 * tid + 1;
        *s_above = before + c0;
    }
    __syncthreads();
    const uint32_t b = *s_bin;
    *above = *s_above;
    __syncthreads();
    return b;
}

// Rows of up to kCacheKeys keys, whose score line the caller bulk-copied into shared memory (one
// memory latency).  A 2048-bin histogram over the line's code range finds the bin holding the k-th
// largest code; a second 2048-bin histogram over that bin alone narrows it to a sub-bin.  Every
// key above that sub-bin's lower edge becomes a candidate (written to key/val).  Returns the
// candidate count, or -1 if it would exceed kCap; *lo receives a lower bound of their codes.
__device__ int select_cached(const Smem& S, int64_t n, int k, uint32_t* lo)
{
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t* cache = S.cache;
    uint32_t mn = 0xFFFFFFFFu, mx = 0;
    for (int64_t j = tid; j < n; j += kThreads) {
        const uint32_t c = cache[j];
        mn = min(mn, c);
        mx = max(mx, c);
    }
    mx = block_max(mx, S.misc);
    mn = ~block_max(~mn, S.misc);
    const uint32_t need = (uint32_t)((int64_t)k < n ? (int64_t)k : n);
    // level 1: the whole range
    int s1 = 0;
    while (s1 < 32 && ((mx - mn) >> s1) >= (uint32_t)kBuckets) ++s1;
    for (int b = tid; b < kBuckets; b += kThreads) S.cnt[b] = 0;
    __syncthreads();
    for (int64_t j = tid; j < n; j += kThreads) atomicAdd(&S.cnt[(mx - cache[j]) >> s1], 1u);
    __syncthreads();
    uint32_t above1;
    const uint32_t b1 = locate_bin(S, need, &above1);
    // level 2: inside bin b1 (offsets below mx in [b1 << s1, (b1 + 1) << s1))
    const int s2 = s1 > 11 ? s1 - 11 : 0;
    for (int b = tid; b < kBuckets; b += kThreads) S.cnt[b] = 0;
    __syncthreads();
    for (int64_t j = tid; j < n; j += kThreads) {
        const uint32_t d = mx - cache[j];
        if ((d >> s1) == b1) atomicAdd(&S.cnt[(d - (b1 << s1)) >> s2], 1u);
    }
    __syncthreads();
    uint32_t above2;
    const uint32_t b2 = locate_bin(S, need - above1, &above2);
    (void)lane;
    const uint64_t lim = (static_cast<uint64_t>(b1) << s1) + ((static_cast<uint64_t>(b2) + 1) << s2);
    // every key with (mx - code) below the end of sub-bin b2 is a candidate: count per thread,
    // scan, then write (thread t owns the keys t, t + kThreads, ...)
    uint32_t mine = 0;
    for (int64_t j = tid; j < n; j += kThreads) mine += (uint64_t)(mx - cache[j]) < lim ? 1u : 0u;
    uint32_t total;
    uint32_t pos = block_excl_scan(mine, &total, S.misc);
    for (int64_t j = tid; j < n; j += kThreads) {
        const uint32_t cj = cache[j];
        if ((uint64_t)(mx - cj) < lim) {
            if (pos < (uint32_t)kCap) {
                S.key[pos] = cj;
                S.val[pos] = (uint32_t)j;
            }
            ++pos;
        }
    }
    uint32_t* s_cnt = S.misc + 48;
    if (tid == 0) *s_cnt = total;
    __syncthreads();
    const int count = (int)*s_cnt;
    *lo = lim > (uint64_t)(mx - mn) ? mn : (uint32_t)(mx - lim + 1);
    __syncthreads();
    return count > kCap ? -1 : count;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const __grid_constant__ TopkArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    Smem S;
    S.key = reinterpret_cast<uint32_t*>(smem);
    S.val = S.key + kCap;
    S.okey = S.val + kCap;
    S.oval = S.okey + kCap;
    S.cnt = S.oval + kCap;
    S.off = S.cnt + kBuckets;
    S.hist = S.off + kBuckets;
    S.misc = S.hist + 256;
    S.cache = S.misc + 64;                                    // 16-byte aligned (offsets are)
    S.bar = reinterpret_cast<uint64_t*>(S.cache + kCacheKeys);
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
    // the score lines and metadata come from earlier kernels; the next call may overwrite them
    // only after this grid completes (it waits too)
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    const bool meta_ok = a.meta[kMhMagic] == kMetaMagic && a.meta[kMhLayoutHash] == p.hash;
    const int32_t* be = a.meta + p.meta.batch_off;

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        int32_t* out = a.out + row * k;
        // ---- which batch / live row / how many visible keys
        int64_t b = -1, r = 0, n = 0;
        if (meta_ok && p.batch > 0) {
            if (!p.layout_tnd) {
                b = row / p.s1;
                r = row % p.s1;
            } else {
                int64_t lo = 0, hi = p.batch - 1;
                while (lo < hi) {
                    const int64_t mid = (lo + hi + 1) >> 1;
                    if (be[mid * kBatchWords + kBeFirstRow] <= row) lo = mid; else hi = mid - 1;
                }
                b = lo;
                r = row - be[b * kBatchWords + kBeFirstRow];
            }
            const int32_t* e = be + b * kBatchWords;
            if (e[kBeOk] && r >= 0)
                n = visible_keys(p.sparse_mode, p.cmp_ratio, e[kBeSq], e[kBeSk], e[kBeLc], r);
        }
        const uint32_t* line = a.scores + row * p.ld;
        // rows cached in shared memory: start the line's bulk copy now, under the page check
        const bool cached_path = n > kCap && n <= kCacheKeys;
        // ---- every page this batch's rows can see must lie in the pool
        __syncthreads();
        if (tid == 0) {
            s_bad = 0;
            if (cached_path) {
                // the previous row's generic reads of the cache came before (barrier above)
                ptx::fence_proxy_async_smem();
                const uint32_t bytes = (uint32_t)(((n * 4) + 15) & ~(int64_t)15);
                ptx::mbar_arrive_expect_tx(S.bar, bytes);
                ptx::bulk_load(S.cache, line, bytes, S.bar);
            }
        }
        __syncthreads();
        if (n > 0) {
            const int64_t pages = ceil_div64(be[b * kBatchWords + kBeLc], p.block_size);
            const int32_t* table = a.block_table + b * p.max_blocks_per_seq;
            bool bad = false;
            for (int64_t i = tid; i < pages; i += kThreads) {
                const int32_t pg = __ldg(table + i);
                bad |= pg < 0 || pg >= p.num_blocks;
            }
            if (bad) s_bad = 1;
        }
        __syncthreads();
        bool copy_ok = true;
        if (cached_path) {
            // bounded wait for the line (also when the row turns out invalid: the copy must land
            // before the cache is reused)
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(S.bar, bar_parity)) {
                if (ptx::globaltimer() - t0 > 2000000000ull) {
                    copy_ok = false;
                    break;
                }
            }
            bar_parity ^= 1u;
            copy_ok = __syncthreads_and(copy_ok);
            if (!copy_ok && tid == 0) atomicOr(a.err, kErrTimeout);
        }
        if (s_bad || !copy_ok) {
            n = 0;
            if (tid == 0 && s_bad) atomicOr(a.err, kErrPage);
        }
        if (n <= 0) {
            for (int i = tid; i < k; i += kThreads) out[i] = -1;
            continue;
        }
        const int64_t m = n < k ? n : k;
        int count;
        uint32_t lo = 0;
        if (n <= kCap) {
            uint32_t mn = 0xFFFFFFFFu;
            for (int64_t j = tid; j < n; j += kThreads) {
                const uint32_t c = __ldg(line + j);
                S.key[j] = c;
                S.val[j] = (uint32_t)j;
                mn = min(mn, c);
            }
            lo = ~block_max(~mn, S.misc);
            count = (int)n;
        } else if (n <= kCacheKeys) {
            count = select_cached(S, n, k, &lo);
            if (count < 0) {
                const uint64_t T = radix_select(
                    S, n, k, [&](int64_t j) { return sort_key(__ldg(line + j), (uint32_t)j); }, 56);
                count = min(gather(S, line, n, T), kCap);
                lo = (uint32_t)(T >> 32);
            }
        } else {
            // ---- threshold: the rank-r largest of evenly spaced samples
            for (int i = tid; i < kSamples; i += kThreads) {
                const int64_t j = ((int64_t)i * n) / kSamples;
                S.key[i] = __ldg(line + j);
            }
            __syncthreads();
            const double lam = (double)k * kSamples / (double)n;   // samples expected above the k-th
            int rank = (int)(1.15 * lam + 4.0 * sqrt(lam) + 2.0);
            rank = rank < 1 ? 1 : (rank > kSamples ? kSamples : rank);
            const uint32_t* samp = S.key;
            const uint64_t t = radix_select(
                S, kSamples, rank, [&](int64_t i) { return static_cast<uint64_t>(samp[i]) << 32; }, 56);
            lo = (uint32_t)(t >> 32);
            count = gather(S, line, n, static_cast<uint64_t>(lo) << 32);
            if (count < k || count > kCap) {
                // ---- exact fallback: the k-th sort key of the row, then exactly k keys >= it
                const uint64_t T = radix_select(
                    S, n, k, [&](int64_t j) { return sort_key(__ldg(line + j), (uint32_t)j); }, 56);
                count = min(gather(S, line, n, T), kCap);
                lo = (uint32_t)(T >> 32);
            }
        }
        order_candidates(S, count, lo);
        for (int i = tid; i < k; i += kThreads) out[i] = i < m ? (int32_t)S.val[i] : -1;
    }
}

}  // namespace

cudaError_t launch_topk(const Params& p, const int32_t* block_table, const int32_t* meta,
                        const uint32_t* scores, uint32_t* err_word, int32_t* out, cudaStream_t st)
{
    if (p.rows == 0) return cudaSuccess;
    TopkArgs a{p, block_table, meta, scores, err_word, out};
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p.rows < (1 << 30) ? p.rows : (1 << 30);
    return launch_pdl(topk_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, a);
}

}  // namespace qli

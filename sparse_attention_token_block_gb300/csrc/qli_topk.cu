// qli_topk.cu -- per-row top-k over the score lines (README function section, step 3: "select the
// top-k indices"; parameter table: sparse_count, sparse_indices).
//
// One CTA per output row.  Each visible key j of the row carries the 64-bit code
//     (ordered(score_j) << 32) | (0xFFFFFFFF - j),
// which is unique and orders keys by score descending, then index ascending.  The CTA finds the
// k-th largest code with an 8-bit-digit radix select (per-warp histograms, warp-aggregated
// counts), gathers the k codes at or above it, sorts them descending with a bitonic network in
// shared memory and writes their indices, then -1 up to sparse_count.  Rows with no visible key,
// rows of an invalid batch, and rows whose batch's block_table names a page outside the pool are
// written as all -1.
#include "qli_internal.cuh"

namespace qli {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheKeys = 16384;                 // score lines up to this length live in smem
constexpr int kSmemBytes = kCacheKeys * 4 + kWarps * 256 * 4 + kMaxSparse * 8 + 256 * 4;

struct TopkArgs {
    Params p;
    const int32_t* block_table;
    const int32_t* meta;
    const uint32_t* scores;
    uint32_t* err;
    int32_t* out;
};

__device__ __forceinline__ uint64_t code_of(const uint32_t* line, int64_t j)
{
    return (static_cast<uint64_t>(line[j]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* cache = reinterpret_cast<uint32_t*>(smem);
    uint32_t* whist = cache + kCacheKeys;                                  // [kWarps][256]
    uint64_t* sel = reinterpret_cast<uint64_t*>(whist + kWarps * 256);     // [kMaxSparse]
    uint32_t* hist = reinterpret_cast<uint32_t*>(sel + kMaxSparse);        // [256]
    __shared__ int s_bad;
    __shared__ uint32_t s_digit, s_rem, s_done, s_cnt;

    const Params& p = a.p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = p.sparse_count;
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
                    int64_t mid = (lo + hi + 1) >> 1;
                    if (be[mid * kBatchWords + kBeFirstRow] <= row) lo = mid; else hi = mid - 1;
                }
                b = lo;
                r = row - be[b * kBatchWords + kBeFirstRow];
            }
            const int32_t* e = be + b * kBatchWords;
            if (e[kBeOk] && r >= 0)
                n = visible_keys(p.sparse_mode, p.cmp_ratio, e[kBeSq], e[kBeSk], e[kBeLc], r);
        }
        // ---- every page this batch's rows can see must lie in the pool
        __syncthreads();
        if (tid == 0) s_bad = 0;
        __syncthreads();
        if (n > 0) {
            const int64_t pages = ceil_div64(be[b * kBatchWords + kBeLc], p.block_size);
            const int32_t* table = a.block_table + b * p.max_blocks_per_seq;
            bool bad = false;
            for (int64_t i = tid; i < pages; i += kThreads) {
                const int32_t pg = table[i];
                bad |= pg < 0 || pg >= p.num_blocks;
            }
            if (bad) s_bad = 1;
        }
        __syncthreads();
        if (s_bad) {
            n = 0;
            if (tid == 0) atomicOr(a.err, kErrPage);
        }
        if (n <= 0) {
            for (int i = tid; i < k; i += kThreads) out[i] = -1;
            continue;
        }
        const uint32_t* gline = a.scores + row * p.ld;
        const bool cached = n <= kCacheKeys;
        if (cached)
            for (int64_t j = tid; j < n; j += kThreads) cache[j] = gline[j];
        __syncthreads();
        const uint32_t* line = cached ? cache : gline;
        const int64_t m = n < k ? n : k;

        if (n <= k) {
            for (int64_t j = tid; j < n; j += kThreads) sel[j] = code_of(line, j);
        } else {
            // ---- radix select of the k-th largest code, 8 bits per pass from the top
            uint64_t prefix = 0, mask = 0;
            uint32_t rem = (uint32_t)k;
            for (int shift = 56; shift >= 0; shift -= 8) {
                for (int i = tid; i < kWarps * 256; i += kThreads) whist[i] = 0;
                __syncthreads();
                uint32_t* myh = whist + warp * 256;
                for (int64_t j0 = 0; j0 < n; j0 += kThreads) {
                    const int64_t j = j0 + tid;
                    bool in = false;
                    uint32_t digit = 0;
                    if (j < n) {
                        const uint64_t c = code_of(line, j);
                        in = (c & mask) == prefix;
                        digit = (uint32_t)(c >> shift) & 0xFFu;
                    }
                    const unsigned act = __ballot_sync(0xffffffffu, in);
                    if (in) {
                        const unsigned peers = __match_any_sync(act, digit);
                        if (lane == __ffs(peers) - 1) myh[digit] += __popc(peers);
                    }
                }
                __syncthreads();
                if (tid < 256) {
                    uint32_t s = 0;
                    for (int w = 0; w < kWarps; ++w) s += whist[w * 256 + tid];
                    hist[tid] = s;
                }
                __syncthreads();
                if (warp == 0) {
                    // lane l owns digits 255-8l .. 248-8l (descending order)
                    uint32_t c8[8], sum = 0;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        c8[q] = hist[255 - 8 * lane - q];
                        sum += c8[q];
                    }
                    uint32_t incl = sum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    const uint32_t excl = incl - sum;
                    const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
                    if (lane == __ffs(hit) - 1) {
                        uint32_t above = excl;
                        for (int q = 0; q < 8; ++q) {
                            if (above + c8[q] >= rem) {
                                s_digit = 255 - 8 * lane - q;
                                s_rem = rem - above;
                                s_done = (c8[q] == rem - above) ? 1u : 0u;
                                break;
                            }
                            above += c8[q];
                        }
                    }
                }
                __syncthreads();
                prefix |= (uint64_t)s_digit << shift;
                mask |= (uint64_t)0xFFu << shift;
                rem = s_rem;
                const bool done = s_done != 0;
                __syncthreads();
                if (done) break;
            }
            // ---- gather the k codes >= threshold (warp-aggregated slot allocation)
            if (tid == 0) s_cnt = 0;
            __syncthreads();
            for (int64_t j0 = 0; j0 < n; j0 += kThreads) {
                const int64_t j = j0 + tid;
                uint64_t c = 0;
                bool take = false;
                if (j < n) {
                    c = code_of(line, j);
                    take = c >= prefix;
                }
                const unsigned bal = __ballot_sync(0xffffffffu, take);
                if (bal) {
                    uint32_t base = 0;
                    if (lane == 0) base = atomicAdd(&s_cnt, (uint32_t)__popc(bal));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (take) {
                        const uint32_t pos = base + __popc(bal & ((1u << lane) - 1u));
                        if (pos < (uint32_t)kMaxSparse) sel[pos] = c;
                    }
                }
            }
        }
        // ---- bitonic sort of sel[0..P) descending, padded with zero codes (below every key)
        int P = 1;
        while (P < m) P <<= 1;
        __syncthreads();
        for (int64_t i = m + tid; i < P; i += kThreads) sel[i] = 0;
        __syncthreads();
        for (int kk = 2; kk <= P; kk <<= 1) {
            for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                for (int i = tid; i < P; i += kThreads) {
                    const int l = i ^ jj;
                    if (l > i) {
                        const uint64_t x = sel[i], y = sel[l];
                        const bool desc = (i & kk) == 0;
                        if (desc ? (x < y) : (x > y)) {
                            sel[i] = y;
                            sel[l] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        for (int i = tid; i < k; i += kThreads)
            out[i] = i < m ? (int32_t)(0xFFFFFFFFu - (uint32_t)(sel[i] & 0xFFFFFFFFu)) : -1;
        __syncthreads();
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
    topk_kernel<<<grid, kThreads, kSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qli

// qli_topk_cluster.cu -- the per-row top-k for problems whose rows can be longer than one CTA's row
// cache (32768 keys) but at most four times that (decodes of 32k to 128k compressed keys): a
// cluster of four 1024-thread CTAs per row, each holding a quarter of the row in its shared memory.
//
//   1. CTA r bulk-copies keys [r q, (r + 1) q) of the row, q = ceil(n / 4) rounded up to a tile.
//   2. The bound, as for an uncached row: of the 8192 evenly spaced keys of the row, each CTA takes
//      those in its quarter; the four CTAs' largest and smallest samples and their 2048-bin
//      histograms are read across the cluster (distributed shared memory), so every CTA finds the
//      same bound L: the lowest code of the bin holding the rank-r largest sample (rows of at most
//      kCap keys take every key).
//   3. Each CTA appends its keys with code >= L, with their row indices, to CTA 0's candidate
//      arrays through remote atomics and stores.
//   4. CTA 0 orders the candidates with the bins of qli_topk.cuh (exact fallback over the line in
//      global memory when they are too few or too many) and writes the row.
// The row's score line is read once, by four SMs at a time; the one-CTA form reads it through one
// SM (for a 2^17-key row its gather alone took ~35k cycles).
#define QLI_TOPK_THREADS 1024
#define QLI_TOPK_CACHE_KEYS 32768
#define QLI_TOPK_BINS 8192
#define QLI_TOPK_LAUNCHER launch_topk_cluster_unused
#define QLI_TOPK_HELPERS_ONLY 1
#include "qli_topk.cuh"

namespace qli {

namespace {

constexpr int kParts = 4;     // CTAs per row (a portable cluster size)

__global__ void __cluster_dims__(kParts, 1, 1) __launch_bounds__(kThreads, 1)
    topk_cluster_kernel(const __grid_constant__ TopkArgs a)
{
    const Smem S = smem_view();
    const uint32_t part = ptx::cluster_rank();
    const int64_t row = blockIdx.x / kParts;
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
        ptx::mbar_init(S.bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    __shared__ int s_bad;
    const Params& p = a.p;
    const int k = p.sparse_count;
    // the score lines and the metadata come from earlier kernels; the next call may overwrite them
    // only after this grid completes (it waits too)
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    const bool meta_ok = __ldcg(a.meta + kMhMagic) == kMetaMagic && __ldcg(a.meta + kMhLayoutHash) == p.hash;
    const RowInfo ri = row_info(a, meta_ok, row);
    const int64_t n = ri.n;               // the same in every CTA of the cluster
    const int need = (int)(n < k ? n : k);
    const uint32_t* line = a.scores + row * p.ld;
    const int64_t q = (((n + kParts - 1) / kParts) + kTileKeys - 1) / kTileKeys * kTileKeys;
    const bool fits = q <= kCacheKeys;    // (the host sends only rows of at most 4 kCacheKeys keys)
    const int64_t b0 = fits ? min(n, (int64_t)part * q) : 0, b1 = fits ? min(n, b0 + q) : 0;
    const int len = (int)(b1 - b0);
    uint32_t* misc = S.misc;               // [112] max sample, [113] min sample, [114] copy landed

    // 1. this CTA's quarter of the row
    bool copy_ok = true;
    if (len > 0) {
        if (tid == 0) {
            ptx::fence_proxy_async_smem();
            const uint32_t bytes = (uint32_t)((((int64_t)len * 4) + 15) & ~(int64_t)15);
            ptx::mbar_arrive_expect_tx(S.bar, bytes);
            ptx::bulk_load(S.cache, line + b0, bytes, S.bar);
        }
        uint32_t parity = 0;
        copy_ok = wait_copy(S.bar, parity);
    }

    // 2. the bound from the samples that fall in each quarter: sample i of the row is key
    // (i n) / kSamples; this CTA holds those with b0 <= (i n) / kSamples < b1
    const int64_t i_lo = n > 0 ? (b0 * kSamples + n - 1) / n : 0;
    const int64_t i_hi = n > 0 ? (b1 * kSamples + n - 1) / n : 0;
    uint32_t smx = 0, smn = 0xFFFFFFFFu;
    for (int64_t i = i_lo + tid; i < i_hi; i += kThreads) {
        const uint32_t x = S.cache[(i * n) / kSamples - b0];
        smx = max(smx, x);
        smn = min(smn, x);
    }
    block_max_min(&smx, &smn, S.misc);
    if (tid == 0) {
        misc[112] = smx;
        misc[113] = smn;
        misc[114] = copy_ok ? 1u : 0u;
        misc[104] = 0;                     // CTA 0: the candidate count
    }
    uint32_t* sb = S.bins;                 // this CTA's sample histogram (kSampleBins)
    for (int b = tid; b < kSampleBins; b += kThreads) sb[b] = 0;
    ptx::cluster_sync();                   // (1) every CTA's extremes, flag and cleared bins
    bool all_ok = true;
    for (uint32_t r = 0; r < (uint32_t)kParts; ++r) {
        smx = max(smx, ptx::ld_cluster(ptx::cluster_addr(misc + 112, r)));
        smn = min(smn, ptx::ld_cluster(ptx::cluster_addr(misc + 113, r)));
        all_ok &= ptx::ld_cluster(ptx::cluster_addr(misc + 114, r)) != 0;
    }
    int s1 = 0;
    while (s1 < 32 && ((smx - smn) >> s1) >= (uint32_t)kSampleBins) ++s1;
    for (int64_t i = i_lo + tid; i < i_hi; i += kThreads)
        atomicAdd(&sb[(smx - S.cache[(i * n) / kSamples - b0]) >> s1], 1u);
    ptx::cluster_sync();                   // (2) every CTA's histogram
    const float lam = n > 0 ? (float)k * (float)kSamples / (float)n : 0.0f;
    int rank = (int)(1.15f * lam + 4.0f * sqrtf(lam) + 2.0f);
    rank = rank < 1 ? 1 : (rank > kSamples ? kSamples : rank);
    constexpr int bpt = kSampleBins / kThreads;
    uint32_t cnt[bpt], sum = 0;
#pragma unroll
    for (int j = 0; j < bpt; ++j) {
        cnt[j] = 0;
        for (uint32_t r = 0; r < (uint32_t)kParts; ++r) cnt[j] += ptx::ld_cluster(ptx::cluster_addr(sb + bpt * tid + j, r));
        sum += cnt[j];
    }
    uint32_t total;
    const uint32_t before = block_excl_scan(sum, &total, S.misc);
    if (tid == 0) misc[110] = kSampleBins - 1;   // (rank beyond the samples: the lowest bin)
    __syncthreads();
    if (before < (uint32_t)rank && before + sum >= (uint32_t)rank) {
        uint32_t run = before;
#pragma unroll
        for (int j = 0; j < bpt; ++j) {
            if (run < (uint32_t)rank && run + cnt[j] >= (uint32_t)rank) misc[110] = bpt * tid + j;
            run += cnt[j];
        }
    }
    __syncthreads();
    const uint64_t span = ((uint64_t)misc[110] + 1) << s1;
    uint32_t L = span > (uint64_t)(smx - smn) ? smn : (uint32_t)(smx - span + 1);
    if (n <= kCap) L = 0;                   // short rows: every key is a candidate
    ptx::cluster_sync();                   // (3) the histograms are read; CTA 0's count is zero

    // 3. this quarter's keys at or above L into CTA 0's candidate arrays, with their row indices
    const uint32_t cnt_addr = ptx::cluster_addr(misc + 104, 0);
    const uint32_t key_addr = ptx::cluster_addr(S.key, 0);
    const uint32_t val_addr = ptx::cluster_addr(S.val, 0);
    for (int i0 = 0; i0 < len; i0 += kThreads * kGatherU) {
        uint32_t c[kGatherU];
#pragma unroll
        for (int u = 0; u < kGatherU; ++u) {
            const int i = i0 + u * kThreads + tid;
            c[u] = i < len ? S.cache[i] : 0u;
        }
#pragma unroll
        for (int u = 0; u < kGatherU; ++u) {
            const int i = i0 + u * kThreads + tid;
            const bool take = i < len && c[u] >= L;
            const unsigned bal = __ballot_sync(0xffffffffu, take);
            if (bal) {
                uint32_t base = 0;
                if (lane == 0) base = ptx::atom_add_cluster(cnt_addr, (uint32_t)__popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (take) {
                    const uint32_t pos = base + __popc(bal & ((1u << lane) - 1u));
                    if (pos < (uint32_t)kCap) {
                        ptx::st_cluster(key_addr + 4 * pos, c[u]);
                        ptx::st_cluster(val_addr + 4 * pos, (uint32_t)(b0 + i));
                    }
                }
            }
        }
    }
    ptx::cluster_sync();                   // (4) every candidate is in CTA 0; no more remote access
    if (part != 0) return;

    // 4. CTA 0: the page check, the order, the row
    const int64_t pages = n > 0 ? ceil_div64(ri.lc, p.block_size) : 0;
    const int32_t* table = a.block_table + (ri.b < 0 ? 0 : ri.b) * p.max_blocks_per_seq;
    bool bad = false;
    for (int64_t i = tid; i < pages; i += kThreads) {
        const int32_t pg = __ldcg(table + i);
        bad |= pg < 0 || pg >= p.num_blocks;
    }
    if (tid == 0) s_bad = 0;
    __syncthreads();
    if (bad) s_bad = 1;
    const uint32_t* result = S.outv;
    const int m = (int)misc[104];
    if (n > 0 && fits && all_ok) {
        int st = kBinTooMany;
        if (m >= need && m <= kCap) {
            uint32_t hi = 0, lo = 0xFFFFFFFFu;
            for (int i = tid; i < m; i += kThreads) {
                hi = max(hi, S.key[i]);
                lo = min(lo, S.key[i]);
            }
            block_max_min(&hi, &lo, S.misc);
            const Binning g = make_binning(lo, hi);
            count_bins(S.key, m, g);
            st = order_bins(S.key, S.val, m, need, g, S.cache, S.cache + kCap);
        }
        if (st == kBinTooMany) {
            exact_topk(line, n, k);
            result = S.val;
        }
    }
    __syncthreads();
    const bool blank = n <= 0 || !fits || !all_ok || s_bad;
    if (tid == 0 && s_bad) atomicOr(a.err, kErrPage);
    if (tid == 0 && n > 0 && (!fits || !all_ok)) atomicOr(a.err, fits ? kErrTimeout : kErrLength);
    int32_t* out = a.out + row * k;
    for (int i = tid; i < k; i += kThreads) out[i] = (!blank && i < need) ? (int32_t)result[i] : -1;
    if (a.values) {
        float* val = a.values + row * k;
        for (int i = tid; i < k; i += kThreads) {
            float v = -__int_as_float(0x7F800000);
            if (!blank && i < need) {
                const uint32_t c = __ldg(line + result[i]);
                v = __uint_as_float((c & 0x80000000u) ? (c & 0x7FFFFFFFu) : ~c);
            }
            val[i] = v;
        }
    }
}

}  // namespace

cudaError_t launch_topk_cluster(const Params& p, const int32_t* block_table, const int32_t* meta,
                                const uint32_t* scores, uint32_t* err_word, int32_t* out, float* values,
                                cudaStream_t st)
{
    if (p.rows == 0) return cudaSuccess;
    TopkArgs a{p, block_table, meta, scores, err_word, out, values, SplitBufs{nullptr, nullptr, nullptr}, 0};
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_cluster_kernel, dim3((unsigned)p.rows * kParts), dim3(kThreads), kSmemBytes, st, a);
}

}  // namespace qli

// qli_metadata.cu -- the work-split scheduler (README: the metadata input of the indexer and its
// companion metadata call, "number of cores used, block size, and each core's start point").
//
// One CTA reads the device lengths and writes, into the caller's int32 buffer:
//   * the header (magic, CTA count G, unit count, total tiles, error bits, problem hash);
//   * per batch: live query rows Sq_b, key tokens Sk_b, compressed keys Lc_b, first output row,
//     validity, query-group count and first group index;
//   * per query group (kGroupTokens consecutive live rows of one batch): the prefix sum of its key
//     tile counts, where a group needs ceil(n_last / 128) tiles and n_last is the visible-key count
//     of its last row (the largest in the group under either mask);
//   * the split: the concatenated tile sequence of all groups is cut into G equal ranges, one per
//     CTA of the score kernel; each range becomes the list of (batch, first row, key_begin,
//     key_end, first output row, Sq_b, Sk_b, Lc_b) units it overlaps, stored CTA by CTA with
//     offsets (one thread per unit).
#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kMetaThreads = 1024;

// Block-wide exclusive scan of one value per thread; returns the exclusive prefix and the total.
// One barrier: every warp scans the warp totals itself.  Calls alternate between the two halves
// of `sh` ([64]) so that a call never overwrites totals another warp may still be reading.
__device__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total, uint32_t* sh, int& parity)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (int)(blockDim.x >> 5);
    uint32_t* buf = sh + 32 * parity;
    parity ^= 1;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) buf[warp] = x;
    __syncthreads();
    const uint32_t wt = lane < nwarps ? buf[lane] : 0u;
    uint32_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
    }
    *total = __shfl_sync(0xffffffffu, wi, 31);
    return __shfl_sync(0xffffffffu, wi - wt, warp) + x - v;
}

// A strided int32 array in shared or global memory
struct View {
    int32_t* p;
    int stride;
    __device__ int32_t& operator[](int64_t i) const { return p[i * stride]; }
};

// Largest i in [0, n) with a[i] <= key, for non-decreasing a (a[0] <= key assumed)
__device__ int64_t upper_index(const View& a, int64_t n, int64_t key)
{
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (a[mid] <= key) lo = mid; else hi = mid - 1;
    }
    return lo;
}

constexpr int kSmemBatch = 2048;     // batches whose fields are staged in shared memory
constexpr int kSmemGroups = 16384;   // groups whose tile prefix is staged in shared memory
constexpr int kMetaSmemBytes = (6 * kSmemBatch + 2 * (kSmemGroups + 1)) * 4;

__global__ void __launch_bounds__(kMetaThreads, 1)
    metadata_kernel(Params p, const int32_t* __restrict__ seq_lens_q,
                    const int32_t* __restrict__ seq_lens_k, int32_t* __restrict__ meta, int G)
{
    extern __shared__ int32_t msm[];
    __shared__ uint32_t scan_sh[64];
    int scan_parity = 0;
    __shared__ uint32_t s_err;
    __shared__ int s_tnd_bad;
    const int tid = threadIdx.x;
    int32_t* be = meta + p.meta.batch_off;
    int32_t* cta_off = meta + p.meta.cta_off;
    int32_t* units = meta + p.meta.unit_off;
    // per-batch fields and the group prefix live in shared memory when they fit, else they are
    // read back from their home in the metadata buffer
    const bool sb = p.batch <= kSmemBatch;
    const bool sg = p.meta.max_groups <= kSmemGroups;
    const View v_sq = sb ? View{msm, 1} : View{be + kBeSq, kBatchWords};
    const View v_sk = sb ? View{msm + kSmemBatch, 1} : View{be + kBeSk, kBatchWords};
    const View v_lc = sb ? View{msm + 2 * kSmemBatch, 1} : View{be + kBeLc, kBatchWords};
    const View v_gb = sb ? View{msm + 3 * kSmemBatch, 1} : View{be + kBeGroupBase, kBatchWords};
    const View v_ok = sb ? View{msm + 4 * kSmemBatch, 1} : View{be + kBeOk, kBatchWords};
    const View v_fr = sb ? View{msm + 5 * kSmemBatch, 1} : View{be + kBeFirstRow, kBatchWords};
    const View v_gp = sg ? View{msm + 6 * kSmemBatch, 1} : View{meta + p.meta.group_off, 1};
    const View v_uf = sg ? View{msm + 6 * kSmemBatch + kSmemGroups + 1, 1} : View{meta + p.meta.ufirst_off, 1};
    int32_t* gpre_home = meta + p.meta.group_off;
    if (tid == 0) { s_err = 0; s_tnd_bad = 0; }
    // the lengths may come from the previous kernel, and the previous indexer call may still read
    // this metadata buffer
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    __syncthreads();

    // ---- per-batch extents and validity
    for (int b = tid; b < p.batch; b += blockDim.x) {
        int64_t sq = 0, first = 0;
        bool ok = true;
        if (!p.layout_tnd) {
            first = (int64_t)b * p.s1;
            const int64_t v = seq_lens_q ? seq_lens_q[b] : p.s1;
            ok = v >= 0 && v <= p.s1;
            sq = ok ? v : 0;
        } else {
            const int64_t lo = b > 0 ? seq_lens_q[b - 1] : 0, hi = seq_lens_q[b];
            ok = lo >= 0 && hi >= lo && hi <= p.total_q;
            if (!ok) atomicOr(&s_tnd_bad, 1);
            first = lo < 0 ? 0 : lo;
            sq = ok ? hi - lo : 0;
        }
        const int64_t sk = seq_lens_k[b];
        ok = ok && sk >= 0 && sk <= p.max_seqlen_k;
        const int64_t lc = ok ? compressed_keys(sk, p.cmp_ratio) : 0;
        ok = ok && lc <= (int64_t)p.max_blocks_per_seq * p.block_size;
        if (!ok) atomicOr(&s_err, kErrLength);
        int32_t* e = be + (int64_t)b * kBatchWords;
        e[kBeSq] = (int32_t)sq;
        e[kBeSk] = (int32_t)(ok ? sk : 0);
        e[kBeLc] = (int32_t)lc;
        e[kBeFirstRow] = (int32_t)first;
        e[kBeOk] = ok ? 1 : 0;
        if (sb) {
            v_sq[b] = (int32_t)sq;
            v_sk[b] = (int32_t)(ok ? sk : 0);
            v_lc[b] = (int32_t)lc;
            v_ok[b] = ok ? 1 : 0;
            v_fr[b] = (int32_t)first;
        }
    }
    __syncthreads();

    // ---- query groups per batch (bad TND prefix sums invalidate every batch) and their prefix
    uint32_t running = 0;
    for (int base = 0; base < p.batch; base += blockDim.x) {
        const int b = base + tid;
        uint32_t groups = 0;
        if (b < p.batch) {
            int32_t* e = be + (int64_t)b * kBatchWords;
            if (s_tnd_bad) e[kBeOk] = 0;
            groups = (!s_tnd_bad && v_ok[b]) ? (uint32_t)((v_sq[b] + kGroupTokens - 1) / kGroupTokens) : 0u;
            e[kBeGroups] = (int32_t)groups;
        }
        uint32_t tot;
        const uint32_t ex = block_exclusive_scan(groups, &tot, scan_sh, scan_parity);
        if (b < p.batch) {
            be[(int64_t)b * kBatchWords + kBeGroupBase] = (int32_t)(running + ex);
            if (sb) v_gb[b] = (int32_t)(running + ex);
        }
        running += tot;
    }
    const int64_t total_groups = running;
    __syncthreads();

    // each thread owns a contiguous run of groups, so each pass below needs one block scan; the
    // batch of a run's first group comes from one binary search, later ones by advancing
    // the block is 256 or 1024 threads: divisions by its size are shifts
    const int lg_threads = __ffs((int)blockDim.x) - 1;
    const int64_t per = (total_groups + blockDim.x - 1) >> lg_threads;
    const int64_t g_lo = min((int64_t)tid * per, total_groups);
    const int64_t g_hi = min(g_lo + per, total_groups);
    // visible keys of group g of batch b (its last row's count, the largest in the group)
    auto keys_of = [&](int64_t b, int64_t g) -> int64_t {
        const int64_t r0 = (g - v_gb[b]) * kGroupTokens;
        const int64_t rl = min((int64_t)(r0 + kGroupTokens), (int64_t)v_sq[b]) - 1;
        return visible_keys(p.sparse_mode, p.cmp_ratio, v_sq[b], v_sk[b], v_lc[b], rl, p.complete_blocks);
    };
    // first batch whose groups include g, moving forward from b (batches without groups share
    // their successor's first group)
    auto advance_batch = [&](int64_t b, int64_t g) -> int64_t {
        while (b + 1 < p.batch && v_gb[b + 1] <= g) ++b;
        return b;
    };

    // ---- tiles per group, then their exclusive prefix (gpre[g]; gpre[total_groups] = total)
    {
        uint32_t mine = 0;
        int64_t b = g_lo < g_hi ? upper_index(v_gb, p.batch, g_lo) : 0;
        for (int64_t g = g_lo; g < g_hi; ++g) {
            b = advance_batch(b, g);
            const uint32_t tiles = (uint32_t)((keys_of(b, g) + kTileKeys - 1) / kTileKeys);
            v_gp[g] = (int32_t)tiles;                 // the count now, its prefix below
            mine += tiles;
        }
        uint32_t tot;
        uint32_t pre = block_exclusive_scan(mine, &tot, scan_sh, scan_parity);
        for (int64_t g = g_lo; g < g_hi; ++g) {
            const uint32_t tiles = (uint32_t)v_gp[g];
            v_gp[g] = (int32_t)pre;
            if (sg) gpre_home[g] = (int32_t)pre;
            pre += tiles;
        }
        running = tot;
    }
    const int64_t T = running;
    if (tid == 0) {
        v_gp[total_groups] = (int32_t)T;
        if (sg) gpre_home[total_groups] = (int32_t)T;
    }
    __syncthreads();

    // ---- split the tile sequence over G CTAs.  CTA c owns tiles [T c / G, T (c + 1) / G); a unit is
    // a (CTA, group) pair whose tile ranges meet.  Both partitions are ordered, so listing units
    // CTA by CTA lists them group by group too: a unit's index is the prefix over groups of their
    // unit counts plus its CTA's offset inside the group.  Work runs in parallel over groups.
    const int64_t Gl = G;
    const bool narrow = T * (Gl + 1) < (int64_t(1) << 32);  // (t + 1) G + T - 1 fits 32 bits
    auto cta_of = [&](int64_t t) -> int64_t {     // largest c with floor(T c / G) <= t
        int64_t c = narrow ? (int64_t)(((uint32_t)(t + 1) * (uint32_t)G + (uint32_t)(T - 1)) / (uint32_t)T) - 1
                           : ((t + 1) * Gl + T - 1) / T - 1;
        return c < 0 ? 0 : (c >= Gl ? Gl - 1 : c);
    };
    // floor(T c / G) without a division per CTA: c * floor(T / G) + floor(c * (T mod G) / G), the
    // last by a multiply with m = ceil(2^32 / G): for x = c (T mod G) < G^2 <= 2^20 the error of
    // x m / 2^32 against x / G is below 2^-12 < 1 / G, so the floor is exact
    // T < 2^31 (the host bounds rows x tiles) and 1 <= G <= 1024, so 32-bit divisions suffice, and
    // ceil(2^32 / G) = floor((2^32 - 1) / G) + 1 (0 for G = 1, where t_mod is 0)
    const uint32_t G32 = (uint32_t)(G > 0 ? G : 1);
    const uint32_t t_div = (uint32_t)T / G32, t_mod = (uint32_t)T % G32;
    const uint32_t inv_g = 0xFFFFFFFFu / G32 + 1u;
    static_assert(kMaxCtas <= 1024, "the reciprocal division needs G <= 1024");
    auto cta_start = [&](int64_t c) -> int64_t {
        return (int64_t)c * t_div + __umulhi((uint32_t)c * t_mod, inv_g);
    };
    if (T == 0)
        for (int c = tid; c <= G; c += blockDim.x) cta_off[c] = 0;
    // With T >= G every CTA owns at least one tile and a group's units are the CTAs from the one
    // holding its first tile to the one holding its last.  With T < G some CTAs own nothing, the
    // others exactly one tile each, and a group has one unit per tile.
    const bool dense = T >= Gl;
    auto group_units = [&](int64_t A, int64_t Bt) -> uint32_t {
        if (Bt <= A) return 0u;
        return dense ? (uint32_t)(cta_of(Bt - 1) - cta_of(A) + 1) : (uint32_t)(Bt - A);
    };
    // units per group and the index of each group's first unit
    {
        uint32_t mine = 0;
        for (int64_t g = g_lo; g < g_hi && T > 0; ++g) mine += group_units(v_gp[g], v_gp[g + 1]);
        uint32_t tot;
        uint32_t u = block_exclusive_scan(mine, &tot, scan_sh, scan_parity);
        for (int64_t g = g_lo; g < g_hi; ++g) {
            v_uf[g] = (int32_t)u;
            if (T > 0) u += group_units(v_gp[g], v_gp[g + 1]);
        }
        if (tid == 0) v_uf[total_groups] = (int32_t)tot;
        running = tot;
    }
    __syncthreads();
    // the records: thread t writes units [t U / n_t, (t + 1) U / n_t) in order; the group of its
    // first unit (the largest with first unit <= u; groups without units share their successor's
    // index) and that group's batch come from binary searches, later ones by advancing
    {
        const int64_t U = running;
        const int64_t u_lo = (U * tid) >> lg_threads, u_hi = (U * (tid + 1)) >> lg_threads;
        int64_t g = -1, b = 0, A = 0, Bt = 0, n = 0, r0 = 0, c = 0;
        int64_t t1 = 0;
        for (int64_t u = u_lo; u < u_hi; ++u) {
            int64_t k;
            if (g < 0 || u >= v_uf[g + 1]) {
                // a new group: this thread's first, or the next one with units
                if (g < 0) {
                    g = upper_index(v_uf, total_groups, u);
                    b = upper_index(v_gb, p.batch, g);
                } else {
                    do { ++g; } while (v_uf[g + 1] <= u);
                }
                b = advance_batch(b, g);
                A = v_gp[g];
                Bt = v_gp[g + 1];
                r0 = (g - v_gb[b]) * kGroupTokens;
                n = keys_of(b, g);
                k = u - v_uf[g];
                c = dense ? cta_of(A) + k : cta_of(A + k);
                t1 = cta_start(c);
            } else {
                k = u - v_uf[g];
                c = dense ? c + 1 : cta_of(A + k);
            }
            const int64_t t0 = dense ? t1 : cta_start(c);
            t1 = cta_start(c + 1);
            int4 w, v;
            w.x = (int32_t)b;
            w.y = (int32_t)r0;
            w.z = (int32_t)((max(t0, A) - A) * kTileKeys);
            w.w = (int32_t)min((min(t1, Bt) - A) * kTileKeys, n);
            v.x = v_fr[b] + (int32_t)r0;
            v.y = v_sq[b];
            v.z = v_sk[b];
            v.w = v_lc[b];
            int4* dst = reinterpret_cast<int4*>(units + u * kUnitWords);
            dst[0] = w;
            dst[1] = v;
            if (t0 >= A && t0 < Bt) {
                // the CTA's first unit; CTAs before it with an empty range (T < G) start here too
                cta_off[c] = (int32_t)u;
                for (int64_t ce = c - 1; ce >= 0 && cta_start(ce) == t0; --ce) cta_off[ce] = (int32_t)u;
            }
        }
    }
    __syncthreads();
    if (tid == 0) cta_off[G] = (int32_t)running;
    __syncthreads();
    if (tid == 0) {
        meta[kMhMagic] = kMetaMagic;
        meta[kMhCtas] = G;
        meta[kMhUnits] = (int32_t)running;
        meta[kMhTiles] = (int32_t)T;
        meta[kMhErr] = (int32_t)s_err;
        meta[kMhBatch] = p.batch;
        meta[kMhRows] = p.rows;
        meta[kMhGroups] = (int32_t)total_groups;
        meta[kMhLayoutHash] = p.hash;
    }
}

}  // namespace

cudaError_t launch_metadata(const Params& p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                            int32_t* meta, int num_ctas, cudaStream_t st)
{
    int G = num_ctas < kMaxCtas ? num_ctas : kMaxCtas;
    cudaError_t e = cudaFuncSetAttribute(metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMetaSmemBytes);
    if (e != cudaSuccess) return e;
    // few groups: fewer warps make each block-wide step cheaper; many groups: more lanes per pass
    const int threads = p.meta.max_groups <= 4096 && p.batch <= 4096 ? 256 : kMetaThreads;   // powers of two
    return launch_pdl(metadata_kernel, dim3(1), dim3(threads), kMetaSmemBytes, st, p, seq_lens_q,
                      seq_lens_k, meta, G);
}

}  // namespace qli

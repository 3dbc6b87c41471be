// qli_metadata.cu -- the work-split scheduler (README: the metadata input of the indexer and its
// companion metadata call, "number of cores used, block size, and each core's start point").
//
// One CTA reads the device lengths and writes, into the caller's int32 buffer:
//   * the header (magic, score CTA count G, live groups, total tiles T, error bits, problem hash);
//   * per batch: live query rows Sq_b, key tokens Sk_b, compressed keys Lc_b, first output row,
//     validity, query-group count and first group index (what the top-k reads per row);
//   * one record per live query group -- group_tokens consecutive live rows of one batch whose last
//     row sees at least one key -- with the batch's fields, its tile count ceil(n_last / 128), n_last
//     being the visible-key count of its last row (the largest in the group under either mask), and
//     the position of its first tile in the sequence the split cuts: every live group, in order,
//     as kUnitCost virtual tiles (its query load) followed by its key tiles, T positions in all;
//   * per score CTA c ("each core's start point"): the range [first, end) of live groups whose key
//     tiles its range [split_start(c), split_start(c + 1)) of the sequence overlaps.  A score CTA
//     derives its units -- (group, tile range) pairs -- from these records alone.
//
// The work is a handful of block-wide passes: per-batch extents (one read of the lengths), a scan
// of the groups per batch, one pass over the groups with a scan of the (live, tiles) pairs that
// also writes the records, and one binary search per CTA over the live groups' first tiles.
#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kMetaThreads = 512;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kSmemBatch = 2048;     // batches whose fields are staged in shared memory
constexpr int kSmemLive = 32768;     // live groups whose first tiles are staged in shared memory
constexpr int kMetaSmemMax = (6 * kSmemBatch + kSmemLive) * 4;

// Block-wide exclusive scan of one 64-bit value per thread (one barrier: every warp scans the
// warp totals itself); returns the exclusive prefix and the total.  Calls alternate between the
// two halves of `sh` ([2 * kMetaWarps]) so that a call never overwrites totals another warp may
// still be reading.
__device__ uint64_t block_scan64(uint64_t v, uint64_t* total, uint64_t* sh, int& parity)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t* buf = sh + kMetaWarps * parity;
    parity ^= 1;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) buf[warp] = x;
    __syncthreads();
    const uint64_t wt = lane < kMetaWarps ? buf[lane] : 0ull;
    uint64_t wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, wi, o);
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

// Largest i in [0, n) with a[i] <= key, for non-decreasing a with a[0] <= key
__device__ int64_t last_at_most(const View& a, int64_t n, int64_t key)
{
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (a[mid] <= key) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Smallest i in [0, n] with a[i] >= key (n if none), for non-decreasing a
__device__ int64_t first_at_least(const View& a, int64_t n, int64_t key)
{
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (a[mid] >= key) hi = mid; else lo = mid + 1;
    }
    return lo;
}

// Problems of at most kSmallMeta batches and query groups: the per-batch extents, the group scan
// and the live-group records worked out by one warp with shuffles (lane i holds batch i, then group
// i) instead of the block-wide passes below, which cost more in barriers and first-time code than
// the work itself.  Writes the batch entries and records as those passes do, the live groups' first
// key-tile positions to v_tb (shared memory), and (live groups, T, groups) to out[0..2].  Inlined:
// out of line, its first call fetched its code from DRAM after an L2 flush (~1 us of a decode call).
constexpr int kSmallMeta = 32;

__device__ __forceinline__ void small_phases(const Params& p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                                          int32_t* be, int32_t* rec, int32_t* v_tb, int64_t* out, uint32_t* err)
{
    const uint32_t full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int B = p.batch, gt = p.group_tokens;
    BatchExtent x{0, 0, 0, 0, false, false};
    if (lane < B) x = batch_extent(p, seq_lens_q, seq_lens_k, lane);
    if (__any_sync(full, lane < B && !x.ok) && lane == 0) atomicOr(err, kErrLength);
    const bool tnd_bad = __any_sync(full, lane < B && x.tnd_bad);   // bad prefix sums invalidate every batch
    const bool okb = lane < B && x.ok && !tnd_bad;
    const int groups = okb ? (x.sq + gt - 1) / gt : 0;
    int g_in = groups;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(full, g_in, o);
        if (lane >= o) g_in += y;
    }
    const int gb = g_in - groups;                    // batch lane's first group
    const int total = __shfl_sync(full, g_in, 31);
    if (lane < B) {
        int4* e = reinterpret_cast<int4*>(be + (int64_t)lane * kBatchWords);
        e[0] = make_int4(x.sq, x.sk, x.lc, x.first);
        e[1] = make_int4(okb ? 1 : 0, groups, gb, 0);
    }
    // group `lane`: its batch (the last batch whose first group is at or before it, as the block
    // passes find it), first row and key tiles
    int b = 0;
    for (int j = 1; j < B; ++j)
        if (__shfl_sync(full, gb, j) <= lane) b = j;
    const int sq = __shfl_sync(full, x.sq, b), sk = __shfl_sync(full, x.sk, b);
    const int lc = __shfl_sync(full, x.lc, b), fr = __shfl_sync(full, x.first, b);
    const int r0 = (lane - __shfl_sync(full, gb, b)) * gt;
    const int t = lane < total ? (int)group_tiles(p, sq, sk, lc, r0) : 0;
    const bool live = t > 0;
    const uint32_t lmask = __ballot_sync(full, live);
    const int li = __popc(lmask & ((1u << lane) - 1));
    int p_in = live ? t + kUnitCost : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(full, p_in, o);
        if (lane >= o) p_in += y;
    }
    const int pos = p_in - t;                        // the group's first key tile in the sequence
    if (live) {
        int4* r = reinterpret_cast<int4*>(rec + (int64_t)li * kGroupWords);
        r[0] = make_int4(b, r0, fr + r0, sq);
        r[1] = make_int4(sk, lc, pos, t);
        v_tb[li] = pos;
    }
    const int T = __shfl_sync(full, p_in, 31);
    if (lane == 0) {
        out[0] = __popc(lmask);
        out[1] = T;
        out[2] = total;
    }
}

__global__ void __launch_bounds__(kMetaThreads, 1)
    metadata_kernel(Params p, const int32_t* __restrict__ seq_lens_q,
                    const int32_t* __restrict__ seq_lens_k, int32_t* __restrict__ meta, int G, int G1)
{
    extern __shared__ int32_t msm[];
    __shared__ uint64_t scan_sh[2 * kMetaWarps];
    __shared__ uint32_t s_err;
    __shared__ int s_tnd_bad;
    int parity = 0;
    const int tid = threadIdx.x;
    const int gt = p.group_tokens;
    int32_t* be = meta + p.meta.batch_off;
    int32_t* cta = meta + p.meta.cta_off;
    int32_t* rec = meta + p.meta.group_off;
    // per-batch fields and the live groups' first tiles live in shared memory when they fit,
    // else they are read back from their home in the metadata buffer
    const bool sb = p.batch <= kSmemBatch;
    // (the shared memory holds nb = min(batch, kSmemBatch) entries per field, then the first tiles
    // of up to min(max_groups, kSmemLive) live groups: the launch requests only that much)
    const int nb = p.batch < kSmemBatch ? p.batch : kSmemBatch;
    const View v_sq = sb ? View{msm, 1} : View{be + kBeSq, kBatchWords};
    const View v_sk = sb ? View{msm + nb, 1} : View{be + kBeSk, kBatchWords};
    const View v_lc = sb ? View{msm + 2 * nb, 1} : View{be + kBeLc, kBatchWords};
    const View v_gb = sb ? View{msm + 3 * nb, 1} : View{be + kBeGroupBase, kBatchWords};
    const View v_ok = sb ? View{msm + 4 * nb, 1} : View{be + kBeOk, kBatchWords};
    const View v_fr = sb ? View{msm + 5 * nb, 1} : View{be + kBeFirstRow, kBatchWords};
    if (tid == 0) { s_err = 0; s_tnd_bad = 0; }
    // the lengths may come from the previous kernel, and the previous indexer call may still read
    // this metadata buffer
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    __syncthreads();

    __shared__ int64_t s_small[3];       // the one-warp passes' live groups, T and groups
    int64_t total_groups = 0, live = 0, T = 0;
    bool sl = true;
    View v_tb{msm + 6 * nb, 1};
    if (p.batch <= kSmallMeta && p.meta.max_groups <= kSmallMeta) {
        if (tid < 32) small_phases(p, seq_lens_q, seq_lens_k, be, rec, msm + 6 * nb, s_small, &s_err);
        __syncthreads();
        live = s_small[0];
        T = s_small[1];
        total_groups = s_small[2];
    } else {
        // ---- per-batch extents and validity
        for (int b = tid; b < p.batch; b += kMetaThreads) {
            const BatchExtent x = batch_extent(p, seq_lens_q, seq_lens_k, b);
            if (x.tnd_bad) s_tnd_bad = 1;
            if (!x.ok) atomicOr(&s_err, kErrLength);
            int4* e = reinterpret_cast<int4*>(be + (int64_t)b * kBatchWords);
            e[0] = make_int4(x.sq, x.sk, x.lc, x.first);
            if (sb) {
                v_sq[b] = x.sq;
                v_sk[b] = x.sk;
                v_lc[b] = x.lc;
                v_ok[b] = x.ok ? 1 : 0;
                v_fr[b] = x.first;
            } else {
                e[1].x = x.ok ? 1 : 0;     // kBeOk, read back below
            }
        }
        __syncthreads();
        const bool tnd_bad = s_tnd_bad != 0;   // bad prefix sums invalidate every batch

        // ---- query groups per batch and their prefix (the batch's first group)
        int64_t running = 0;
        for (int base = 0; base < p.batch; base += kMetaThreads) {
            const int b = base + tid;
            uint32_t groups = 0;
            const bool okb = b < p.batch && !tnd_bad && v_ok[b];
            if (b < p.batch) groups = okb ? (uint32_t)((v_sq[b] + gt - 1) / gt) : 0u;
            uint64_t tot;
            const uint64_t ex = block_scan64(groups, &tot, scan_sh, parity);
            if (b < p.batch) {
                int4* e = reinterpret_cast<int4*>(be + (int64_t)b * kBatchWords);
                e[1] = make_int4(okb ? 1 : 0, (int32_t)groups, (int32_t)(running + ex), 0);
                if (sb) {
                    v_gb[b] = (int32_t)(running + ex);
                    v_ok[b] = okb ? 1 : 0;
                }
            }
            running += (int64_t)tot;
        }
        total_groups = running;
        __syncthreads();

        // ---- groups: each thread owns a contiguous run; a group's batch comes from one binary search
        // for the run's first group, then by advancing.  One scan of (live, tiles) gives every live
        // group its record index and first tile.
        const int64_t per = (total_groups + kMetaThreads - 1) / kMetaThreads;
        const int64_t g_lo = min((int64_t)tid * per, total_groups);
        const int64_t g_hi = min(g_lo + per, total_groups);
        auto tiles_of = [&](int64_t b, int64_t g, int64_t* r0) -> int64_t {
            *r0 = (g - v_gb[b]) * gt;
            return group_tiles(p, v_sq[b], v_sk[b], v_lc[b], *r0);
        };
        auto advance = [&](int64_t b, int64_t g) -> int64_t {   // batches without groups share their successor's base
            while (b + 1 < p.batch && v_gb[b + 1] <= g) ++b;
            return b;
        };
        const int64_t b_lo = g_lo < g_hi ? last_at_most(v_gb, p.batch, g_lo) : 0;
        uint64_t mine = 0;     // live groups << 32 | tiles (T < 2^31: the host bounds rows x tiles)
        {
            int64_t b = b_lo, r0;
            for (int64_t g = g_lo; g < g_hi; ++g) {
                b = advance(b, g);
                const int64_t t = tiles_of(b, g, &r0);
                if (t > 0) mine += (uint64_t(1) << 32) + (uint64_t)(t + kUnitCost);
            }
        }
        uint64_t tot;
        const uint64_t pre = block_scan64(mine, &tot, scan_sh, parity);
        live = (int64_t)(tot >> 32);
        T = (int64_t)(tot & 0xFFFFFFFFull);
        sl = live <= kSmemLive;
        v_tb = sl ? View{msm + 6 * nb, 1} : View{rec + kGrTile, kGroupWords};
        {
            int64_t li = (int64_t)(pre >> 32), tile = (int64_t)(pre & 0xFFFFFFFFull);
            int64_t b = b_lo, r0;
            for (int64_t g = g_lo; g < g_hi; ++g) {
                b = advance(b, g);
                const int64_t t = tiles_of(b, g, &r0);
                if (t == 0) continue;
                int4* r = reinterpret_cast<int4*>(rec + li * kGroupWords);
                r[0] = make_int4((int32_t)b, (int32_t)r0, v_fr[b] + (int32_t)r0, v_sq[b]);
                r[1] = make_int4(v_sk[b], v_lc[b], (int32_t)(tile + kUnitCost), (int32_t)t);
                if (sl) v_tb[li] = (int32_t)(tile + kUnitCost);
                ++li;
                tile += t + kUnitCost;
            }
        }
        if (!sl) __threadfence_block();
        __syncthreads();

    }

    // ---- the split: CTA c owns positions [split_start(c), split_start(c + 1)) of the sequence; its
    // live groups run from the one whose block (virtual tiles, then key tiles) holds its first
    // position to (excluding) the first whose key tiles start at or after its end -- each of them
    // has key tiles inside the range, and first = end when the range holds only virtual tiles
    // split_start(T, G, G1, c) = T W(c) / W(G) in 32-bit divisions: with T = q W(G) + r it is
    // q W(c) + (r W(c)) / W(G), exactly (W(G) < 2^14, so r W(c) < 2^28; T < 2^31)
    const uint32_t WG = (uint32_t)split_weight(G1, G);
    const uint32_t tq = (uint32_t)T / WG, tr = (uint32_t)T % WG;
    auto start_of = [&](int64_t c) -> int64_t {
        const uint32_t w = (uint32_t)split_weight(G1, c);
        return (int64_t)tq * w + (tr * w) / WG;
    };
    for (int c = tid; c < G; c += kMetaThreads) {
        const int64_t t0 = start_of(c), t1 = start_of(c + 1);
        int32_t first = 0, end = 0;
        if (t1 > t0) {
            first = (int32_t)last_at_most(v_tb, live, t0 + kUnitCost);
            end = (int32_t)max((int64_t)first, first_at_least(v_tb, live, t1));
        }
        reinterpret_cast<int2*>(cta)[c] = make_int2(first, end);
    }
    if (tid == 0) {
        int4* h = reinterpret_cast<int4*>(meta);
        h[0] = make_int4(kMetaMagic, G, (int32_t)live, (int32_t)T);
        h[1] = make_int4((int32_t)s_err, p.batch, p.rows, (int32_t)total_groups);
        h[2] = make_int4(p.hash, G1, kUnitCost, 0);
    }
}

}  // namespace

cudaError_t launch_metadata(const Params& p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                            int32_t* meta, int num_ctas, int first_ctas, cudaStream_t st)
{
    int G = num_ctas < kMaxCtas ? num_ctas : kMaxCtas;
    const int G1 = first_ctas < 1 ? 1 : (first_ctas > G ? G : first_ctas);
    cudaError_t e = cudaFuncSetAttribute(metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMetaSmemMax);
    if (e != cudaSuccess) return e;
    // only what the problem needs, so that score CTAs can share the SM with this one
    const int64_t nb = p.batch < kSmemBatch ? p.batch : kSmemBatch;
    const int64_t ng = p.meta.max_groups < kSmemLive ? p.meta.max_groups : kSmemLive;
    const size_t smem = (size_t)(6 * nb + ng) * 4 + 16;
    return launch_pdl(metadata_kernel, dim3(1), dim3(kMetaThreads), smem, st, p, seq_lens_q,
                      seq_lens_k, meta, G, G1);
}

}  // namespace qli

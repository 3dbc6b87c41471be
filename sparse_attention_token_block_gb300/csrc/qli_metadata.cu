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
//     key_end) units it overlaps, stored CTA by CTA with offsets (computed in parallel over
//     groups).
#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kMetaThreads = 1024;

// Block-wide exclusive scan of one int64 per thread; returns the exclusive prefix and the total.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* total, int64_t* sh /* [32] */)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int64_t warp_excl = warp > 0 ? sh[warp - 1] : 0;
    *total = sh[(blockDim.x >> 5) - 1];
    __syncthreads();
    return warp_excl + x - v;
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
constexpr int kMetaSmemBytes = (5 * kSmemBatch + kSmemGroups + 1) * 4;

__global__ void __launch_bounds__(kMetaThreads, 1)
    metadata_kernel(Params p, const int32_t* __restrict__ seq_lens_q,
                    const int32_t* __restrict__ seq_lens_k, int32_t* __restrict__ meta, int G)
{
    extern __shared__ int32_t msm[];
    __shared__ int64_t scan_sh[32];
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
    const View v_gp = sg ? View{msm + 5 * kSmemBatch, 1} : View{meta + p.meta.group_off, 1};
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
        }
    }
    __syncthreads();

    // ---- query groups per batch (bad TND prefix sums invalidate every batch) and their prefix
    int64_t running = 0;
    for (int base = 0; base < p.batch; base += blockDim.x) {
        const int b = base + tid;
        int64_t groups = 0;
        if (b < p.batch) {
            int32_t* e = be + (int64_t)b * kBatchWords;
            if (s_tnd_bad) e[kBeOk] = 0;
            groups = (!s_tnd_bad && v_ok[b]) ? (v_sq[b] + kGroupTokens - 1) / kGroupTokens : 0;
            e[kBeGroups] = (int32_t)groups;
        }
        int64_t tot;
        const int64_t ex = block_exclusive_scan(groups, &tot, scan_sh);
        if (b < p.batch) {
            be[(int64_t)b * kBatchWords + kBeGroupBase] = (int32_t)(running + ex);
            if (sb) v_gb[b] = (int32_t)(running + ex);
        }
        running += tot;
    }
    const int64_t total_groups = running;
    __syncthreads();

    // ---- tiles per group, then their exclusive prefix (gpre[g]; gpre[total_groups] = total)
    running = 0;
    for (int64_t base = 0; base < total_groups; base += blockDim.x) {
        const int64_t g = base + tid;
        int64_t tiles = 0;
        if (g < total_groups) {
            const int64_t b = upper_index(v_gb, p.batch, g);
            const int64_t r0 = (g - v_gb[b]) * kGroupTokens;
            const int64_t rl = min((int64_t)(r0 + kGroupTokens), (int64_t)v_sq[b]) - 1;
            const int64_t n = visible_keys(p.sparse_mode, p.cmp_ratio, v_sq[b], v_sk[b], v_lc[b], rl);
            tiles = ceil_div64(n, kTileKeys);
        }
        int64_t tot;
        const int64_t ex = block_exclusive_scan(tiles, &tot, scan_sh);
        if (g < total_groups) {
            v_gp[g] = (int32_t)(running + ex);
            if (sg) gpre_home[g] = (int32_t)(running + ex);
        }
        running += tot;
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
    auto cta_of = [&](int64_t t) -> int64_t {     // largest c with floor(T c / G) <= t
        int64_t c = ((t + 1) * Gl + T - 1) / T - 1;
        return c < 0 ? 0 : (c >= Gl ? Gl - 1 : c);
    };
    if (T == 0)
        for (int c = tid; c <= G; c += blockDim.x) cta_off[c] = 0;
    running = 0;
    for (int64_t base = 0; base < total_groups; base += blockDim.x) {
        const int64_t g = base + tid;
        int64_t nu = 0, A = 0, Bt = 0, c0 = 0;
        if (g < total_groups && T > 0) {
            A = v_gp[g];
            Bt = v_gp[g + 1];
            if (Bt > A) {
                c0 = cta_of(A);
                nu = cta_of(Bt - 1) - c0 + 1;
            }
        }
        int64_t tot;
        const int64_t ex = block_exclusive_scan(nu, &tot, scan_sh);
        if (nu > 0) {
            const int64_t b = upper_index(v_gb, p.batch, g);
            const int64_t r0 = (g - v_gb[b]) * kGroupTokens;
            const int64_t rl = min((int64_t)(r0 + kGroupTokens), (int64_t)v_sq[b]) - 1;
            const int64_t n = visible_keys(p.sparse_mode, p.cmp_ratio, v_sq[b], v_sk[b], v_lc[b], rl);
            for (int64_t q = 0; q < nu; ++q) {
                const int64_t c = c0 + q;
                const int64_t t0 = (T * c) / Gl, t1 = (T * (c + 1)) / Gl;
                const int64_t u = running + ex + q;
                int32_t* w = units + u * kUnitWords;
                w[0] = (int32_t)b;
                w[1] = (int32_t)r0;
                w[2] = (int32_t)((max(t0, A) - A) * kTileKeys);
                w[3] = (int32_t)min((min(t1, Bt) - A) * kTileKeys, n);
                if (t0 >= A && t0 < Bt) {
                    // the CTA's first unit; CTAs before it with an empty range (T < G) start here too
                    cta_off[c] = (int32_t)u;
                    for (int64_t ce = c - 1; ce >= 0 && (T * ce) / Gl == t0; --ce) cta_off[ce] = (int32_t)u;
                }
            }
        }
        running += tot;
    }
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
    const int threads = p.meta.max_groups <= 4096 && p.batch <= 4096 ? 256 : kMetaThreads;
    return launch_pdl(metadata_kernel, dim3(1), dim3(threads), kMetaSmemBytes, st, p, seq_lens_q,
                      seq_lens_k, meta, G);
}

}  // namespace qli

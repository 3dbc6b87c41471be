// qli_gather.cu -- the downstream sparse-attention gather (README function section: the selected
// indices are the token indices the sparse attention takes as its input; block_table is the
// PageAttention KV block map).  For every output row r of batch b and every i < sparse_count, with
// j = sparse_indices[r][i]:
//     out[r][i] = kv[block_table[b][j / block_size]][j % block_size]     (entry_bytes bytes)
// and an all-zero entry for j = -1 or an invalid j or page (which also sets an error bit).
//
// A pure copy, bound by HBM: entry_bytes read and written per selected index.  The flattened output
// [rows * k] is cut into runs of kw consecutive entries, one run per warp, kw chosen so that about
// 4096 warps share the work (at most 32 entries a run).  The warp's lanes first resolve the run's entries in parallel (row ->
// batch, bounds, block_table page), then stream the run's bytes as 16-byte chunks, chunk t of the
// run (entry t / n16, piece t % n16) on lane t % 32: the run's output is one contiguous range, and
// each entry's source bytes are contiguous, so both sides coalesce.  Each lane keeps kInFlight
// chunks in flight.  counts[r] comes from CTA r, whose warps re-check the row's indices after their
// own runs: no atomics and no separate zeroing launch, and those CTAs run in the first wave.  (A
// persistent form, each warp resolving its next run while the current one copied, measured no
// faster: the time goes to the random entry reads, not to the address chain.)
#include <cuda_runtime.h>

#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherWarps = kGatherThreads / 32;
constexpr int kInFlight = 8;          // 16-byte chunks each lane has in flight

struct GatherArgs {
    Params p;
    const int32_t* seq_lens_q;        // TND prefix sums (BSND: unused)
    const int32_t* seq_lens_k;        // optional: bounds j by the batch's compressed length
    const int32_t* block_table;
    const int32_t* idx;               // [rows, k]
    const uint4* kv;
    uint4* out;                       // [rows, k, n16] chunks
    int32_t* counts;                  // optional [rows]
    uint32_t* err;                    // optional sticky error word
    int64_t kv_stride16;              // page stride in chunks
    int64_t total;                    // rows * k
    uint32_t n16;                     // chunks per entry (entry_bytes / 16)
    uint32_t n16_magic;               // ceil(2^32 / n16) for n16 > 1: t / n16 = umulhi(t, magic)
                                      // whenever t * n16 < 2^32 (here t < 32 * n16 + 256, n16 <= 4096)
    int32_t kw;                       // entries per warp run
};

// Batch of global row r, or -1: BSND r / S1; TND the b with cum[b-1] <= r < cum[b] (cum[-1] = 0),
// found by binary search for the first prefix sum above r and then checked, so prefix sums that
// are not non-decreasing can never yield an index outside [0, batch).
__device__ __forceinline__ int64_t row_batch(const GatherArgs& a, int64_t r)
{
    const Params& p = a.p;
    if (!p.layout_tnd) return p.s1 > 0 ? r / p.s1 : -1;
    int lo = 0, hi = p.batch;                  // first b in [lo, hi) with cum[b] > r
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a.seq_lens_q[mid] > r) hi = mid;
        else lo = mid + 1;
    }
    if (lo >= p.batch) return -1;
    const int64_t first = lo > 0 ? a.seq_lens_q[lo - 1] : 0, end = a.seq_lens_q[lo];
    return (first <= r && r < end && end <= p.total_q) ? lo : -1;
}

// Exclusive upper bound of valid j in batch b (-1 when the batch's length is invalid).
__device__ __forceinline__ int64_t index_limit(const GatherArgs& a, int64_t b)
{
    const Params& p = a.p;
    int64_t limit = (int64_t)p.max_blocks_per_seq * p.block_size;
    if (a.seq_lens_k) {
        const int64_t sk = a.seq_lens_k[b];
        const int64_t lc = sk < 0 ? -1 : (sk + p.cmp_ratio - 1) / p.cmp_ratio;
        limit = lc < limit ? lc : limit;
    }
    return limit;
}

// Chunk offset of index j's entry in the pool, -1 for a zero entry; error bits into *bits.
__device__ __forceinline__ int64_t entry_source(const GatherArgs& a, int64_t b, int64_t limit, int64_t j,
                                                uint32_t* bits)
{
    if (j == -1) return -1;
    if (b < 0 || j < 0 || j >= limit) {
        *bits |= kErrLength;
        return -1;
    }
    const int64_t bs = a.p.block_size;
    const int64_t page = a.block_table[b * a.p.max_blocks_per_seq + j / bs];
    if (page < 0 || page >= a.p.num_blocks) {
        *bits |= kErrPage;
        return -1;
    }
    return page * a.kv_stride16 + (j % bs) * (int64_t)a.n16;
}

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherArgs a)
{
    __shared__ int warp_counts[kGatherWarps];
    ptx::pdl_wait();                           // the indices may come from the previous kernel
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t warp = (int64_t)blockIdx.x * kGatherWarps + wid;
    const int64_t k = a.p.sparse_count;
    uint32_t bits = 0;
    const int64_t e0 = warp * a.kw;
    if (e0 < a.total) {
        // resolve the run's entries, one per lane (the batch depends on the position only, so the
        // length and the index loads are independent)
        int64_t src = -1;
        const int64_t e = e0 + lane;
        if (lane < a.kw && e < a.total) {
            const int64_t b = row_batch(a, e / k);
            const int64_t limit = b >= 0 ? index_limit(a, b) : -1;
            src = entry_source(a, b, limit, a.idx[e], &bits);
        }
        // copy: chunk t of the run belongs to entry t / n16
        const int64_t run_entries = a.total - e0 < a.kw ? a.total - e0 : a.kw;
        const uint32_t chunks = (uint32_t)run_entries * a.n16;
        uint4* dst = a.out + e0 * a.n16;
        for (uint32_t base = 0; base < chunks; base += 32 * kInFlight) {
            uint4 v[kInFlight];
#pragma unroll
            for (int u = 0; u < kInFlight; ++u) {
                const uint32_t t = base + u * 32 + lane;
                const uint32_t ent = a.n16 == 1 ? t : __umulhi(t, a.n16_magic);
                const int64_t s = __shfl_sync(0xffffffffu, src, ent & 31);
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (t < chunks && s >= 0) v[u] = a.kv[s + (t - ent * a.n16)];
            }
#pragma unroll
            for (int u = 0; u < kInFlight; ++u) {
                const uint32_t t = base + u * 32 + lane;
                if (t < chunks) dst[t] = v[u];
            }
        }
    }
    bits = __reduce_or_sync(0xffffffffu, bits);
    if (bits && lane == 0 && a.err) atomicOr(a.err, bits);
    // counts[r] from CTA r (CTAs of the first wave, so the count overlaps other CTAs' copies): its
    // warps re-check the row's indices, each lane 8 at a time with every load issued before any is
    // used (an invalid index reads table entry 0, which exists whenever limit > 0), and add up
    // through shared memory
    if (a.counts && blockIdx.x < a.p.rows) {
        const int64_t r = blockIdx.x;
        const int64_t b = row_batch(a, r);                 // uniform over the CTA
        const int64_t limit = b >= 0 ? index_limit(a, b) : -1;
        int c = 0;
        if (limit > 0) {
            const int64_t bs = a.p.block_size;
            const int32_t* row = a.idx + r * k;
            const int32_t* table = a.block_table + b * a.p.max_blocks_per_seq;
            for (int64_t i0 = (int64_t)wid * 32 * 8; i0 < k; i0 += (int64_t)kGatherThreads * 8) {
                int32_t j[8], pg[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t i = i0 + u * 32 + lane;
                    j[u] = i < k ? row[i] : -1;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) pg[u] = table[(j[u] >= 0 && j[u] < limit) ? j[u] / bs : 0];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    c += (j[u] >= 0 && j[u] < limit && pg[u] >= 0 && pg[u] < a.p.num_blocks) ? 1 : 0;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0) warp_counts[wid] = c;
        __syncthreads();
        if (threadIdx.x == 0) {
            int total = 0;
#pragma unroll
            for (int w = 0; w < kGatherWarps; ++w) total += warp_counts[w];
            a.counts[r] = total;
        }
    }
}

}  // namespace

cudaError_t launch_gather(const Params& p, const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                          const int32_t* block_table, const int32_t* idx, const void* kv, int64_t entry_bytes,
                          int64_t kv_stride, void* out, int32_t* counts, uint32_t* err, cudaStream_t st)
{
    GatherArgs a;
    a.p = p;
    a.seq_lens_q = seq_lens_q;
    a.seq_lens_k = seq_lens_k;
    a.block_table = block_table;
    a.idx = idx;
    a.kv = static_cast<const uint4*>(kv);
    a.out = static_cast<uint4*>(out);
    a.counts = counts;
    a.err = err;
    a.n16 = (uint32_t)(entry_bytes / 16);
    a.kv_stride16 = kv_stride / 16;
    a.total = (int64_t)p.rows * p.sparse_count;
    // entries per warp: as many as keep about 4096 warps (the GPU's resident warps, a few times
    // over), at most 32 (one per lane)
    const int64_t kw = a.total / 4096;
    a.kw = kw < 1 ? 1 : (kw > 32 ? 32 : (int)kw);
    a.n16_magic = a.n16 > 1 ? (uint32_t)((((uint64_t)1 << 32) + a.n16 - 1) / a.n16) : 0u;
    if (a.total == 0) return cudaSuccess;
    const int64_t warps = (a.total + a.kw - 1) / a.kw;
    int64_t grid = (warps + kGatherWarps - 1) / kGatherWarps;
    if (counts && grid < p.rows) grid = p.rows;           // CTA r counts row r
    return launch_pdl(gather_kernel, dim3((unsigned)grid), dim3(kGatherThreads), 0, st, a);
}

}  // namespace qli

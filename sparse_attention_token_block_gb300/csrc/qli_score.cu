// qli_score.cu -- the scoring kernel: paged key gather, Q.K^T on the tensor cores and the fused
// dequantise / ReLU / weighted head-sum / mask epilogue (README function section, steps 1-3 of
// the out = Top-k{...} formula, up to but excluding the top-k).
//
// One persistent CTA per SM walks the units the metadata assigned to it.  A unit is a query group
// (up to kGroupTokens tokens of one batch, 64 heads each) and a range of its compressed keys, cut
// into tiles of 128 keys.  Per tile:
//
//   producer warp   TMA-loads the tile's key rows (128 B each, 128-byte swizzle) and their scales
//                   from the pages the block_table names into a ring of shared-memory stages;
//   4 convert warps one thread per key: read the row, convert int8 / e4m3 to fp16 exactly and
//                   store it into tensor memory as the MMA's A operand (key = TMEM lane);
//   MMA thread      D[128 keys x 64*tokens] = K_tile[128 x 128] . Q_group^T with tcgen05 kind::f16
//                   (A from tensor memory, B = the group's fp16 query rows in shared memory, fp32
//                   accumulation: int8 products and sums are integers below 2^21, exact in fp32);
//   4 convert warps (epilogue, one tile behind) read their key's row of D and form
//                   score = sK * sum_h (W[h]*|sQ[h]|) * relu_or_min(dot'_h), where dot' uses the
//                   query head negated when sQ[h] < 0 -- algebraically the README's
//                   sum_h W[h] * ReLU(sQ[h] * sK * dot_h) -- then write it as an order-preserving
//                   uint32 into the row's score line if the key is visible under the mask.
//
// Tensor memory: A operand double-buffered in columns [0, 128), D double-buffered in [128, 384).
// Every wait is bounded (about two seconds of wall time); on expiry the kernel records
// kErrTimeout, raises a CTA-wide abort flag and drains out instead of hanging.
#include <cuda.h>
#include <cuda_fp16.h>

#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kStages = 4;                       // key ring depth
constexpr int kConvThreads = 128;                // 4 warps, one key (TMEM lane) per thread
constexpr int kThreads = kConvThreads + 64;      // + producer warp + MMA warp
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = 0;                   // A buffers: 64 columns each (128 fp16 per lane)
constexpr uint32_t kDcol0 = 128;                 // D buffers: 128 columns each (2 tokens x 64)

constexpr int kQbufBytes = kGroupTokens * kHeads * kDim * 2;   // fp16 B operand, 32 KB
constexpr int kKstageBytes = kTileKeys * kDim;                 // 16 KB of key codes
constexpr int kSstageBytes = kTileKeys * 4;                    // scales (fp32 max)
constexpr int kQrawBytes = kGroupTokens * kHeads * kDim;       // 16 KB of query codes
constexpr int kVecRawBytes = kGroupTokens * kHeads * 4;        // weights / q_scale (fp32 max)

// shared memory carve-up (offsets from a 1024-aligned base)
constexpr int kOffQbuf = 0;                                        // 2 x 32 KB
constexpr int kOffKring = kOffQbuf + 2 * kQbufBytes;               // kStages x 16 KB
constexpr int kOffSring = kOffKring + kStages * kKstageBytes;      // kStages x 512 B
constexpr int kOffQraw = kOffSring + kStages * kSstageBytes;       // 2 x 16 KB
constexpr int kOffWraw = kOffQraw + 2 * kQrawBytes;                // 2 x 512 B
constexpr int kOffSQraw = kOffWraw + 2 * kVecRawBytes;             // 2 x 512 B
constexpr int kOffWq = kOffSQraw + 2 * kVecRawBytes;               // 2 x 128 floats
constexpr int kOffSign = kOffWq + 2 * kGroupTokens * kHeads * 4;   // 2 x 128 words
constexpr int kOffBars = kOffSign + 2 * kGroupTokens * kHeads * 4;
enum { kBarKfull = 0, kBarKempty = kStages, kBarQrfull = 2 * kStages, kBarQrempty = kBarQrfull + 2,
       kBarQfull = kBarQrempty + 2, kBarAfull = kBarQfull + 2, kBarDfull = kBarAfull + 2,
       kBarDempty = kBarDfull + 2, kNumBars = kBarDempty + 2 };
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;   // + slack to align the base to 1024

constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct ScoreArgs {
    Params p;
    const uint8_t* query;
    const uint8_t* weights;
    const uint8_t* q_scale;
    const uint8_t* k_scale;
    const int32_t* block_table;
    const int32_t* meta;
    uint32_t* scores;
    uint32_t* err;
};

struct Shared {
    uint8_t* base;
    uint64_t* bars;
    uint32_t* tmem_slot;
    volatile int* abort;
};

// Bounded mbarrier wait: false when the CTA must abort (this wait expired or another did).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         uint32_t* err)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort) return false;
            if (ptx::globaltimer() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(err, kErrTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ float load_scale(const uint8_t* base, int64_t i, bool f32)
{
    if (f32) return reinterpret_cast<const float*>(base)[i];
    return __half2float(reinterpret_cast<const __half*>(base)[i]);
}

// order-preserving map of a float to uint32 (larger float -> larger code); -0 becomes +0
__device__ __forceinline__ uint32_t ordered_code(float s)
{
    if (s == 0.0f) s = 0.0f;
    uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Unit {
    int32_t b, r0, kb, ke;
    int32_t q_cnt, row0, sq, sk, lc;
};

__device__ __forceinline__ Unit read_unit(const ScoreArgs& a, int64_t u)
{
    const int32_t* w = a.meta + a.p.meta.unit_off + u * kUnitWords;
    Unit x;
    x.b = w[0];
    x.r0 = w[1];
    x.kb = w[2];
    x.ke = w[3];
    const int32_t* e = a.meta + a.p.meta.batch_off + (int64_t)x.b * kBatchWords;
    x.sq = e[kBeSq];
    x.sk = e[kBeSk];
    x.lc = e[kBeLc];
    x.row0 = e[kBeFirstRow] + x.r0;
    x.q_cnt = min(kGroupTokens, x.sq - x.r0);
    return x;
}

// ------------------------------------------------------------------------------------------------
// Producer warp: query rows (bulk copies) and key tiles (tensor TMA + scale bulk copies)
// ------------------------------------------------------------------------------------------------
template <bool kScaleF32>
__device__ void producer(const CUtensorMap* tmap, const ScoreArgs& a, const Shared& S, int64_t ubeg,
                         int64_t uend)
{
    const int lane = threadIdx.x & 31;
    const Params& p = a.p;
    constexpr int esz = kScaleF32 ? 4 : 2;
    const int R = p.box_rows;
    const int cpt = kTileKeys / R;            // chunks (TMA boxes) per tile
    uint32_t tile_i = 0;
    for (int64_t u = ubeg; u < uend; ++u) {
        const int uu = (int)(u - ubeg);
        const Unit x = read_unit(a, u);
        const int qb = uu & 1;
        if (!wait_bar(&S.bars[kBarQrempty + qb], ((uu >> 1) & 1) ^ 1, S.abort, a.err)) return;
        if (lane == 0) {
            const uint32_t qbytes = x.q_cnt * kHeads * kDim;
            const uint32_t vbytes = x.q_cnt * kHeads * esz;
            uint64_t* bar = &S.bars[kBarQrfull + qb];
            ptx::mbar_arrive_expect_tx(bar, qbytes + 2 * vbytes);
            ptx::bulk_load(S.base + kOffQraw + qb * kQrawBytes,
                           a.query + (int64_t)x.row0 * kHeads * kDim, qbytes, bar);
            ptx::bulk_load(S.base + kOffWraw + qb * kVecRawBytes,
                           a.weights + (int64_t)x.row0 * kHeads * esz, vbytes, bar);
            ptx::bulk_load(S.base + kOffSQraw + qb * kVecRawBytes,
                           a.q_scale + (int64_t)x.row0 * kHeads * esz, vbytes, bar);
        }
        // key chunks of this unit: chunk c covers keys [kb + c*R, kb + (c+1)*R), inside one page
        const int64_t nchunks = ceil_div64(x.ke - x.kb, R);
        const int32_t* table = a.block_table + (int64_t)x.b * p.max_blocks_per_seq;
        auto page_of = [&](int64_t c) -> int32_t {
            if (c >= nchunks) return 0;
            return __ldg(table + (x.kb + c * R) / p.block_size);
        };
        int32_t cur = page_of(lane), nxt = page_of(32 + lane);
        const int ntiles = (int)ceil_div64(x.ke - x.kb, kTileKeys);
        for (int t = 0; t < ntiles; ++t, ++tile_i) {
            const int s = tile_i % kStages;
            if (!wait_bar(&S.bars[kBarKempty + s], ((tile_i / kStages) & 1) ^ 1, S.abort, a.err)) return;
            const int64_t c0 = (int64_t)t * cpt;
            const int64_t c1 = min((int64_t)(c0 + cpt), nchunks);
            uint64_t* bar = &S.bars[kBarKfull + s];
            if (lane == 0)
                ptx::mbar_arrive_expect_tx(bar, (uint32_t)((c1 - c0) * R * (kDim + esz)));
            for (int64_t c = c0; c < c1; ++c) {
                if ((c & 31) == 0 && c > 0) {   // next window of 32 chunk pages
                    cur = nxt;
                    nxt = page_of(c + 32 + lane);
                }
                int32_t page = __shfl_sync(0xffffffffu, cur, (int)(c & 31));
                if (lane == 0) {
                    if (page < 0 || page >= p.num_blocks) {
                        atomicOr(a.err, kErrPage);
                        page = 0;
                    }
                    const int64_t key0 = x.kb + c * R;
                    const int64_t slot = key0 % p.block_size;
                    const int64_t prow = (int64_t)page * p.block_size + slot;
                    const int r_in_tile = (int)(c - c0) * R;
                    ptx::tma_load_2d(S.base + kOffKring + s * kKstageBytes + r_in_tile * kDim, tmap,
                                     0, (int32_t)prow, bar);
                    ptx::bulk_load(S.base + kOffSring + s * kSstageBytes + r_in_tile * esz,
                                   a.k_scale + prow * esz, (uint32_t)(R * esz), bar);
                }
            }
            __syncwarp();
        }
    }
}

// ------------------------------------------------------------------------------------------------
// MMA thread
// ------------------------------------------------------------------------------------------------
__device__ void mma_issuer(const ScoreArgs& a, const Shared& S, uint32_t tmem, int64_t ubeg,
                           int64_t uend)
{
    uint32_t tile_i = 0;
    for (int64_t u = ubeg; u < uend; ++u) {
        const int uu = (int)(u - ubeg);
        const Unit x = read_unit(a, u);
        const int qb = uu & 1;
        if (!wait_bar(&S.bars[kBarQfull + qb], (uu >> 1) & 1, S.abort, a.err)) return;
        const uint32_t n = kHeads * x.q_cnt;
        const uint32_t idesc = ptx::idesc_f16_f32(128, n);
        const uint32_t qaddr = ptx::smem_addr(S.base + kOffQbuf + qb * kQbufBytes);
        const int ntiles = (int)ceil_div64(x.ke - x.kb, kTileKeys);
        for (int t = 0; t < ntiles; ++t, ++tile_i) {
            const uint32_t ab = tile_i & 1, v = tile_i >> 1;
            if (!wait_bar(&S.bars[kBarAfull + ab], v & 1, S.abort, a.err)) return;
            if (!wait_bar(&S.bars[kBarDempty + ab], (v & 1) ^ 1, S.abort, a.err)) return;
            ptx::tc_fence_after();
            const uint32_t d_t = tmem + kDcol0 + ab * 128;
            const uint32_t a_t = tmem + kAcol0 + ab * 64;
#pragma unroll
            for (int kk = 0; kk < kDim / 16; ++kk) {
                // K step of 16 fp16 = 32 bytes inside a 128-byte swizzle row; the second half of
                // K (dims 64..127) sits in the second block of n rows
                const uint32_t baddr = qaddr + (kk >> 2) * (n * 128) + (kk & 3) * 32;
                ptx::mma_f16_ts(d_t, a_t + kk * 8, ptx::sdesc_kmajor_sw128(baddr), idesc, kk > 0);
            }
            ptx::mma_commit(&S.bars[kBarDfull + ab]);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// Convert + epilogue warps
// ------------------------------------------------------------------------------------------------
struct TileCtx {
    uint32_t tile_i;
    int32_t qb, q_cnt, row0, r0, sq, sk, lc, kend, key0;
    float sk_scale;
};

template <bool kScaleF32>
__device__ bool epilogue(const ScoreArgs& a, const Shared& S, uint32_t tmem, const TileCtx& c)
{
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t ab = c.tile_i & 1, v = c.tile_i >> 1;
    if (!wait_bar(&S.bars[kBarDfull + ab], v & 1, S.abort, a.err)) return false;
    ptx::tc_fence_after();
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float* wq = reinterpret_cast<const float*>(S.base + kOffWq) + c.qb * kGroupTokens * kHeads;
    const int64_t j = c.key0 + tid;
    const Params& p = a.p;
    float score[kGroupTokens];
#pragma unroll
    for (int tt = 0; tt < kGroupTokens; ++tt) {
        score[tt] = 0.0f;
        if (tt < c.q_cnt) {
            uint32_t d[64];
            const uint32_t taddr = tmem + lane_base + kDcol0 + ab * 128 + tt * 64;
            QLI_TMEM_LD_X32(taddr, d);
            QLI_TMEM_LD_X32(taddr + 32, (d + 32));
            ptx::tmem_wait_ld();
            float acc = 0.0f;
            const float* w = wq + tt * kHeads;
            if (c.sk_scale >= 0.0f) {
#pragma unroll
                for (int h = 0; h < kHeads; ++h) acc = fmaf(w[h], fmaxf(__uint_as_float(d[h]), 0.0f), acc);
            } else {
#pragma unroll
                for (int h = 0; h < kHeads; ++h) acc = fmaf(w[h], fminf(__uint_as_float(d[h]), 0.0f), acc);
            }
            score[tt] = c.sk_scale * acc;
        }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if ((tid & 31) == 0) ptx::mbar_arrive(&S.bars[kBarDempty + ab]);
#pragma unroll
    for (int tt = 0; tt < kGroupTokens; ++tt) {
        if (tt < c.q_cnt) {
            const int64_t n = visible_keys(p.sparse_mode, p.cmp_ratio, c.sq, c.sk, c.lc, c.r0 + tt);
            if (j < n && j < c.kend)
                a.scores[(int64_t)(c.row0 + tt) * p.ld + j] = ordered_code(score[tt]);
        }
    }
    return true;
}

template <bool kFp8, bool kScaleF32>
__device__ void converter(const ScoreArgs& a, const Shared& S, uint32_t tmem, int64_t ubeg,
                          int64_t uend)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t tile_i = 0;
    TileCtx prev;
    bool have_prev = false;
    for (int64_t u = ubeg; u < uend; ++u) {
        const int uu = (int)(u - ubeg);
        const Unit x = read_unit(a, u);
        const int qb = uu & 1;
        if (!wait_bar(&S.bars[kBarQrfull + qb], (uu >> 1) & 1, S.abort, a.err)) return;
        // weights folded with |sQ|; heads with sQ < 0 get their query row negated instead
        float* wq = reinterpret_cast<float*>(S.base + kOffWq) + qb * kGroupTokens * kHeads;
        uint32_t* sgn = reinterpret_cast<uint32_t*>(S.base + kOffSign) + qb * kGroupTokens * kHeads;
        const uint8_t* wraw = S.base + kOffWraw + qb * kVecRawBytes;
        const uint8_t* sqraw = S.base + kOffSQraw + qb * kVecRawBytes;
        if (tid < x.q_cnt * kHeads) {
            const float w = load_scale(wraw, tid, kScaleF32);
            const float sq = load_scale(sqraw, tid, kScaleF32);
            wq[tid] = w * fabsf(sq);
            sgn[tid] = sq < 0.0f ? 0x80008000u : 0u;
        }
        ptx::named_bar_sync(1, kConvThreads);
        // query codes -> fp16 B operand: row n = token*64 + head, K-major, 128-byte swizzle, the
        // K halves [0,64) and [64,128) in two blocks of n rows
        const int nrows = x.q_cnt * kHeads;
        const uint8_t* qraw = S.base + kOffQraw + qb * kQrawBytes;
        uint8_t* qbuf = S.base + kOffQbuf + qb * kQbufBytes;
        for (int item = tid; item < nrows * 8; item += kConvThreads) {
            const int n = item >> 3, c16 = item & 7;   // 16 codes = dims [16*c16, 16*c16 + 16)
            const uint4 raw = *reinterpret_cast<const uint4*>(qraw + n * kDim + c16 * 16);
            const uint32_t neg = sgn[n];
            uint32_t h[8];
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (kFp8) ptx::e4m3x4_to_f16x4(wv[q], h[2 * q], h[2 * q + 1]);
                else ptx::int8x4_to_f16x4(wv[q], h[2 * q], h[2 * q + 1]);
                h[2 * q] ^= neg;
                h[2 * q + 1] ^= neg;
            }
            const int blk = c16 >> 2;                   // which 64-dim half
            const int ch = (c16 & 3) * 2;               // first 16-byte chunk within the 128-B row
            uint8_t* row = qbuf + blk * (nrows * 128) + n * 128;
            *reinterpret_cast<uint4*>(row + (((ch) ^ (n & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(row + (((ch + 1) ^ (n & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(1, kConvThreads);
        if (lane == 0) {
            ptx::mbar_arrive(&S.bars[kBarQfull + qb]);
            ptx::mbar_arrive(&S.bars[kBarQrempty + qb]);
        }
        const int ntiles = (int)ceil_div64(x.ke - x.kb, kTileKeys);
        for (int t = 0; t < ntiles; ++t, ++tile_i) {
            const int s = tile_i % kStages;
            if (!wait_bar(&S.bars[kBarKfull + s], (tile_i / kStages) & 1, S.abort, a.err)) return;
            // this thread's key row: 8 chunks of 16 B, chunk c stored at c ^ (row & 7)
            const uint8_t* krow = S.base + kOffKring + s * kKstageBytes + tid * kDim;
            uint4 kr[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                kr[c] = *reinterpret_cast<const uint4*>(krow + ((c ^ (tid & 7)) << 4));
            const float sk = load_scale(S.base + kOffSring + s * kSstageBytes, tid, kScaleF32);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&S.bars[kBarKempty + s]);
            const uint32_t ab = tile_i & 1;
            uint32_t h[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 r = kr[half * 4 + c];
                    const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (kFp8) ptx::e4m3x4_to_f16x4(wv[q], h[c * 8 + 2 * q], h[c * 8 + 2 * q + 1]);
                        else ptx::int8x4_to_f16x4(wv[q], h[c * 8 + 2 * q], h[c * 8 + 2 * q + 1]);
                    }
                }
                QLI_TMEM_ST_X32(tmem + lane_base + kAcol0 + ab * 64 + half * 32, h);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&S.bars[kBarAfull + ab]);
            if (have_prev && !epilogue<kScaleF32>(a, S, tmem, prev)) return;
            prev.tile_i = tile_i;
            prev.qb = qb;
            prev.q_cnt = x.q_cnt;
            prev.row0 = x.row0;
            prev.r0 = x.r0;
            prev.sq = x.sq;
            prev.sk = x.sk;
            prev.lc = x.lc;
            prev.kend = x.ke;
            prev.key0 = x.kb + t * kTileKeys;
            prev.sk_scale = sk;
            have_prev = true;
        }
    }
    if (have_prev) epilogue<kScaleF32>(a, S, tmem, prev);
}

template <bool kFp8, bool kScaleF32>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmap, const ScoreArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Shared S;
    S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    S.bars = reinterpret_cast<uint64_t*>(S.base + kOffBars);
    S.tmem_slot = reinterpret_cast<uint32_t*>(S.base + kOffMisc);
    S.abort = reinterpret_cast<volatile int*>(S.base + kOffMisc + 8);
    const int tid = threadIdx.x, warp = tid >> 5;

    // the metadata must have been written for this problem
    const int32_t* meta = a.meta;
    if (meta[kMhMagic] != kMetaMagic || meta[kMhLayoutHash] != a.p.hash) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(a.err, kErrMetadata);
        return;
    }
    if (blockIdx.x == 0 && tid == 0 && meta[kMhErr]) atomicOr(a.err, (uint32_t)meta[kMhErr]);
    const int G = meta[kMhCtas];

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&S.bars[kBarKfull + i], 1);
            ptx::mbar_init(&S.bars[kBarKempty + i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&S.bars[kBarQrfull + i], 1);
            ptx::mbar_init(&S.bars[kBarQrempty + i], 4);
            ptx::mbar_init(&S.bars[kBarQfull + i], 4);
            ptx::mbar_init(&S.bars[kBarAfull + i], 4);
            ptx::mbar_init(&S.bars[kBarDfull + i], 1);
            ptx::mbar_init(&S.bars[kBarDempty + i], 4);
        }
        *S.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(S.tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *S.tmem_slot;

    // this CTA's unit lists: CTA-lists blockIdx.x, blockIdx.x + gridDim.x, ... (normally one)
    for (int c = blockIdx.x; c < G; c += gridDim.x) {
        const int64_t ubeg = meta[a.p.meta.cta_off + c];
        const int64_t uend = meta[a.p.meta.cta_off + c + 1];
        if (uend <= ubeg) continue;
        if (warp < 4) {
            converter<kFp8, kScaleF32>(a, S, tmem, ubeg, uend);
        } else if (warp == kProducerWarp) {
            producer<kScaleF32>(&tmap, a, S, ubeg, uend);
        } else if (tid == kMmaWarp * 32) {
            mma_issuer(a, S, tmem, ubeg, uend);
        }
        // each CTA-list restarts the barrier phases: only one list per CTA unless the grid is
        // smaller than the split, so re-initialise between lists
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if (c + (int)gridDim.x < G) {
            if (tid == 0) {
                for (int i = 0; i < kNumBars; ++i) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(ptx::smem_addr(&S.bars[i])) : "memory");
                for (int i = 0; i < kStages; ++i) {
                    ptx::mbar_init(&S.bars[kBarKfull + i], 1);
                    ptx::mbar_init(&S.bars[kBarKempty + i], 4);
                }
                for (int i = 0; i < 2; ++i) {
                    ptx::mbar_init(&S.bars[kBarQrfull + i], 1);
                    ptx::mbar_init(&S.bars[kBarQrempty + i], 4);
                    ptx::mbar_init(&S.bars[kBarQfull + i], 4);
                    ptx::mbar_init(&S.bars[kBarAfull + i], 4);
                    ptx::mbar_init(&S.bars[kBarDfull + i], 1);
                    ptx::mbar_init(&S.bars[kBarDempty + i], 4);
                }
                ptx::fence_mbar_init();
            }
            __syncthreads();
        }
        if (*S.abort) break;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

template <bool kFp8, bool kScaleF32>
cudaError_t launch_variant(const CUtensorMap* tmap, const ScoreArgs& a, int grid, cudaStream_t st)
{
    auto k = score_kernel<kFp8, kScaleF32>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, kSmemBytes, st>>>(*tmap, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const Params& p, const void* tmap_key, const void* query, const void* key,
                         const void* weights, const void* q_scale, const void* k_scale,
                         const int32_t* block_table, const int32_t* meta, uint32_t* scores,
                         uint32_t* err_word, int grid, cudaStream_t st)
{
    (void)key;
    ScoreArgs a;
    a.p = p;
    a.query = static_cast<const uint8_t*>(query);
    a.weights = static_cast<const uint8_t*>(weights);
    a.q_scale = static_cast<const uint8_t*>(q_scale);
    a.k_scale = static_cast<const uint8_t*>(k_scale);
    a.block_table = block_table;
    a.meta = meta;
    a.scores = scores;
    a.err = err_word;
    const CUtensorMap* tm = static_cast<const CUtensorMap*>(tmap_key);
    if (p.qk_fp8) {
        return p.scale_f32 ? launch_variant<true, true>(tm, a, grid, st)
                           : launch_variant<true, false>(tm, a, grid, st);
    }
    return p.scale_f32 ? launch_variant<false, true>(tm, a, grid, st)
                       : launch_variant<false, false>(tm, a, grid, st);
}

}  // namespace qli

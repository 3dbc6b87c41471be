// qli_score.cuh -- the scoring kernel: paged key gather, Q.K^T on the tensor cores and the fused
// dequantise / ReLU / weighted head-sum / mask epilogue (README function section, steps 1-3 of
// the out = Top-k{...} formula, up to but excluding the top-k).  Included by two translation units
// that set QLI_SCORE_GT, the most query tokens a group scores together:
//   qli_score.cu        QLI_SCORE_GT 1: two CTAs per SM, 256 tensor-memory columns each (decode
//                       with one query token per sequence: more key copies in flight per SM);
//   qli_score_multi.cu  QLI_SCORE_GT 3: one CTA per SM, all 512 columns (several query tokens per
//                       sequence: each converted key tile serves up to three tokens, MMA N <= 192).
//
// A persistent CTA walks the units the metadata assigned to it.  A unit is a query group (up to
// QLI_SCORE_GT tokens of one batch, 64 heads each) and a range of its compressed keys, cut into tiles
// of 128 keys.  Ten warps (fourteen with two epilogue groups), four roles, connected by mbarriers:
//
//   producer warp    per unit: bulk-copies the group's query codes, weights and query scales;
//                    per tile: TMA-loads the 128 key rows (128 B each, 128-byte swizzle) from the
//                    pages the block_table names into a ring of key stages (the lanes look the
//                    pages up a batch of tiles ahead); its 32 lanes copy the keys' scales with
//                    cp.async into a 10-slot scale ring (own barriers: the epilogue releases them);
//   converter warps  (4) per unit: fold W * |sQ|, convert the query codes to fp16 (negating heads
//                    with sQ < 0) into the MMA's B operand (K-major, 128-byte swizzle), two
//                    buffers;  per tile: one thread per key reads its row, converts int8 / e4m3
//                    to fp16 exactly and stores it into tensor memory as the MMA's A operand (key =
//                    TMEM lane), two A buffers;
//   MMA thread       D[128 keys x 64*tokens] = K_tile[128 x 128] . Q_group^T, tcgen05 kind::f16,
//                    A from tensor memory, B from shared memory, fp32 accumulation (int8 products
//                    and sums are integers below 2^21: exact), two D buffers;
//   epilogue warps   (4 per group; tile i goes to group i mod groups) one thread per key reads
//                    its row of D and forms, per token,
//                    score = sK * sum_h (W[h]*|sQ[h]|) * relu_or_min(dot'_h), where dot' uses the
//                    negated query head when sQ[h] < 0 -- algebraically the README's
//                    sum_h W[h] * ReLU(sQ[h] * sK * dot_h) -- and writes it as an order-preserving
//                    uint32 into the row's score line when the key is visible under the mask.
//
// Tensor memory: A buffers in columns [0, 128), D buffers after them.  The roles are inlined into
// the kernel: as separate functions, each warp's first call fetched its role's code from DRAM
// after the benchmark's L2 flush (long decode score kernel 27.0 -> 24.9 us inlined, prefill
// 742 -> 717 us; ptxas fits every build in the same registers).  Every wait is bounded
// (about two seconds of wall time); on expiry the kernel records kErrTimeout, raises a CTA-wide
// abort flag and drains out instead of hanging.
#ifndef QLI_SCORE_GT
#error "include through qli_score.cu or qli_score_multi.cu"
#endif
#include <cuda.h>
#include <cuda_fp16.h>

#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

constexpr int kGT = QLI_SCORE_GT;                 // most query tokens per group
#if QLI_SCORE_SPLIT
constexpr bool kSplit = true;                     // split-local selection in the epilogue
static_assert(QLI_SCORE_GT == 1, "split-local selection is built for one-token groups");
#else
constexpr bool kSplit = false;
#endif
constexpr int kCtasPerSm = kGT == 1 ? 2 : 1;      // resident score CTAs per SM
// key ring depth (measured): the one-token kernel runs as fast with two, three or four stages and
// three leave the call shortest; groups of three tokens run best with five (with the roles
// inlined: three to five stages 720, 716, 707 us on the prefill), pairs keep five (seven: no
// change); the split build takes two to make room for its chunk
constexpr int kStages = kSplit ? 2 : (kGT == 1 ? 3 : 5);
constexpr int kScaleSlots = 10;                  // scale ring depth (released by the epilogue)
constexpr int kGroups = 1;                       // converter groups; tile i -> i % groups
// epilogue groups: tile i -> group i % kEpiGroups, which drains D buffer i % kNumD.  Groups of
// several tokens give each tile kGT times the epilogue work, so those builds have two groups.
// Groups of two tokens (N = 128) leave tensor memory for a third D buffer, whose use lets the MMAs
// of a tile start before the same group has drained its previous one; a buffer's phases then go
// to the two groups in turn (each phase is drained by one group's four warps).
constexpr int kEpiGroups = kGT == 1 ? 1 : 2;
constexpr int kNumA = 2;                         // A buffers in tensor memory
constexpr int kNumD = kGT == 2 ? 3 : 2;          // D buffers in tensor memory
constexpr int kGroupThreads = 128;               // 4 warps, one key (TMEM lane) per thread
constexpr int kConvWarp0 = 0;                    // converter group g: warps 4g .. 4g+3
constexpr int kEpiWarp0 = 4 * kGroups;           // epilogue group g: warps kEpiWarp0 + 4g ..
constexpr int kProducerWarp = kEpiWarp0 + 4 * kEpiGroups;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kDcols = kHeads * kGT;        // one D buffer (fp32 per lane)
constexpr uint32_t kAcol0 = 0;                   // A buffers: 64 columns each (128 fp16 per lane)
constexpr uint32_t kDcol0 = kNumA * 64;
constexpr uint32_t kTmemCols = 512 / kCtasPerSm; // the CTAs on an SM share its 512 columns
static_assert(kDcol0 + kNumD * kDcols <= kTmemCols, "tensor memory budget");

constexpr int kQbufBytes = kGT * kHeads * kDim * 2;            // fp16 B operand
constexpr int kKstageBytes = kTileKeys * kDim;                 // 16 KB of key codes
constexpr int kSslotBytes = kTileKeys * 4;                     // scales (fp32 max)
constexpr int kQrawBytes = kGT * kHeads * kDim;                // query codes of one group
constexpr int kVecRawBytes = kGT * kHeads * 4;                 // weights / q_scale (fp32 max)

// shared memory carve-up (offsets from a 1024-aligned base)
constexpr int kOffQbuf = 0;                                        // 2 B operands
constexpr int kOffKring = kOffQbuf + 2 * kQbufBytes;               // kStages x 16 KB
constexpr int kOffSring = kOffKring + kStages * kKstageBytes;      // kScaleSlots x 512 B
constexpr int kOffQraw = kOffSring + kScaleSlots * kSslotBytes;    // 1 raw query group
constexpr int kOffWraw = kOffQraw + kQrawBytes;                    // 1 x weights
constexpr int kOffSQraw = kOffWraw + kVecRawBytes;                 // 1 x q_scale
constexpr int kOffWq = kOffSQraw + kVecRawBytes;                   // 2 x W*|sQ|
constexpr int kOffSign = kOffWq + 2 * kGT * kHeads * 4;            // 2 x sign masks
constexpr int kOffBars = kOffSign + 2 * kGT * kHeads * 4;
enum {
    kBarKfull = 0,
    kBarKempty = kBarKfull + kStages,
    kBarSfull = kBarKempty + kStages,
    kBarSempty = kBarSfull + kScaleSlots,
    kBarQrfull = kBarSempty + kScaleSlots,
    kBarQrempty = kBarQrfull + 2,
    kBarQfull = kBarQrempty + 2,
    kBarQempty = kBarQfull + 2,
    kBarAfull = kBarQempty + 2,
    kBarAempty = kBarAfull + kNumA,
    kBarDfull = kBarAempty + kNumA,
    kBarDempty = kBarDfull + kNumD,
    kBarDrain = kBarDempty + kNumD,      // the MMA thread's final commit (all its MMAs done)
    kBarEpi = kBarDrain + 1,             // split build: the epilogue warps meet (4 arrivals)
    kNumBars = kBarEpi + (kSplit ? 1 : 0)
};
// split build: one chunk of scores, then the selection's histograms (two buffers of one 256-bin
// histogram per epilogue warp) and 16 scratch words
constexpr int kOffChunk = (kOffBars + kNumBars * 8 + 15) & ~15;
constexpr int kOffSel = kOffChunk + (kSplit ? kChunkKeys * 4 : 0);
constexpr int kOffMisc = kOffSel + (kSplit ? (2 * 4 * 256 + 16) * 4 : 0);
static_assert(kOffKring % 1024 == 0 && kOffQbuf % 1024 == 0, "shared-memory alignment");
constexpr int kSmemBytes = kOffMisc + 64 + 1024;   // + slack to align the base to 1024
static_assert(kSmemBytes <= (kCtasPerSm == 2 ? 113 : 226) * 1024, "the CTAs of an SM must fit in its shared memory");

constexpr uint64_t kWaitLimitNs = 2000000000ull;

// The epilogue's ReLU as a saturating multiply (FMA pipe) instead of a maximum (half-rate ALU
// pipe): every head dot has |dot| <= 2^25 (int8: 128 * 128^2 = 2^21; e4m3: 128 * 448^2 < 2^25),
// so sat(dot * 2^-25) = ReLU(dot) * 2^-25 exactly, and with the folded weight W|sQ| scaled by 2^25
// (exact) each fma adds the same product W|sQ| ReLU(dot) as before, rounded the same way.  sat
// also sends a NaN dot (an e4m3 NaN code) to 0, as the maximum did.
constexpr float kReluUp = 0x1p25f;
constexpr float kReluDown = 0x1p-25f;


struct ScoreArgs {
    Params p;
    const uint8_t* query;
    const uint8_t* weights;
    const uint8_t* q_scale;
    const uint8_t* k_scale;
    const int32_t* block_table;
    const int32_t* meta;
    const int32_t* seq_lens_q;
    const int32_t* seq_lens_k;
    uint32_t* scores;
    uint32_t* err;
#if QLI_SCORE_SPLIT
    SplitBufs split;
#endif
};

struct Shared {
    uint8_t* base;
    uint64_t* bars;
    uint32_t* tmem_slot;
    volatile int* abort;
};

extern __shared__ uint8_t smem_raw[];

// The CTA's shared-memory carve-up, rebuilt from the dynamic shared memory symbol (cheaper than
// passing it between non-inlined functions through local memory)
__device__ __forceinline__ Shared shared_view()
{
    Shared S;
    S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    S.bars = reinterpret_cast<uint64_t*>(S.base + kOffBars);
    S.tmem_slot = reinterpret_cast<uint32_t*>(S.base + kOffMisc);
    S.abort = reinterpret_cast<volatile int*>(S.base + kOffMisc + 8);
    return S;
}

// Bounded mbarrier wait: false when the CTA must abort (this wait expired or another did).  Each
// test lets the thread sleep up to 100 us until the phase completes.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         uint32_t* err)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort) return false;
        if (ptx::globaltimer() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// Wait, bounded (about 0.2 s) and regardless of the abort flag, for an asynchronous operation this
// CTA issued (a copy into its shared memory, its MMAs) before the CTA releases what it targets.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err)
{
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > 200000000ull) {
            atomicOr(err, kErrTimeout);
            return;
        }
    }
}

__device__ __forceinline__ float load_scale(const uint8_t* base, int i, bool f32)
{
    if (f32) return reinterpret_cast<const float*>(base)[i];
    return __half2float(reinterpret_cast<const __half*>(base)[i]);
}

// order-preserving map of a float to uint32 (larger float -> larger code); -0 becomes +0
__device__ __forceinline__ uint32_t ordered_code(float s)
{
    if (s == 0.0f) s = 0.0f;
    const uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Unit {
    int32_t b, r0, kb, ke;
    int32_t q_cnt, row0, sq, sk, lc;
    int32_t ntiles;
};

// This CTA's tile range [t0, t1) and the live group records [g0, g1) it overlaps, in `recs` (the
// metadata buffer's group records)
struct Span {
    int64_t g0, g1, t0, t1;
    const int32_t* recs;
};

// The unit of live group g within the span: the group's tiles that fall in [t0, t1)
__device__ __forceinline__ Unit read_unit(const ScoreArgs& a, int64_t g, const Span& s)
{
    const int4* w = reinterpret_cast<const int4*>(s.recs + g * kGroupWords);
    const int4 w0 = w[0], w1 = w[1];
    Unit x;
    x.b = w0.x;
    x.r0 = w0.y;
    x.row0 = w0.z;
    x.sq = w0.w;
    x.sk = w1.x;
    x.lc = w1.y;
    const int64_t tb = w1.z, tn = w1.w;
    x.q_cnt = min(a.p.group_tokens, x.sq - x.r0);
    const int64_t n = visible_keys(a.p.sparse_mode, a.p.cmp_ratio, x.sq, x.sk, x.lc, x.r0 + x.q_cnt - 1,
                                   a.p.complete_blocks);
    const int64_t lo = max(s.t0, tb) - tb, hi = max(lo, min(s.t1, tb + tn) - tb);
    x.kb = (int32_t)(lo * kTileKeys);
    x.ke = (int32_t)max((int64_t)x.kb, min(hi * kTileKeys, n));
    x.ntiles = (x.ke - x.kb + kTileKeys - 1) / kTileKeys;
    return x;
}

// ------------------------------------------------------------------------------------------------
// Producer warp
// ------------------------------------------------------------------------------------------------
// The producer's 32 lanes resolve the block_table for a batch of tiles at a time: lane l owns chunk
// (l mod cpt) of tile (l / cpt) of the batch, cpt = 128 / R chunks of R keys per tile, and holds
// that chunk's first row in the key pool (page * block_size + slot).  The next batch (or the next
// unit's first batch) is looked up while the current one is issued, so a tile costs a barrier
// wait, a scale copy and one TMA box per chunk issued by the chunk's lane.  The lanes also fetch
// the key scales (4 keys per lane) with per-thread cp.async copies whose completion the scale
// slot's barrier tracks: TMA copies of a few hundred bytes would double the copy operations per
// tile, and the TMA engine's throughput here is per operation.
template <bool kScaleF32>
__device__ __forceinline__ void produce(const CUtensorMap* tmap, const ScoreArgs& a, const Span& sp,
                                        uint32_t& tile_i, int& q_unit)
{
    const Shared S = shared_view();
    const int lane = threadIdx.x & 31;
    const Params& p = a.p;
    constexpr int esz = kScaleF32 ? 4 : 2;
    const int lgR = __ffs(p.box_rows) - 1;          // R = keys per TMA box: a power of two >= 16
    const int R = 1 << lgR;
    const int lgc = 7 - lgR;                         // cpt = 128 / R chunks per tile
    const int cpt = 1 << lgc;
    const int tpb = 32 >> lgc;                       // tiles per batch
    const int bs = p.block_size;
    const uint64_t key_policy = ptx::policy_evict_first();   // keys are read once: leave L2 to the rest
    if (p.test_stall == 1) return;   // test switch: nothing arrives, the consumers' waits run out
    // this lane's chunk of tile t0 + lane / cpt of unit y: its first key's page (x) and its row in
    // the scale pool, page * bs + slot (y); y = -1 past the unit's keys (a page outside the pool is
    // reported and read as page 0)
    auto chunk_row = [&](const Unit& y, int t0) -> int2 {
        const int key = y.kb + ((t0 + (lane >> lgc)) << 7) + ((lane & (cpt - 1)) << lgR);
        if (key >= y.ke) return make_int2(0, -1);
        const int lp = key / bs;
        int32_t page = __ldg(a.block_table + (int64_t)y.b * p.max_blocks_per_seq + lp);
        if (page < 0 || page >= p.num_blocks) {
            atomicOr(a.err, kErrPage);
            page = 0;
        }
        return make_int2(page, page * bs + (key - lp * bs));
    };
    Unit xn = read_unit(a, sp.g0, sp);
    int2 rows_next = chunk_row(xn, 0);
    for (int64_t u = sp.g0; u < sp.g1; ++u) {
        const int uu = (int)(u - sp.g0);
        const Unit x = xn;
        if (u + 1 < sp.g1) xn = read_unit(a, u + 1, sp);   // in flight while this unit runs
        // one raw query buffer: unit uu's codes land after the converters took unit uu - 1's
        if (!wait_bar(&S.bars[kBarQrempty], (uu & 1) ^ 1, S.abort, a.err)) return;
        if (lane == 0) {
            const uint32_t qbytes = x.q_cnt * kHeads * kDim;
            const uint32_t vbytes = x.q_cnt * kHeads * esz;
            uint64_t* bar = &S.bars[kBarQrfull];
            ptx::mbar_arrive_expect_tx(bar, qbytes + 2 * vbytes);
            ptx::bulk_load(S.base + kOffQraw, a.query + (int64_t)x.row0 * kHeads * kDim, qbytes, bar);
            ptx::bulk_load(S.base + kOffWraw, a.weights + (int64_t)x.row0 * kHeads * esz, vbytes, bar);
            ptx::bulk_load(S.base + kOffSQraw, a.q_scale + (int64_t)x.row0 * kHeads * esz, vbytes, bar);
        }
        q_unit = uu;
        for (int t0 = 0; t0 < x.ntiles; t0 += tpb) {
            const int32_t pages = rows_next.x, rows = rows_next.y;
            // look up the next batch of this unit, else the next unit's first batch
            if (t0 + tpb < x.ntiles) rows_next = chunk_row(x, t0 + tpb);
            else if (u + 1 < sp.g1) rows_next = chunk_row(xn, 0);
            const int nt = min(tpb, x.ntiles - t0);
            for (int tt = 0; tt < nt; ++tt, ++tile_i) {
                const int t = t0 + tt;
                const int s = tile_i % kStages;
                if (!wait_bar(&S.bars[kBarKempty + s], ((tile_i / kStages) & 1) ^ 1, S.abort, a.err)) return;
                const int first = x.kb + (t << 7);
                // scales of this tile: lane l copies those of keys first + 4l .. first + 4l + 3 (one
                // chunk, since R >= 16)
                {
                    const int ss = tile_i % kScaleSlots;
                    if (!wait_bar(&S.bars[kBarSempty + ss], ((tile_i / kScaleSlots) & 1) ^ 1, S.abort, a.err)) return;
                    const int k4 = 4 * lane;
                    const int32_t crow = __shfl_sync(0xffffffffu, rows, (tt << lgc) + (k4 >> lgR));
                    if (first + k4 < x.ke)
                        ptx::cp_async<4 * esz>(S.base + kOffSring + ss * kSslotBytes + lane * 4 * esz,
                                               a.k_scale + ((int64_t)crow + (k4 & (R - 1))) * esz);
                    ptx::cp_async_arrive_noinc(&S.bars[kBarSfull + ss]);
                }
                // key rows: one box per chunk, issued by the chunk's lane
                const int nch = (min(first + kTileKeys, x.ke) - first + R - 1) >> lgR;
                uint64_t* bar = &S.bars[kBarKfull + s];
                const int c = lane - (tt << lgc);
                if (c == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)(nch * R * kDim));
                __syncwarp();
                if (c >= 0 && c < nch)      // the key pool is [pages, bs, 128] with a page stride
                    ptx::tma_load_3d_hint(S.base + kOffKring + s * kKstageBytes + c * R * kDim, tmap, 0,
                                          rows - pages * bs, pages, bar, key_policy);
            }
        }
    }
}

template <bool kScaleF32>
__device__ __forceinline__ void producer(const CUtensorMap* tmap, const ScoreArgs& a, Span sp)
{
    uint32_t tile_i = 0;        // tiles whose copies were issued
    int q_unit = -1;            // last unit whose query copies were issued
    produce<kScaleF32>(tmap, a, sp, tile_i, q_unit);
    // every copy this warp issued lands before the CTA moves on (normally all have been consumed
    // and these waits return at once; after an abort some may still be in flight)
    asm volatile("cp.async.wait_all;" ::: "memory");
    const Shared S = shared_view();
    if ((threadIdx.x & 31) == 0) {
        for (uint32_t t = tile_i > (uint32_t)kStages ? tile_i - kStages : 0u; t < tile_i; ++t)
            drain_wait(&S.bars[kBarKfull + t % kStages], (t / kStages) & 1, a.err);
        if (q_unit >= 0) drain_wait(&S.bars[kBarQrfull], (uint32_t)q_unit & 1, a.err);
    }
    __syncwarp();
}

// ------------------------------------------------------------------------------------------------
// MMA warp
// ------------------------------------------------------------------------------------------------
// The whole warp runs the loop and waits on the barriers; one elected lane issues each tile's MMAs
// and commits.  Every operand is then warp-uniform (the tensor-memory base and the unit's fields
// are broadcast from lane 0), which lets the issuing lane keep the tensor pipe fed: issued from a
// lone thread, the same MMAs go out at about a third of the rate.
__device__ __forceinline__ void issue_mmas(const ScoreArgs& a, uint32_t tmem_any, const Span& sp)
{
    const Shared S = shared_view();
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_any, 0);
    uint32_t tile_i = 0;
    Unit xn = read_unit(a, sp.g0, sp);
    for (int64_t u = sp.g0; u < sp.g1; ++u) {
        const int uu = (int)(u - sp.g0);
        const int q_cnt = __shfl_sync(0xffffffffu, xn.q_cnt, 0);
        const int ntiles = __shfl_sync(0xffffffffu, xn.ntiles, 0);
        if (u + 1 < sp.g1) xn = read_unit(a, u + 1, sp);   // in flight while this unit runs
        const int qb = uu & 1;
        if (!wait_bar(&S.bars[kBarQfull + qb], (uu >> 1) & 1, S.abort, a.err)) return;
        const uint32_t n = kHeads * q_cnt;
        const uint32_t idesc = ptx::idesc_f16_f32(128, n);
        const uint64_t qdesc = ptx::sdesc_kmajor_sw128(ptx::smem_addr(S.base + kOffQbuf + qb * kQbufBytes));
        for (int t = 0; t < ntiles; ++t, ++tile_i) {
            const uint32_t ab = tile_i % kNumA, db = tile_i % kNumD;
            if (!wait_bar(&S.bars[kBarAfull + ab], (tile_i / kNumA) & 1, S.abort, a.err)) return;
            if (!wait_bar(&S.bars[kBarDempty + db], ((tile_i / kNumD) & 1) ^ 1, S.abort, a.err)) return;
            ptx::tc_fence_after();
            const uint32_t d_t = tmem + kDcol0 + db * kDcols;
            const uint32_t a_t = tmem + kAcol0 + ab * 64;
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kDim / 16; ++kk) {
                    // K step of 16 fp16 = 32 bytes inside a 128-byte swizzle row; dims 64..127 sit
                    // in the second block of n rows (the descriptor's address field counts 16 B)
                    const uint64_t bdesc = qdesc + (uint64_t)((((kk >> 2) * (n * 128)) + (kk & 3) * 32) >> 4);
                    ptx::mma_f16_ts(d_t, a_t + kk * 8, bdesc, idesc, kk > 0);
                }
                ptx::mma_commit(&S.bars[kBarDfull + db]);
                ptx::mma_commit(&S.bars[kBarAempty + ab]);
            }
            __syncwarp();
        }
    }
}

__device__ __forceinline__ void mma_issuer(const ScoreArgs& a, uint32_t tmem, Span sp)
{
    issue_mmas(a, tmem, sp);
    // every MMA this warp issued has completed before tensor memory can be released
    const Shared S = shared_view();
    if (ptx::elect_one()) {
        ptx::mma_commit(&S.bars[kBarDrain]);
        drain_wait(&S.bars[kBarDrain], 0, a.err);
    }
    __syncwarp();
}

// ------------------------------------------------------------------------------------------------
// Converter warps: query group -> B operand; key tiles -> A operand in tensor memory
// ------------------------------------------------------------------------------------------------
template <bool kFp8, bool kScaleF32>
__device__ __forceinline__ void converter(const ScoreArgs& a, uint32_t tmem, Span sp)
{
    const Shared S = shared_view();
    if (a.p.test_stall == 2) return;   // test switch: no tile is consumed; the copies wait in the ring
    const int gtid = threadIdx.x - kConvWarp0 * 32;
    const int grp = gtid / kGroupThreads;
    const int tid = gtid % kGroupThreads, lane = tid & 31, warp = tid >> 5;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t tile_i = 0;
    Unit xn = read_unit(a, sp.g0, sp);
    for (int64_t u = sp.g0; u < sp.g1; ++u) {
        const int uu = (int)(u - sp.g0);
        const Unit x = xn;
        if (u + 1 < sp.g1) xn = read_unit(a, u + 1, sp);   // in flight while this unit runs
        const int qb = uu & 1;
        if (uu % kGroups == grp) {   // this group converts the unit's query group
            if (!wait_bar(&S.bars[kBarQrfull], uu & 1, S.abort, a.err)) return;
            if (!wait_bar(&S.bars[kBarQempty + qb], ((uu >> 1) & 1) ^ 1, S.abort, a.err)) return;
            // weights folded with |sQ|; heads with sQ < 0 get their query row negated instead
            float* wq = reinterpret_cast<float*>(S.base + kOffWq) + qb * kGT * kHeads;
            uint32_t* sgn = reinterpret_cast<uint32_t*>(S.base + kOffSign) + qb * kGT * kHeads;
            const uint8_t* wraw = S.base + kOffWraw;
            const uint8_t* sqraw = S.base + kOffSQraw;
            for (int i = tid; i < x.q_cnt * kHeads; i += kGroupThreads) {
                const float w = load_scale(wraw, i, kScaleF32);
                const float sq = load_scale(sqraw, i, kScaleF32);
                wq[i] = w * fabsf(sq) * kReluUp;
                sgn[i] = sq < 0.0f ? 0x80008000u : 0u;
            }
            ptx::named_bar_sync(1 + grp, kGroupThreads);
            // query codes -> fp16 B operand: row n = token*64 + head, K-major, 128-byte swizzle,
            // the K halves [0,64) and [64,128) in two blocks of n rows
            const int nrows = x.q_cnt * kHeads;
            const uint8_t* qraw = S.base + kOffQraw;
            uint8_t* qbuf = S.base + kOffQbuf + qb * kQbufBytes;
            for (int item = tid; item < nrows * 8; item += kGroupThreads) {
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
                const int ch = (c16 & 3) * 2;               // first 16-byte chunk in the 128-B row
                uint8_t* row = qbuf + blk * (nrows * 128) + n * 128;
                *reinterpret_cast<uint4*>(row + ((ch ^ (n & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(row + (((ch + 1) ^ (n & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&S.bars[kBarQfull + qb]);
                ptx::mbar_arrive(&S.bars[kBarQrempty]);
            }
        }
        for (int t = 0; t < x.ntiles; ++t, ++tile_i) {
            if ((int)(tile_i % kGroups) != grp) continue;
            const int s = tile_i % kStages;
            const uint32_t ab = tile_i % kNumA;
            if (!wait_bar(&S.bars[kBarKfull + s], (tile_i / kStages) & 1, S.abort, a.err)) return;
            // this thread's key row: 8 chunks of 16 B, chunk c stored at c ^ (row & 7); converted
            // and stored to tensor memory one 64-dim half at a time
            const uint8_t* krow = S.base + kOffKring + s * kKstageBytes + tid * kDim;
            if (!wait_bar(&S.bars[kBarAempty + ab], ((tile_i / kNumA) & 1) ^ 1, S.abort, a.err)) return;
            ptx::tc_fence_after();
            // the whole 128-byte row comes in first, so the stage is released before any conversion
            uint4 kr[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) kr[c] = *reinterpret_cast<const uint4*>(krow + ((c ^ (tid & 7)) << 4));
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&S.bars[kBarKempty + s]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t h[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = kr[half * 4 + c];
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
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
        }
    }
}

#if QLI_SCORE_SPLIT
// ------------------------------------------------------------------------------------------------
// Split-local selection (epilogue warps of the split build)
// ------------------------------------------------------------------------------------------------
// The four epilogue warps meet on an mbarrier (one arrival per warp) whose wait is bounded like
// every other: a named barrier could not give up if a warp had left on an abort.  The waiters spin
// on the non-blocking test (the other warps arrive within a few hundred cycles; a suspended
// wait resumes far later) and look at the abort flag and the clock every 256 tests.
__device__ __forceinline__ bool epi_sync(const Shared& S, uint32_t& par, uint32_t* err)
{
    __syncwarp();
    uint64_t* bar = &S.bars[kBarEpi];
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
    bool ok = true;
    uint64_t t0 = 0;
    for (uint32_t spin = 1; !ptx::mbar_test_wait(bar, par); ++spin) {
        if ((spin & 255) == 0) {
            if (*S.abort) {
                ok = false;
                break;
            }
            const uint64_t now = ptx::globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitLimitNs) {
                *S.abort = 1;
                atomicOr(err, kErrTimeout);
                ok = false;
                break;
            }
        }
    }
    par ^= 1u;
    return ok;
}

// The chunk [c0, c1) of output row `row` has all its codes in the chunk buffer (position j mod
// kChunkKeys).  A chunk of at most k keys keeps them in the score line; a longer one writes its
// exact top k by (code descending, index ascending) to the candidate lines at [c0, c0 + k), in
// index order.  Either way the chunk's tile words say where its candidates are.  Within a chunk
// the index part of the sort key is fixed above bit 11, so the selection ranks the 44-bit keys
// K = code << 12 | (4095 - position): a radix select from the highest bit in which the chunk's
// keys differ, 8 bits a pass, until the digit that holds the k-th key holds exactly the keys still
// needed; every key with K at or above the prefix found is kept.  Each epilogue warp runs alone on
// its SM sub-partition here, so the loops take four keys a thread per 16-byte load and count into
// a histogram per warp with plain shared atomics, and the histograms are double-buffered (the
// next pass's is cleared while warp 0 scans this one).  False: the CTA is aborting.  Inlined like
// the roles (out of line it spilled, and its code came from DRAM at its first call: split long
// decode call 62.1 -> 61.3 us).
__device__ __forceinline__ bool chunk_select(const ScoreArgs& a, int64_t row, int c0, int c1, uint32_t& par)
{
    const Shared S = shared_view();
    const int tid = threadIdx.x - kEpiWarp0 * 32, lane = tid & 31, warp = tid >> 5;
    const int L = c1 - c0, k = a.p.sparse_count;
    uint32_t* info = a.split.info + row * (a.p.ld / kTileKeys);
    const int t0 = c0 / kTileKeys, nt = (L + kTileKeys - 1) / kTileKeys;
    if (L <= k) {
        // every key is a candidate: the chunk's tiles point at the score line (no one reads the
        // chunk buffer, so the next tiles may overwrite it at once)
        if (tid < nt) info[t0 + tid] = (uint32_t)min(kTileKeys, L - tid * kTileKeys);
        return true;
    }
    // c0 is a multiple of 128, so the chunk's 4-key vectors are 16-byte aligned and the last one
    // ends inside the buffer
    const uint4* buf4 = reinterpret_cast<const uint4*>(S.base + kOffChunk) + ((c0 & (kChunkKeys - 1)) >> 2);
    const int nv = (L + 3) >> 2;
    uint32_t* hist = reinterpret_cast<uint32_t*>(S.base + kOffSel);    // [2][4 warps][256]
    uint32_t* misc = hist + 2 * 4 * 256;                                // [16] scratch
    const uint32_t p0 = (uint32_t)(kChunkKeys - 1 - (c0 & (kChunkKeys - 1)));   // 4095 - position of c0
    if (!epi_sync(S, par, a.err)) return false;                         // every code is in place
    // the highest bit in which the keys differ; the first histogram buffer is cleared meanwhile
    uint32_t mx = 0, mn = 0xFFFFFFFFu;
    for (int v = tid; v < nv; v += kGroupThreads) {
        const uint4 q = buf4[v];
        const uint32_t c[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (4 * v + e < L) {
                mx = max(mx, c[e]);
                mn = min(mn, c[e]);
            }
    }
    for (int i = tid; i < 4 * 256; i += kGroupThreads) hist[i] = 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
        misc[warp] = mx;
        misc[4 + warp] = mn;
    }
    if (!epi_sync(S, par, a.err)) return false;
    mx = max(max(misc[0], misc[1]), max(misc[2], misc[3]));
    mn = min(min(misc[4], misc[5]), min(misc[6], misc[7]));
    // (L >= 2 keys: the positions of the first and last differ)
    int hi = mx != mn ? 12 + 31 - __clz(mx ^ mn) : 31 - __clz(p0 ^ (p0 - (uint32_t)(L - 1)));
    // every key shares the bits above hi (those of the first key): the prefix starts with them
    uint64_t mask = ~((2ull << hi) - 1ull);
    uint64_t prefix = (((uint64_t)mx << 12) | p0) & mask;
    uint32_t rem = (uint32_t)k;
    for (int ps = 0;; ++ps) {
        const int lo = hi >= 7 ? hi - 7 : 0;
        const uint32_t dmask = (2u << (hi - lo)) - 1u;
        uint32_t* H = hist + (ps & 1) * 1024;
        uint32_t* Hw = H + warp * 256;
        // a chunk's leading digits take few values, so most lanes would add to one bin: the lanes
        // whose digit is lane 0's add through one atomic, the others each through their own
        for (int vw = warp * 32; vw < nv; vw += kGroupThreads) {       // warp-uniform trip count
            const int v = vw + lane;
            uint32_t c[4] = {0u, 0u, 0u, 0u};
            if (v < nv) {
                const uint4 q = buf4[v];
                c[0] = q.x;
                c[1] = q.y;
                c[2] = q.z;
                c[3] = q.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 4 * v + e;
                const uint64_t K = ((uint64_t)c[e] << 12) | (p0 - (uint32_t)i);
                const bool in = v < nv && i < L && (K & mask) == prefix;
                const uint32_t d = in ? (uint32_t)(K >> lo) & dmask : 0xFFFFFFFFu;
                const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
                const unsigned same = __ballot_sync(0xffffffffu, in && d == d0);
                if (lane == 0 && same) atomicAdd(&Hw[d0], (uint32_t)__popc(same));
                else if (in && d != d0) atomicAdd(&Hw[d], 1u);
            }
        }
        if (!epi_sync(S, par, a.err)) return false;
        if (warp == 0) {
            // lane l sums digits 255 - 8l down to 248 - 8l over the four warps' histograms; the
            // running count from the top finds the digit where it reaches rem
            uint32_t c8[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int d = 255 - 8 * lane - q;
                c8[q] = H[d] + H[256 + d] + H[512 + d] + H[768 + d];
                sum += c8[q];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
            if (lane == __ffs(hit) - 1) {
                uint32_t above = incl - sum;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (above + c8[q] >= rem) {
                        misc[8] = 255 - 8 * lane - q;
                        misc[9] = rem - above;
                        misc[10] = c8[q] == rem - above ? 1u : 0u;
                        break;
                    }
                    above += c8[q];
                }
            }
        } else {
            uint32_t* Hn = hist + ((ps + 1) & 1) * 1024;       // the next pass's histograms
            for (int i = tid - 32; i < 1024; i += kGroupThreads - 32) Hn[i] = 0;
        }
        if (!epi_sync(S, par, a.err)) return false;
        prefix |= (uint64_t)misc[8] << lo;
        mask |= (uint64_t)dmask << lo;
        rem = misc[9];
        if (misc[10] != 0 || lo == 0) break;     // (all bits fixed: one key, rem = 1)
        hi = lo - 1;
    }
    // the kept keys (K >= prefix) in index order: warp w takes vectors [w per, (w + 1) per), lane
    // l the vector of its step at offset l; a scan of the lanes' counts places each key
    uint32_t* out_code = a.split.code + row * a.p.ld + c0;
    uint32_t* out_idx = a.split.idx + row * a.p.ld + c0;
    const int per = (nv + 3) >> 2;
    const int v0 = warp * per, v1 = min(nv, v0 + per);
    auto takes = [&](int v, uint32_t (&c)[4]) -> uint32_t {    // bit e: key 4v + e is kept
        uint32_t m = 0;
        if (v < v1) {
            const uint4 q = buf4[v];
            c[0] = q.x;
            c[1] = q.y;
            c[2] = q.z;
            c[3] = q.w;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 4 * v + e;
                if (i < L && (((uint64_t)c[e] << 12) | (p0 - (uint32_t)i)) >= prefix) m |= 1u << e;
            }
        }
        return m;
    };
    uint32_t cnt = 0;
    for (int vs = v0; vs < v1; vs += 32) {
        uint32_t c[4];
        cnt += __popc(takes(vs + lane, c));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) misc[12 + warp] = cnt;
    if (!epi_sync(S, par, a.err)) return false;
    uint32_t base = 0;
    for (int w = 0; w < warp; ++w) base += misc[12 + w];
    for (int vs = v0; vs < v1; vs += 32) {
        uint32_t c[4];
        const int v = vs + lane;
        uint32_t m = takes(v, c);
        const uint32_t n = __popc(m);
        uint32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        uint32_t pos = base + incl - n;
        while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1;
            out_code[pos] = c[e];
            out_idx[pos] = (uint32_t)(c0 + 4 * v + e);
            ++pos;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid < nt) info[t0 + tid] = kTileFromCandidates | (uint32_t)max(0, min(kTileKeys, k - tid * kTileKeys));
    return epi_sync(S, par, a.err);               // the chunk buffer may be overwritten again
}
#endif

// ------------------------------------------------------------------------------------------------
// Epilogue warps
// ------------------------------------------------------------------------------------------------
template <bool kScaleF32>
__device__ __forceinline__ void epilogue(const ScoreArgs& a, uint32_t tmem, Span sp)
{
    const Shared S = shared_view();
    const int gtid = threadIdx.x - kEpiWarp0 * 32;
    const int grp = gtid / kGroupThreads;
    const int tid = gtid % kGroupThreads, lane = tid & 31, warp = tid >> 5;
    // a warp reaches the TMEM lanes of its warp index modulo 4; group warps are 4-aligned
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int key_lane = tid;
    const Params& p = a.p;
    uint32_t tile_i = 0;
#if QLI_SCORE_SPLIT
    uint32_t epi_par = 0;       // phase of the epilogue warps' meeting barrier
#endif
    Unit xn = read_unit(a, sp.g0, sp);
    for (int64_t u = sp.g0; u < sp.g1; ++u) {
        const int uu = (int)(u - sp.g0);
        const Unit x = xn;
        if (u + 1 < sp.g1) xn = read_unit(a, u + 1, sp);   // in flight while this unit runs
        const int qb = uu & 1;
        if (!wait_bar(&S.bars[kBarQfull + qb], (uu >> 1) & 1, S.abort, a.err)) return;
        const float* wq = reinterpret_cast<const float*>(S.base + kOffWq) + qb * kGT * kHeads;
        int32_t nvis[kGT];
#pragma unroll
        for (int tt = 0; tt < kGT; ++tt)
            nvis[tt] = tt < x.q_cnt
                           ? (int32_t)min((int64_t)x.ke, visible_keys(p.sparse_mode, p.cmp_ratio, x.sq, x.sk,
                                                                      x.lc, x.r0 + tt, p.complete_blocks))
                           : 0;
        for (int t = 0; t < x.ntiles; ++t, ++tile_i) {
            if ((int)(tile_i % kEpiGroups) != grp) continue;
            const uint32_t db = tile_i % kNumD;
            const int ss = tile_i % kScaleSlots;
            if (!wait_bar(&S.bars[kBarDfull + db], (tile_i / kNumD) & 1, S.abort, a.err)) return;
            ptx::tc_fence_after();
            if (!wait_bar(&S.bars[kBarSfull + ss], (tile_i / kScaleSlots) & 1, S.abort, a.err)) return;
            const float sk = load_scale(S.base + kOffSring + ss * kSslotBytes, key_lane, kScaleF32);
            const int j = x.kb + t * kTileKeys + key_lane;
            float score[kGT];
#pragma unroll
            for (int tt = 0; tt < kGT; ++tt) {
                score[tt] = 0.0f;
                if (tt < x.q_cnt) {
                    const float4* w4 = reinterpret_cast<const float4*>(wq + tt * kHeads);
                    // heads h, h+1 in acc0 and h+2, h+3 in acc1 (packed pairs: four fma chains)
                    uint64_t acc0 = 0, acc1 = 0;
                    // the weighted ReLU sum of heads [h0, h0 + len): W|sQ| 2^25 times
                    // sat(dot 2^-25), i.e. ReLU(dot) for sK >= 0 and ReLU(-dot) = -min(dot, 0)
                    // for sK < 0 (whose sum then takes |sK|)
                    auto accumulate = [&](const uint32_t* d, int h0, int len) {
                        if (sk >= 0.0f) {
#pragma unroll
                            for (int h = 0; h < len; h += 4) {
                                const float4 w = w4[(h0 + h) >> 2];
                                acc0 = ptx::fma2(ptx::pack2(w.x, w.y),
                                                 ptx::pack2(ptx::mul_sat(__uint_as_float(d[h]), kReluDown),
                                                            ptx::mul_sat(__uint_as_float(d[h + 1]), kReluDown)),
                                                 acc0);
                                acc1 = ptx::fma2(ptx::pack2(w.z, w.w),
                                                 ptx::pack2(ptx::mul_sat(__uint_as_float(d[h + 2]), kReluDown),
                                                            ptx::mul_sat(__uint_as_float(d[h + 3]), kReluDown)),
                                                 acc1);
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < len; h += 4) {
                                const float4 w = w4[(h0 + h) >> 2];
                                acc0 = ptx::fma2(ptx::pack2(w.x, w.y),
                                                 ptx::pack2(ptx::mul_sat(__uint_as_float(d[h]), -kReluDown),
                                                            ptx::mul_sat(__uint_as_float(d[h + 1]), -kReluDown)),
                                                 acc0);
                                acc1 = ptx::fma2(ptx::pack2(w.z, w.w),
                                                 ptx::pack2(ptx::mul_sat(__uint_as_float(d[h + 2]), -kReluDown),
                                                            ptx::mul_sat(__uint_as_float(d[h + 3]), -kReluDown)),
                                                 acc1);
                            }
                        }
                    };
                    const uint32_t dcol = tmem + lane_base + kDcol0 + db * kDcols + tt * 64;
                    if constexpr (kGT == 1) {
                        // two loads of 32 heads: the one-token build has registers for 32 at a time
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t d[32];
                            QLI_TMEM_LD_X32(dcol + half * 32, d);
                            ptx::tmem_wait_ld();
                            accumulate(d, half * 32, 32);
                        }
                    } else {
                        // the token's 64 head dots in one load, one wait
                        uint32_t d[64];
                        QLI_TMEM_LD_X64(dcol, d);
                        ptx::tmem_wait_ld();
                        accumulate(d, 0, 64);
                    }
                    float a0, a1, a2, a3;
                    ptx::unpack2(acc0, a0, a1);
                    ptx::unpack2(acc1, a2, a3);
                    score[tt] = fabsf(sk) * ((a0 + a2) + (a1 + a3));
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&S.bars[kBarDempty + db]);
                ptx::mbar_arrive(&S.bars[kBarSempty + ss]);
            }
#pragma unroll
            for (int tt = 0; tt < kGT; ++tt)
                if (tt < x.q_cnt && j < nvis[tt])
                    a.scores[(int64_t)(x.row0 + tt) * p.ld + j] = ordered_code(score[tt]);
#if QLI_SCORE_SPLIT
            // the chunk buffer takes the code too; a chunk ends with the unit or at an aligned
            // kChunkKeys boundary (the units of one-token groups hold visible keys only)
            if (j < nvis[0]) reinterpret_cast<uint32_t*>(S.base + kOffChunk)[j & (kChunkKeys - 1)] = ordered_code(score[0]);
            {
                const int f = x.kb + t * kTileKeys;
                if (t == x.ntiles - 1 || ((f + kTileKeys) & (kChunkKeys - 1)) == 0) {
                    const int c0 = max(x.kb, f & ~(kChunkKeys - 1)), c1 = min(nvis[0], f + kTileKeys);
                    if (!chunk_select(a, x.row0, c0, c1, epi_par)) return;
                }
            }
#endif
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.bars[kBarQempty + qb]);
    }
}

__device__ void init_barriers(const Shared& S)
{
    for (int i = 0; i < kStages; ++i) {
        ptx::mbar_init(&S.bars[kBarKfull + i], 1);
        ptx::mbar_init(&S.bars[kBarKempty + i], 4);
    }
    for (int i = 0; i < kScaleSlots; ++i) {
        ptx::mbar_init(&S.bars[kBarSfull + i], 32);   // one cp.async arrival per producer lane
        ptx::mbar_init(&S.bars[kBarSempty + i], 4);
    }
    for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(&S.bars[kBarQrfull + i], 1);
        ptx::mbar_init(&S.bars[kBarQrempty + i], 4);
        ptx::mbar_init(&S.bars[kBarQfull + i], 4);
        ptx::mbar_init(&S.bars[kBarQempty + i], 4 * kEpiGroups);   // every epilogue warp, per unit
    }
    for (int i = 0; i < kNumA; ++i) {
        ptx::mbar_init(&S.bars[kBarAfull + i], 4);
        ptx::mbar_init(&S.bars[kBarAempty + i], 1);
    }
    for (int i = 0; i < kNumD; ++i) {
        ptx::mbar_init(&S.bars[kBarDfull + i], 1);
        ptx::mbar_init(&S.bars[kBarDempty + i], 4);
    }
    ptx::mbar_init(&S.bars[kBarDrain], 1);
    if (kSplit) ptx::mbar_init(&S.bars[kBarEpi], 4);
    ptx::fence_mbar_init();
}

template <bool kFp8, bool kScaleF32>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    score_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ ScoreArgs a)
{
    const Shared S = shared_view();
    const int tid = threadIdx.x, warp = tid >> 5;

    // prologue that touches no global memory, overlapping the previous kernel's tail
    if (tid == 0) {
        init_barriers(S);
        *S.abort = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(S.tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *S.tmem_slot;
    // the header fields every launch reports: the metadata kernel's error bits, or a mismatch
    auto report_metadata = [&](const int4& h0, const int4& h1, int32_t hash) {
        if (blockIdx.x != 0 || tid != 0) return;
        const bool ok = h0.x == kMetaMagic && hash == a.p.hash;
        if (!ok) atomicOr(a.err, kErrMetadata);
        else if (h1.x) atomicOr(a.err, (uint32_t)h1.x);
    };
    static_assert(kMhMagic == 0 && kMhCtas == 1 && kMhLive == 2 && kMhTiles == 3 && kMhErr == 4, "header layout");
    auto run_span = [&](const Span& sp) {
        if (sp.g1 > sp.g0 && sp.t1 > sp.t0) {
            if (warp < kEpiWarp0) converter<kFp8, kScaleF32>(a, tmem, sp);
            else if (warp < kProducerWarp) epilogue<kScaleF32>(a, tmem, sp);
            else if (warp == kProducerWarp) producer<kScaleF32>(&tmap, a, sp);
            else mma_issuer(a, tmem, sp);
        }
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
    };

    // the metadata comes from the previous kernel and the previous top-k may still read the
    // score lines this kernel overwrites
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    {
        // the metadata must have been written for this problem: the header and this CTA's group
        // range are loaded together (the grid never exceeds kMaxCtas, so the range is inside the
        // buffer whatever it holds)
        const int32_t* meta = a.meta;
        const int4 h0 = *reinterpret_cast<const int4*>(meta);          // magic, G, live groups, tiles
        const int4 h1 = *reinterpret_cast<const int4*>(meta + 4);      // err, batch, rows, groups
        const int32_t h_hash = meta[kMhLayoutHash];
        const int2 mine = reinterpret_cast<const int2*>(meta + a.p.meta.cta_off)[blockIdx.x];
        report_metadata(h0, h1, h_hash);
        const bool meta_ok = h0.x == kMetaMagic && h_hash == a.p.hash;
        const int G = meta_ok ? max(0, min(h0.y, kMaxCtas)) : 0;
        const int64_t live = meta_ok ? max((int64_t)0, min((int64_t)h0.z, a.p.meta.max_groups)) : 0;
        const int64_t T = meta_ok ? max(0, h0.w) : 0;
        const int64_t G1 = meta_ok ? max(1, min(meta[kMhFirst], G)) : 1;   // first-wave CTAs
        // this CTA's tile ranges: CTA-ranges blockIdx.x, blockIdx.x + gridDim.x, ... (normally one)
        for (int c = blockIdx.x; c < G; c += gridDim.x) {
            // group range clamped to the records written, whatever the buffer holds
            const int2 gr = c == (int)blockIdx.x ? mine : reinterpret_cast<const int2*>(meta + a.p.meta.cta_off)[c];
            Span sp;
            sp.t0 = split_start(T, G, G1, c);
            sp.t1 = split_start(T, G, G1, c + 1);
            sp.g0 = max((int64_t)0, min((int64_t)gr.x, live));
            sp.g1 = max(sp.g0, min((int64_t)gr.y, live));
            sp.recs = meta + a.p.meta.group_off;
            run_span(sp);
            if (*S.abort) break;
            if (c + (int)gridDim.x < G) {
                // another range follows: restart every barrier's phase
                if (tid == 0) {
                    for (int i = 0; i < kNumBars; ++i)
                        asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(ptx::smem_addr(&S.bars[i])) : "memory");
                    init_barriers(S);
                }
                __syncthreads();
            }
        }
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
    return launch_pdl(k, dim3(grid), dim3(kThreads), kSmemBytes, st, *tmap, a);
}

}  // namespace

cudaError_t QLI_SCORE_LAUNCHER(const Params& p, const void* tmap_key, const void* query, const void* key,
                         const void* weights, const void* q_scale, const void* k_scale,
                         const int32_t* seq_lens_q, const int32_t* seq_lens_k,
                         const int32_t* block_table, const int32_t* meta, uint32_t* scores,
                         const SplitBufs& split, uint32_t* err_word, int grid, cudaStream_t st)
{
    (void)key;
    (void)split;
    ScoreArgs a;
    a.p = p;
    a.seq_lens_q = seq_lens_q;
    a.seq_lens_k = seq_lens_k;
    a.query = static_cast<const uint8_t*>(query);
    a.weights = static_cast<const uint8_t*>(weights);
    a.q_scale = static_cast<const uint8_t*>(q_scale);
    a.k_scale = static_cast<const uint8_t*>(k_scale);
    a.block_table = block_table;
    a.meta = meta;
    a.scores = scores;
    a.err = err_word;
#if QLI_SCORE_SPLIT
    a.split = split;
#endif
    const CUtensorMap* tm = static_cast<const CUtensorMap*>(tmap_key);
    if (p.qk_fp8) {
        return p.scale_f32 ? launch_variant<true, true>(tm, a, grid, st)
                           : launch_variant<true, false>(tm, a, grid, st);
    }
    return p.scale_f32 ? launch_variant<false, true>(tm, a, grid, st)
                       : launch_variant<false, false>(tm, a, grid, st);
}

}  // namespace qli

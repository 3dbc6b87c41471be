// qli_peak.cu -- rate of the score kernel's tensor-core contraction form (see include/qli_peak.h):
// tcgen05.mma kind::f16, M = 64 or 128, K = 16, N columns, A from tensor memory or shared memory,
// fp32 accumulators in tensor memory.  One warp per CTA issues the MMAs back to back (one elected
// lane, warp-uniform operands), cycling over `chains` accumulators, so the measured interval is the
// tensor pipe's throughput for that shape when each accumulator's MMAs depend on one another
// (chains = 1) or not (chains > 1).
#include <cuda_runtime.h>

#include "qli_peak.h"
#include "qli_ptx.cuh"

namespace {

using namespace qli;

constexpr int kThreads = 128;
constexpr int kMaxN = 256;
constexpr int kAbytes = 128 * 256;                 // A: 128 rows x 128 fp16, two 64-dim blocks
constexpr int kBbytes = kMaxN * 256;               // B: N rows x 128 fp16, two 64-dim blocks
// shared memory per CTA: more than half of an SM's for one CTA per SM, more than a third for two
constexpr int kSmem1 = 120 * 1024;
constexpr int kSmem2 = 100 * 1024;
static_assert(kAbytes + kBbytes + 64 + 1024 <= kSmem2, "shared-memory carve-up");

__global__ void __launch_bounds__(kThreads, 1)
    mma_rate_kernel(int a_tmem, int m, int n, int chains, uint32_t tmem_cols, int iters,
                    unsigned long long* cycles, unsigned long long* nanos, unsigned int* err)
{
    extern __shared__ uint8_t peak_smem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(peak_smem) + 1023) & ~uintptr_t(1023));
    uint8_t* a_s = base;
    uint8_t* b_s = base + kAbytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(b_s + kBbytes);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    // operands: fp16 1.0 everywhere (the values do not change the rate)
    uint32_t* w = reinterpret_cast<uint32_t*>(base);
    for (int i = tid; i < (kAbytes + n * 256) / 4; i += kThreads) w[i] = 0x3C003C00u;
    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(slot, tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *slot;
    if (a_tmem) {
        // A in columns [0, 64): each warp writes its 32 lanes
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0x3C003C00u;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        QLI_TMEM_ST_X32(tmem + lane_base, r);
        QLI_TMEM_ST_X32(tmem + lane_base + 32, r);
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) {
        // the whole warp runs the loop with warp-uniform operands and one elected lane issues (the
        // score kernel's form; issued from a lone thread the same MMAs go out far slower)
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t idesc = ptx::idesc_f16_f32((uint32_t)m, (uint32_t)n);
        const uint64_t ad0 = ptx::sdesc_kmajor_sw128(ptx::smem_addr(a_s));
        const uint64_t bd0 = ptx::sdesc_kmajor_sw128(ptx::smem_addr(b_s));
        const bool leader = ptx::elect_one();
        const unsigned long long c0 = clock64();
        const unsigned long long g0 = ptx::globaltimer();
        // groups of 8 MMAs (the K steps of a 128-dim row, offsets fixed at compile time), group i
        // into accumulator i mod chains, as the score kernel issues one key tile
        int ch = 0;
        for (int i = 0; i < iters / 8; ++i) {
            const uint32_t d = tm + 64 + ch * n;            // accumulator ch: columns [64 + ch n, +n)
            const bool first = i < chains;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    // K step kk: 32 bytes into the 128-byte swizzle row; dims 64..127 in the second block
                    const uint64_t bd = bd0 + (uint64_t)((((kk >> 2) * (n * 128)) + (kk & 3) * 32) >> 4);
                    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
                    if (a_tmem) {
                        ptx::mma_f16_ts(d, tm + kk * 8, bd, idesc, acc);
                    } else {
                        const uint64_t ad = ad0 + (uint64_t)((((kk >> 2) * (128 * 128)) + (kk & 3) * 32) >> 4);
                        ptx::mma_f16_ss(d, ad, bd, idesc, acc);
                    }
                }
            }
            if (++ch == chains) ch = 0;
        }
        if (leader) {
            ptx::mma_commit(bar);
            // bounded wait for every MMA to complete (about 1 s); on expiry record the error and
            // wait once more, bounded, before the tensor memory is released
            bool ok = false;
            for (long long spin = 0; spin < (1ll << 26) && !ok; ++spin) ok = ptx::mbar_try_wait(bar, 0);
            const unsigned long long c1 = clock64();
            const unsigned long long g1 = ptx::globaltimer();
            if (!ok) {
                atomicOr(err, 1u);
                for (long long spin = 0; spin < (1ll << 26) && !ok; ++spin) ok = ptx::mbar_try_wait(bar, 0);
            }
            cycles[blockIdx.x] = c1 - c0;
            nanos[blockIdx.x] = g1 - g0;
        }
        __syncwarp();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, tmem_cols);
}

}  // namespace

extern "C" int qli_peak_mma_f16(int a_from_tmem, int m, int n, int chains, int ctas_per_sm, int iters, int ctas,
                                unsigned long long* cycles, unsigned long long* nanos, unsigned int* err,
                                void* stream)
{
    const bool shape_ok = (m == 128 && n % 16 == 0 && n >= 16) || (m == 64 && !a_from_tmem && n % 8 == 0 && n >= 8);
    if (!shape_ok || n > kMaxN || (ctas_per_sm != 1 && ctas_per_sm != 2) || chains < 1 || iters % 8 != 0 ||
        64 + chains * n > 512 / ctas_per_sm || iters < 1 || ctas < 1 || !cycles || !nanos || !err)
        return (int)cudaErrorInvalidValue;
    const int smem = ctas_per_sm == 1 ? kSmem1 : kSmem2;
    cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    mma_rate_kernel<<<ctas, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
        a_from_tmem ? 1 : 0, m, n, chains, 512u / (uint32_t)ctas_per_sm, iters, cycles, nanos, err);
    return (int)cudaGetLastError();
}

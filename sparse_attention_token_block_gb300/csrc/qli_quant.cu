// qli_quant.cu -- the upstream quantizer (README function section: query and key are quantized per
// token and head, quant mode 0, "store 8-bit, compute 8-bit"; the dequant scales are the formula's
// ScaleQ / ScaleK), and the paged key-cache write of new keys.
//
// Per 128-element (token, head) vector of bfloat16 (symmetric absmax; the README names the mode
// only):  amax = max |x|;  s = amax / Qmax (Qmax = 127 for int8, 448 for e4m3) in fp32, rounded to
// the scale's storage type (fp16: nearest, ties to even, saturating at 65504);  code = x / s in fp32
// rounded to nearest (ties to even) and saturated to the code range;  s = 0 gives zero codes.
//
// Eight lanes per vector: each lane loads 16 bfloat16 as two 16-byte words (elements 8 * lane.. and
// 64 + 8 * lane..), so one warp load instruction reads four whole 128-byte half-vectors.  The group
// reduces |x| on the packed bfloat16 bits (non-negative floats order like unsigned integers), and
// the per-element arithmetic runs two elements at a time in packed fp32 (the same IEEE operations
// as scalar code).  The work is a stream over HBM (2 bytes read and 1 written per element); every
// group loads kUnroll vectors before it computes any, to keep enough bytes in flight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qli_internal.cuh"
#include "qli_ptx.cuh"

namespace qli {

namespace {

using ptx::add2;
using ptx::fma2;
using ptx::mul2;
using ptx::pack2;
using ptx::unpack2;

constexpr int kGroup = 8;                             // lanes per vector
constexpr int kQuantThreads = 256;
constexpr int kVecPerStep = kQuantThreads / kGroup;   // vectors per CTA per unrolled step
#ifndef QLI_QUANT_UNROLL
#define QLI_QUANT_UNROLL 2
#endif
#ifndef QLI_QUANT_MIN_CTAS
#define QLI_QUANT_MIN_CTAS 5     // 5 resident CTAs per SM (at most 51 registers): measured best
#endif
constexpr int kUnroll = QLI_QUANT_UNROLL;             // vectors each group has in flight
constexpr int kVecPerCta = kVecPerStep * kUnroll;
constexpr float kMagic = 12582912.0f;                 // 1.5 * 2^23

struct QuantOut {
    uint2 lo, hi;      // codes of elements 8 * lane + 0..7 and 64 + 8 * lane + 0..7, in byte order
    float scale;       // as stored (fp16 values are exact in fp32)
    uint16_t scale_h;  // the fp16 bits when the storage is fp16
};

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t e4m3x2(uint64_t v)
{
    float lo, hi;
    unpack2(v, lo, hi);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));   // hi -> upper byte
    return r;
}

// Low bytes of the four fp32 lanes of two packed pairs, in lane order.
__device__ __forceinline__ uint32_t low_bytes(uint64_t p, uint64_t q)
{
    float a, b, c, d;
    unpack2(p, a, b);
    unpack2(q, c, d);
    const uint32_t lo = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// The quotient x / s correctly rounded to fp32 (what an IEEE division gives), for 2^-126 <= s <
// 2^125, from r = RN(1/s): q = RN(x * r), then two remainder corrections q <- RN(q + (x - q * s) * r)
// with the remainder formed exactly by a fused multiply-add.  By Markstein's theorem (r within half
// an ulp of 1/s and q within one ulp of x / s give the correctly rounded quotient) the second
// correction is exact; the first brings RN(x * r), which can lie up to 1.5 ulp from x / s, within
// one ulp.  Quotients below 2^-126 in magnitude may differ from the division's, but every such
// quotient gives the code +-0 either way.  X, R and NS (= -s) hold two lanes each.
__device__ __forceinline__ uint64_t quotient2(uint64_t X, uint64_t R, uint64_t NS)
{
    uint64_t Q = mul2(X, R);
    Q = fma2(fma2(Q, NS, X), R, Q);
    return fma2(fma2(Q, NS, X), R, Q);
}

__device__ __forceinline__ bool reciprocal_ok(float s) { return s >= 1.17549435e-38f && s < 4.2535296e37f; }

// Quantize the group's vector; (a, b) hold this lane's 16 elements.  Every lane of the warp must
// call it (the shuffles span the warp; offsets below 8 stay within a group).
__device__ __forceinline__ QuantOut quantize_group(const uint4& a, const uint4& b, bool fp8, bool scale_f32)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max_u16x2(m, w[i] & 0x7FFF7FFFu);
    uint32_t am = max(m & 0xFFFFu, m >> 16);
#pragma unroll
    for (int o = kGroup / 2; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float amax = __uint_as_float(am << 16);
    QuantOut q;
    float s = __fdiv_rn(amax, fp8 ? 448.0f : 127.0f);
    q.scale_h = 0;
    if (!scale_f32) {
        const __half h = __float2half_rn(fminf(s, 65504.0f));
        q.scale_h = __half_as_ushort(h);
        s = __half2float(h);
    }
    q.scale = s;
    q.lo = q.hi = make_uint2(0u, 0u);
    if (s == 0.0f) return q;
    uint64_t y[8];
    float qa;                                   // the largest quotient's magnitude, amax / s
    if (reciprocal_ok(s)) {
        const float r = __frcp_rn(s);
        const uint64_t R = pack2(r, r), NS = pack2(-s, -s);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            y[i] = quotient2(pack2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u)), R, NS);
        float dummy;
        unpack2(quotient2(pack2(amax, 0.0f), R, NS), qa, dummy);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            y[i] = pack2(__fdiv_rn(__uint_as_float(w[i] << 16), s), __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), s));
        qa = __fdiv_rn(amax, s);
    }
    if (fp8) {
        // the quotient of x and s > 0 has x's sign; the remainder corrections can turn a -0 quotient
        // (x = -0, or an underflow) into +0, and e4m3 keeps the sign of zero, so copy x's sign back
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint64_t sign = ((uint64_t)(w[i] & 0x80000000u) << 32) | ((w[i] << 16) & 0x80000000u);
            y[i] = (y[i] & 0x7FFFFFFF7FFFFFFFull) | sign;
        }
        q.lo = make_uint2(e4m3x2(y[0]) | (e4m3x2(y[1]) << 16), e4m3x2(y[2]) | (e4m3x2(y[3]) << 16));
        q.hi = make_uint2(e4m3x2(y[4]) | (e4m3x2(y[5]) << 16), e4m3x2(y[6]) | (e4m3x2(y[7]) << 16));
        return q;
    }
    // int8: round half to even and saturate to [-127, 127].  Quotients are monotone in |x|, so the
    // clamp is needed only when the largest one reaches 127.5 (a scale rounded far below amax / 127:
    // an fp16 subnormal or the 65504 saturation).  After it, y + 1.5 * 2^23 lies in [2^23, 2^24),
    // where fp32 spacing is 1, so the addition rounds y to an integer (ties to even: 1.5 * 2^23 is
    // even) whose two's-complement byte is the sum's low byte (0x4B400000 has a zero low byte).
    if (qa >= 127.5f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float lo, hi;
            unpack2(y[i], lo, hi);
            y[i] = pack2(fminf(fmaxf(lo, -127.0f), 127.0f), fminf(fmaxf(hi, -127.0f), 127.0f));
        }
    }
    const uint64_t M = pack2(kMagic, kMagic);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = add2(y[i], M);
    q.lo = make_uint2(low_bytes(y[0], y[1]), low_bytes(y[2], y[3]));
    q.hi = make_uint2(low_bytes(y[4], y[5]), low_bytes(y[6], y[7]));
    return q;
}

__device__ __forceinline__ void store_scale(void* scales, int64_t i, const QuantOut& q, bool scale_f32)
{
    if (scale_f32) reinterpret_cast<float*>(scales)[i] = q.scale;
    else reinterpret_cast<uint16_t*>(scales)[i] = q.scale_h;
}

// Vector u of CTA c is c * kVecPerCta + u * kVecPerStep + group.
__global__ void __launch_bounds__(kQuantThreads, QLI_QUANT_MIN_CTAS)
    quantize_vectors_kernel(const uint4* __restrict__ x, int64_t nvec, uint2* __restrict__ codes,
                            void* __restrict__ scales, int fp8, int scale_f32)
{
    const int sub = threadIdx.x & (kGroup - 1), grp = threadIdx.x / kGroup;
    const int64_t base = (int64_t)blockIdx.x * kVecPerCta + grp;
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kVecPerStep;
        a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
        if (i < nvec) {
            a[u] = __ldcs(x + i * 16 + sub);
            b[u] = __ldcs(x + i * 16 + 8 + sub);
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kVecPerStep;
        const QuantOut q = quantize_group(a[u], b[u], fp8 != 0, scale_f32 != 0);
        if (i < nvec) {
            codes[i * 16 + sub] = q.lo;
            codes[i * 16 + 8 + sub] = q.hi;
            if (sub == 0) store_scale(scales, i, q, scale_f32 != 0);
        }
    }
}

// Token t as above; the pool slot is looked up through block_table first, and a skipped token
// (bad batch, position or page) still takes part in its group's shuffles.
__global__ void __launch_bounds__(kQuantThreads, QLI_QUANT_MIN_CTAS)
    quantize_keys_kernel(Params p, const uint4* __restrict__ k, int64_t tokens, const int32_t* __restrict__ tok_batch,
                         const int32_t* __restrict__ tok_pos, const int32_t* __restrict__ block_table,
                         uint8_t* __restrict__ pool, void* __restrict__ k_scale, uint32_t* err)
{
    const int sub = threadIdx.x & (kGroup - 1), grp = threadIdx.x / kGroup;
    const int64_t base = (int64_t)blockIdx.x * kVecPerCta + grp;
    const int64_t bs = p.block_size;
    int64_t slot_of[kUnroll];
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t t = base + u * kVecPerStep;
        slot_of[u] = -1;
        a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
        if (t >= tokens) continue;
        const int64_t bt = tok_batch[t], pos = tok_pos[t];
        if (bt < 0 || bt >= p.batch || pos < 0 || pos >= (int64_t)p.max_blocks_per_seq * bs) {
            if (sub == 0 && err) atomicOr(err, kErrLength);
            continue;
        }
        const int64_t page = block_table[bt * p.max_blocks_per_seq + pos / bs];
        if (page < 0 || page >= p.num_blocks) {
            if (sub == 0 && err) atomicOr(err, kErrPage);
            continue;
        }
        slot_of[u] = page * bs + pos % bs;
        a[u] = __ldcs(k + t * 16 + sub);
        b[u] = __ldcs(k + t * 16 + 8 + sub);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const QuantOut q = quantize_group(a[u], b[u], p.qk_fp8 != 0, p.scale_f32 != 0);
        if (slot_of[u] < 0) continue;
        const int64_t page = slot_of[u] / bs, slot = slot_of[u] - page * bs;
        uint2* dst = reinterpret_cast<uint2*>(pool + page * (int64_t)p.key_stride + slot * kDim);
        dst[sub] = q.lo;
        dst[8 + sub] = q.hi;
        if (sub == 0) store_scale(k_scale, slot_of[u], q, p.scale_f32 != 0);
    }
}

}  // namespace

cudaError_t launch_quantize_vectors(const void* x_bf16, int64_t nvec, void* codes, void* scales, bool fp8,
                                    bool scale_f32, cudaStream_t st)
{
    if (nvec == 0) return cudaSuccess;
    const int64_t grid = (nvec + kVecPerCta - 1) / kVecPerCta;
    quantize_vectors_kernel<<<(unsigned)grid, kQuantThreads, 0, st>>>(
        static_cast<const uint4*>(x_bf16), nvec, static_cast<uint2*>(codes), scales, fp8 ? 1 : 0,
        scale_f32 ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_quantize_keys(const Params& p, const void* k_bf16, int64_t tokens, const int32_t* tok_batch,
                                 const int32_t* tok_pos, const int32_t* block_table, void* pool, void* k_scale,
                                 uint32_t* err, cudaStream_t st)
{
    if (tokens == 0) return cudaSuccess;
    const int64_t grid = (tokens + kVecPerCta - 1) / kVecPerCta;
    quantize_keys_kernel<<<(unsigned)grid, kQuantThreads, 0, st>>>(
        p, static_cast<const uint4*>(k_bf16), tokens, tok_batch, tok_pos, block_table, static_cast<uint8_t*>(pool),
        k_scale, err);
    return cudaGetLastError();
}

}  // namespace qli

// qli_quant.cu -- the upstream quantizer (README function section: query and key are quantized per
// token and head, quant mode 0, "store 8-bit, compute 8-bit"; the dequant scales are the formula's
// ScaleQ / ScaleK), and the paged key-cache write of new keys.
//
// Per 128-element (token, head) vector of bfloat16 (symmetric absmax; the README names the mode
// only):  amax = max |x|;  s = amax / Qmax (Qmax = 127 for int8, 448 for e4m3) in fp32, rounded to
// the scale's storage type (fp16: nearest, ties to even, saturating at 65504);  code = x / s in fp32
// rounded to nearest (ties to even) and saturated to the code range;  s = 0 gives zero codes.
//
// One warp per vector: each lane loads 4 bfloat16 (8 bytes), the warp reduces |x|, and each lane
// writes its 4 codes as one 32-bit word.  The work is a stream over HBM (2 bytes read and 1 written
// per element), so the grid simply covers the vectors with 8 warps per CTA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qli_internal.cuh"

namespace qli {

namespace {

constexpr int kQuantWarps = 8;

struct QuantOut {
    uint32_t codes;    // 4 codes, element 4 * lane + i in byte i
    float scale;       // as stored (fp16 values are exact in fp32)
    uint16_t scale_h;  // the fp16 bits when the storage is fp16
};

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));   // hi -> upper byte
    return r;
}

// Quantize the warp's vector; `v` holds this lane's 4 elements (bfloat16 pairs in two words).
__device__ __forceinline__ QuantOut quantize_warp(uint2 v, bool fp8, bool scale_f32)
{
    float x[4];
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    QuantOut q;
    float s = __fdiv_rn(amax, fp8 ? 448.0f : 127.0f);
    q.scale_h = 0;
    if (!scale_f32) {
        const __half h = __float2half_rn(fminf(s, 65504.0f));
        q.scale_h = __half_as_ushort(h);
        s = __half2float(h);
    }
    q.scale = s;
    q.codes = 0;
    if (s != 0.0f) {
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = __fdiv_rn(x[i], s);
        if (fp8) {
            q.codes = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = min(max(__float2int_rn(y[i]), -127), 127);
                q.codes |= (uint32_t)(c & 0xFF) << (8 * i);
            }
        }
    }
    return q;
}

__device__ __forceinline__ void store_scale(void* scales, int64_t i, const QuantOut& q, bool scale_f32)
{
    if (scale_f32) reinterpret_cast<float*>(scales)[i] = q.scale;
    else reinterpret_cast<uint16_t*>(scales)[i] = q.scale_h;
}

__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_vectors_kernel(const uint2* __restrict__ x, int64_t nvec, uint32_t* __restrict__ codes,
                            void* __restrict__ scales, int fp8, int scale_f32)
{
    const int lane = threadIdx.x & 31;
    const int64_t v = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    if (v >= nvec) return;
    const QuantOut q = quantize_warp(x[v * 32 + lane], fp8 != 0, scale_f32 != 0);
    codes[v * 32 + lane] = q.codes;
    if (lane == 0) store_scale(scales, v, q, scale_f32 != 0);
}

__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_keys_kernel(Params p, const uint2* __restrict__ k, int64_t tokens, const int32_t* __restrict__ tok_batch,
                         const int32_t* __restrict__ tok_pos, const int32_t* __restrict__ block_table,
                         uint8_t* __restrict__ pool, void* __restrict__ k_scale, uint32_t* err)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    if (t >= tokens) return;
    const int64_t b = tok_batch[t], pos = tok_pos[t];
    const int64_t bs = p.block_size;
    if (b < 0 || b >= p.batch || pos < 0 || pos >= (int64_t)p.max_blocks_per_seq * bs) {
        if (lane == 0 && err) atomicOr(err, kErrLength);
        return;
    }
    const int64_t page = block_table[b * p.max_blocks_per_seq + pos / bs], slot = pos % bs;
    if (page < 0 || page >= p.num_blocks) {
        if (lane == 0 && err) atomicOr(err, kErrPage);
        return;
    }
    const QuantOut q = quantize_warp(k[t * 32 + lane], p.qk_fp8 != 0, p.scale_f32 != 0);
    reinterpret_cast<uint32_t*>(pool + page * (int64_t)p.key_stride + slot * kDim)[lane] = q.codes;
    if (lane == 0) store_scale(k_scale, page * bs + slot, q, p.scale_f32 != 0);
}

}  // namespace

cudaError_t launch_quantize_vectors(const void* x_bf16, int64_t nvec, void* codes, void* scales, bool fp8,
                                    bool scale_f32, cudaStream_t st)
{
    if (nvec == 0) return cudaSuccess;
    const int64_t grid = (nvec + kQuantWarps - 1) / kQuantWarps;
    quantize_vectors_kernel<<<(unsigned)grid, kQuantWarps * 32, 0, st>>>(
        static_cast<const uint2*>(x_bf16), nvec, static_cast<uint32_t*>(codes), scales, fp8 ? 1 : 0,
        scale_f32 ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_quantize_keys(const Params& p, const void* k_bf16, int64_t tokens, const int32_t* tok_batch,
                                 const int32_t* tok_pos, const int32_t* block_table, void* pool, void* k_scale,
                                 uint32_t* err, cudaStream_t st)
{
    if (tokens == 0) return cudaSuccess;
    const int64_t grid = (tokens + kQuantWarps - 1) / kQuantWarps;
    quantize_keys_kernel<<<(unsigned)grid, kQuantWarps * 32, 0, st>>>(
        p, static_cast<const uint2*>(k_bf16), tokens, tok_batch, tok_pos, block_table, static_cast<uint8_t*>(pool),
        k_scale, err);
    return cudaGetLastError();
}

}  // namespace qli

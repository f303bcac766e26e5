// pkv_quant.cuh -- the per-(block, kv head) symmetric INT8 quantization of
// one 16 x head_dim fp16 tile (PagedKV-Fusion README, "Overview" component B;
// "Architecture": per-block,head symmetric INT8), shared by the quantize
// kernel and the fused append + re-quantize kernel.
//
// A 128-thread CTA owns one tile; thread `tid` holds the 16-byte chunks
// c * 128 + tid (c < kChunks) as raw fp16 bits.  amax = max |x| (NaN
// ignored), scale = fl32(amax / 127), code = round-half-even(fl32(x / scale))
// clamped to [-127, 127], a NaN quotient giving 0; for FP8 (E4M3) codes the
// same with 448 and the nearest E4M3 value of the quotient.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace pkv {

constexpr int kQuantThreads = 128;  // one CTA per (block, kv head, K|V) tile

// RNE(y) for |y| < 2^22 by the exact add of 1.5 * 2^23: the fp32 sum rounds
// to nearest even at unit spacing; its low bits then hold the integer.
constexpr float kRoundMagic = 12582912.0f;

// code = round-half-even(fl32(x / scale)), clamped to [-127, 127]; a NaN
// quotient gives 0.  y' = x * fl32(1/scale) is within 2 ulp of fl32(x/scale);
// ulp <= 2^-17 for |x/scale| <= 127, so when y' is more than 2^-14 away from
// every half-integer both round to the same integer.  Only quotients that
// close to a tie (and NaN/inf cases) take the IEEE division.
__device__ __forceinline__ int quant_code(float x, float scale, float rcp)
{
    const float yf = x * rcp;
    const float t = yf + kRoundMagic;
    const float r = t - kRoundMagic;
    if (fabsf(yf - r) < 0.5f - 0.00006103515625f) {  // 0.5 - 2^-14; false for NaN/inf
        return __float_as_int(t) - 0x4B400000;       // |r| <= 127: no clamp needed
    }
    const float y = __fdiv_rn(x, scale);
    if (isnan(y)) return 0;  // 0/0, inf/inf or a NaN input
    int c = __float2int_rn(y);
    c = c > 127 ? 127 : c;
    c = c < -127 ? -127 : c;
    return c;
}

// max |x| over this thread's chunks (fmaxf drops a NaN operand).
template <int kChunks>
__device__ __forceinline__ float chunks_absmax(const uint4 (&raw)[kChunks])
{
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const __half2 *hp = reinterpret_cast<const __half2 *>(&raw[c]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(hp[e]);
            amax = fmaxf(amax, fabsf(f.x));
            amax = fmaxf(amax, fabsf(f.y));
        }
    }
    return amax;
}

// CTA-wide max of the per-thread values over kThreads threads; warp_max holds
// kThreads / 32 floats of shared memory and may be reused once this returns.
template <int kThreads = kQuantThreads>
__device__ __forceinline__ float cta_absmax(float amax, float *warp_max)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
    __syncthreads();
    return amax;
}

// Threads of a one-tile CTA: one 16-byte chunk (8 values) each.
template <int kHeadDim>
__host__ __device__ constexpr int tile_threads()
{
    return 16 * kHeadDim / 8;
}

// Eight codes of one 16-byte chunk, packed little-endian into a uint2.
__device__ __forceinline__ uint2 chunk_codes(const uint4 &raw, float scale, float rcp)
{
    const __half2 *hp = reinterpret_cast<const __half2 *>(&raw);
    uint32_t packed[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const float2 f0 = __half22float2(hp[2 * w]);
        const float2 f1 = __half22float2(hp[2 * w + 1]);
        const uint32_t b0 = static_cast<uint32_t>(quant_code(f0.x, scale, rcp)) & 0xffu;
        const uint32_t b1 = static_cast<uint32_t>(quant_code(f0.y, scale, rcp)) & 0xffu;
        const uint32_t b2 = static_cast<uint32_t>(quant_code(f1.x, scale, rcp)) & 0xffu;
        const uint32_t b3 = static_cast<uint32_t>(quant_code(f1.y, scale, rcp)) & 0xffu;
        packed[w] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
    return make_uint2(packed[0], packed[1]);
}

// FP8 (OCP E4M3) code of x: the IEEE fp32 quotient x / scale rounded to the
// nearest E4M3 value (ties to even), saturated to +-448; a NaN quotient (0/0,
// inf/inf, NaN input) gives code 0.
__device__ __forceinline__ uint32_t fp8_code(float x, float scale)
{
    const float y = __fdiv_rn(x, scale);
    if (isnan(y)) return 0u;
    return static_cast<uint32_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
}

// Eight FP8 codes of one 16-byte chunk, packed little-endian into a uint2.
__device__ __forceinline__ uint2 chunk_codes_fp8(const uint4 &raw, float scale)
{
    const __half2 *hp = reinterpret_cast<const __half2 *>(&raw);
    uint32_t packed[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const float2 f0 = __half22float2(hp[2 * w]);
        const float2 f1 = __half22float2(hp[2 * w + 1]);
        packed[w] = fp8_code(f0.x, scale) | (fp8_code(f0.y, scale) << 8) |
                    (fp8_code(f1.x, scale) << 16) | (fp8_code(f1.y, scale) << 24);
    }
    return make_uint2(packed[0], packed[1]);
}

}  // namespace pkv

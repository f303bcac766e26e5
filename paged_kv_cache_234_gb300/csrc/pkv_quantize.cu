// pkv_quantize.cu -- symmetric per-(block, kv head) INT8 quantization of fp16
// K and V tiles (PagedKV-Fusion README, "Overview" component B and the
// "Architecture" sequence diagram, where the blocks kept after eviction are
// handed on as INT8 codes with their scales), and the
// same with FP8 (OCP E4M3) codes and scale = amax / 448 ("PagedAttention &
// KV-Cache Memory Management", section 5.1: per-block scaled FP8 KV).
//
// One CTA per (block, kv head, K|V) tile of 16 x head_dim fp16 values, one
// thread per 16-byte chunk (256 threads at head_dim 128; grid-strided when
// there are many tiles).  The tile is read once with
// 16-byte loads (coalesced), max |x| is reduced with warp shuffles and shared
// memory, scale = max / 127 with an IEEE fp32 division, and every code is the
// half-even rounding of the IEEE fp32 quotient x / scale.  HBM-bound for large
// jobs: 2 bytes read and 1 byte written per value, plus 4 bytes of scale per
// tile; for a decode step's few tail blocks it is latency-bound, hence one
// chunk per thread.
#include <cuda_fp16.h>
#include <stdint.h>

#include "pkv_host.cuh"
#include "pkv_ptx.cuh"
#include "pkv_quant.cuh"

namespace pkv {
namespace {

template <int kHeadDim, bool kFp8>
__global__ void __launch_bounds__(tile_threads<kHeadDim>())
    quantize_kernel(const __half *__restrict__ k_in, const __half *__restrict__ v_in,
                    uint8_t *__restrict__ k_out, uint8_t *__restrict__ v_out,
                    float *__restrict__ k_scales, float *__restrict__ v_scales,
                    const int32_t *__restrict__ block_ids, int64_t tiles_per_pool,
                    int num_kv_heads, int num_blocks, int32_t *dev_status)
{
    constexpr int kTileElems = 16 * kHeadDim;
    constexpr int kThreads = tile_threads<kHeadDim>();
    constexpr int kChunks = kTileElems / 8 / kThreads;  // 16-byte chunks per thread (1)
    __shared__ float warp_max[kThreads / 32];
    // programmatic dependent launch: the previous kernel's writes (and its
    // reads of the pools this kernel overwrites) are complete past this point
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    for (int64_t task = blockIdx.x; task < 2 * tiles_per_pool; task += gridDim.x) {
        const bool is_v = task >= tiles_per_pool;
        const int64_t t = is_v ? task - tiles_per_pool : task;
        const int64_t j = t / num_kv_heads;
        const int h = static_cast<int>(t - j * num_kv_heads);
        const int64_t blk = block_ids ? static_cast<int64_t>(__ldg(block_ids + j)) : j;
        if (blk < 0 || blk >= num_blocks) {  // uniform across the CTA
            if (threadIdx.x == 0 && h == 0 && !is_v && dev_status)
                atomicOr(dev_status, PKV_DEV_BAD_BLOCK);
            continue;
        }
        const int64_t tile = blk * num_kv_heads + h;
        const uint4 *src =
            reinterpret_cast<const uint4 *>((is_v ? v_in : k_in) + tile * kTileElems);
        uint2 *dst = reinterpret_cast<uint2 *>((is_v ? v_out : k_out) + tile * kTileElems);

        uint4 raw[kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) raw[c] = __ldcs(src + c * kThreads + threadIdx.x);

        const float amax = cta_absmax<kThreads>(chunks_absmax(raw), warp_max);
        const float scale = __fdiv_rn(amax, kFp8 ? 448.0f : 127.0f);
        const float rcp = __frcp_rn(scale);

#pragma unroll
        for (int c = 0; c < kChunks; ++c)
            __stcs(dst + c * kThreads + threadIdx.x,
                   kFp8 ? chunk_codes_fp8(raw[c], scale) : chunk_codes(raw[c], scale, rcp));
        if (threadIdx.x == 0) (is_v ? v_scales : k_scales)[tile] = scale;
    }
}

}  // namespace
}  // namespace pkv

namespace pkv {
namespace {

pkv_status quantize_entry(const void *k_fp16, const void *v_fp16, void *k_codes, void *v_codes,
                          float *k_scales, float *v_scales, const int32_t *block_ids,
                          int num_ids, int num_blocks, int num_kv_heads, int head_dim,
                          int block_size, int32_t *dev_status, void *stream, bool fp8)
{
    if (!k_fp16 || !v_fp16 || !k_codes || !v_codes || !k_scales || !v_scales)
        return PKV_ERR_INVALID_ARG;
    if (num_blocks <= 0 || num_kv_heads <= 0 || num_ids < 0 || head_dim <= 0 || block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    if (block_size != 16 || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k_fp16, 16) || !aligned(v_fp16, 16) || !aligned(k_codes, 16) ||
        !aligned(v_codes, 16) || !aligned(k_scales, 4) || !aligned(v_scales, 4) ||
        (block_ids && !aligned(block_ids, 4)) || (dev_status && !aligned(dev_status, 4)))
        return PKV_ERR_MISALIGNED;
    const int64_t count = block_ids ? num_ids : num_blocks;
    const int64_t tiles = count * num_kv_heads;
    if (tiles == 0) return PKV_OK;
    // one CTA per tile, grid-strided beyond sixteen CTAs per SM
    DeviceInfo di;
    if (!current_device_info(&di)) return PKV_ERR_CUDA;
    int64_t grid = 2 * tiles;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * 16;
    if (grid > cap) grid = cap;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 g(static_cast<unsigned>(grid)), b(16 * head_dim / 8);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = g;
    cfg.blockDim = b;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const __half *kin = static_cast<const __half *>(k_fp16);
    const __half *vin = static_cast<const __half *>(v_fp16);
    uint8_t *kc = static_cast<uint8_t *>(k_codes), *vc = static_cast<uint8_t *>(v_codes);
    cudaError_t e;
    if (head_dim == 128)
        e = fp8 ? cudaLaunchKernelEx(&cfg, quantize_kernel<128, true>, kin, vin, kc, vc, k_scales,
                                     v_scales, block_ids, tiles, num_kv_heads, num_blocks,
                                     dev_status)
                : cudaLaunchKernelEx(&cfg, quantize_kernel<128, false>, kin, vin, kc, vc,
                                     k_scales, v_scales, block_ids, tiles, num_kv_heads,
                                     num_blocks, dev_status);
    else
        e = fp8 ? cudaLaunchKernelEx(&cfg, quantize_kernel<64, true>, kin, vin, kc, vc, k_scales,
                                     v_scales, block_ids, tiles, num_kv_heads, num_blocks,
                                     dev_status)
                : cudaLaunchKernelEx(&cfg, quantize_kernel<64, false>, kin, vin, kc, vc,
                                     k_scales, v_scales, block_ids, tiles, num_kv_heads,
                                     num_blocks, dev_status);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_quantize_blocks(const void *k_fp16, const void *v_fp16, int8_t *k_codes,
                                          int8_t *v_codes, float *k_scales, float *v_scales,
                                          const int32_t *block_ids, int num_ids, int num_blocks,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int32_t *dev_status, void *stream)
{
    return pkv::quantize_entry(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales, block_ids,
                               num_ids, num_blocks, num_kv_heads, head_dim, block_size,
                               dev_status, stream, false);
}

extern "C" pkv_status pkv_quantize_blocks_fp8(const void *k_fp16, const void *v_fp16,
                                              uint8_t *k_codes, uint8_t *v_codes,
                                              float *k_scales, float *v_scales,
                                              const int32_t *block_ids, int num_ids,
                                              int num_blocks, int num_kv_heads, int head_dim,
                                              int block_size, int32_t *dev_status, void *stream)
{
    return pkv::quantize_entry(k_fp16, v_fp16, k_codes, v_codes, k_scales, v_scales, block_ids,
                               num_ids, num_blocks, num_kv_heads, head_dim, block_size,
                               dev_status, stream, true);
}

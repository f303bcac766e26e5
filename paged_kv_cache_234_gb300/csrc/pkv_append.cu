// pkv_append.cu -- the KV write that precedes a decode step: the new token of
// each sequence goes to slot t % 16 of physical block table[s][t / 16]
// ("PagedAttention & KV-Cache Memory Management", section 2.1 "Logical Token
// Blocks & Page Tables" and the prefill step of "Kernel Mechanics" that
// writes each token at phys_block_id * B + token_offset; section 3.3.2,
// where each step adds only the new tokens to the cache).
//
// fp16 cache: one thread per 16-byte chunk of a new row; a row of head_dim
// fp16 values is 8 or 16 threads, so a warp writes 2 or 4 full rows.
//
// INT8 (or FP8 E4M3) cache: the written (block, kv head) tile is
// re-quantized in the same kernel.  One CTA per (sequence, kv head, K|V)
// tile (a thread per 16-byte chunk) reads the 15 other rows from the fp16 pool, takes the new
// row from the input (and writes it to the fp16 pool), then quantizes the
// tile exactly as the quantize kernel does: bit-identical codes and scale to
// quantizing the tile after a plain fp16 append.  Latency-bound for a decode
// batch: 4 KiB read and about 2.3 KiB written per tile at head_dim 128.
#include <cuda_fp16.h>
#include <stdint.h>

#include "pkv_host.cuh"
#include "pkv_ptx.cuh"
#include "pkv_quant.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

// Physical block of sequence s's new token, or -1 (no token, or an error
// recorded in *dev_status by the caller-chosen reporting thread).
__device__ __forceinline__ int64_t append_block(const int32_t *__restrict__ block_tables,
                                                int max_blocks_per_seq,
                                                const int32_t *__restrict__ positions, int s,
                                                int num_blocks, bool report, int32_t *dev_status,
                                                int *slot)
{
    const int t = __ldg(positions + s);
    if (t < 0) return -1;
    if (t >= max_blocks_per_seq * 16) {
        if (report && dev_status) atomicOr(dev_status, PKV_DEV_BAD_CTX);
        return -1;
    }
    const int64_t blk =
        __ldg(block_tables + static_cast<int64_t>(s) * max_blocks_per_seq + (t >> 4));
    if (blk < 0 || blk >= num_blocks) {
        if (report && dev_status) atomicOr(dev_status, PKV_DEV_BAD_BLOCK);
        return -1;
    }
    *slot = t & 15;
    return blk;
}

__global__ void __launch_bounds__(kAppendThreads)
    append_fp16_kernel(__half *__restrict__ k_pool, __half *__restrict__ v_pool,
                       const __half *__restrict__ k_new, const __half *__restrict__ v_new,
                       const int32_t *__restrict__ block_tables, int max_blocks_per_seq,
                       const int32_t *__restrict__ positions, int num_seqs, int num_kv_heads,
                       int row_chunks, int num_blocks, int32_t *dev_status)
{
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int64_t per_seq = static_cast<int64_t>(2) * num_kv_heads * row_chunks;
    const int64_t total = per_seq * num_seqs;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(i / per_seq);
        const int r = static_cast<int>(i - s * per_seq);
        const int chunk = r % row_chunks;
        const int hv = r / row_chunks;           // (K|V, kv head)
        const bool is_v = hv >= num_kv_heads;
        const int h = is_v ? hv - num_kv_heads : hv;
        int slot = 0;
        const int64_t blk = append_block(block_tables, max_blocks_per_seq, positions, s,
                                         num_blocks, r == 0, dev_status, &slot);
        if (blk < 0) continue;
        const int64_t row = ((blk * num_kv_heads + h) * 16 + slot) * row_chunks;
        const uint4 *src = reinterpret_cast<const uint4 *>(is_v ? v_new : k_new) +
                           (static_cast<int64_t>(s) * num_kv_heads + h) * row_chunks;
        uint4 *dst = reinterpret_cast<uint4 *>(is_v ? v_pool : k_pool) + row;
        dst[chunk] = __ldg(src + chunk);
    }
}

template <int kHeadDim, bool kFp8>
__global__ void __launch_bounds__(tile_threads<kHeadDim>())
    append_int8_kernel(__half *__restrict__ k_pool, __half *__restrict__ v_pool,
                       uint8_t *__restrict__ k_codes, uint8_t *__restrict__ v_codes,
                       float *__restrict__ k_scales, float *__restrict__ v_scales,
                       const __half *__restrict__ k_new, const __half *__restrict__ v_new,
                       const int32_t *__restrict__ block_tables, int max_blocks_per_seq,
                       const int32_t *__restrict__ positions, int num_seqs, int num_kv_heads,
                       int num_blocks, int32_t *dev_status)
{
    constexpr int kRowChunks = kHeadDim / 8;                  // 16-byte chunks per row
    constexpr int kTileChunks = 16 * kRowChunks;
    constexpr int kThreads = tile_threads<kHeadDim>();       // one chunk per thread
    constexpr int kChunks = kTileChunks / kThreads;
    __shared__ float warp_max[kThreads / 32];
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int64_t tiles = static_cast<int64_t>(num_seqs) * num_kv_heads;
    for (int64_t task = blockIdx.x; task < 2 * tiles; task += gridDim.x) {
        const bool is_v = task >= tiles;
        const int64_t t = is_v ? task - tiles : task;
        const int s = static_cast<int>(t / num_kv_heads);
        const int h = static_cast<int>(t - static_cast<int64_t>(s) * num_kv_heads);
        int slot = 0;
        const int64_t blk =
            append_block(block_tables, max_blocks_per_seq, positions, s, num_blocks,
                         threadIdx.x == 0 && h == 0 && !is_v, dev_status, &slot);
        if (blk < 0) continue;  // uniform across the CTA
        const int64_t tile = blk * num_kv_heads + h;
        uint4 *pool = reinterpret_cast<uint4 *>(is_v ? v_pool : k_pool) + tile * kTileChunks;
        const uint4 *fresh = reinterpret_cast<const uint4 *>(is_v ? v_new : k_new) +
                             (static_cast<int64_t>(s) * num_kv_heads + h) * kRowChunks;

        uint4 raw[kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const int idx = c * kThreads + threadIdx.x;
            if (idx / kRowChunks == slot) {
                raw[c] = __ldg(fresh + (idx % kRowChunks));
                pool[idx] = raw[c];
            } else {
                raw[c] = pool[idx];
            }
        }
        const float amax = cta_absmax<kThreads>(chunks_absmax(raw), warp_max);
        const float scale = __fdiv_rn(amax, kFp8 ? 448.0f : 127.0f);
        const float rcp = __frcp_rn(scale);
        uint2 *dst =
            reinterpret_cast<uint2 *>(is_v ? v_codes : k_codes) + tile * kTileChunks;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
            dst[c * kThreads + threadIdx.x] =
                kFp8 ? chunk_codes_fp8(raw[c], scale) : chunk_codes(raw[c], scale, rcp);
        if (threadIdx.x == 0) (is_v ? v_scales : k_scales)[tile] = scale;
    }
}

pkv_status check_append(const void *k_pool, const void *v_pool, const void *k_new,
                        const void *v_new, int num_blocks, const int32_t *block_tables,
                        int max_blocks_per_seq, const int32_t *positions, int num_seqs,
                        int num_kv_heads, int head_dim, int block_size, int32_t *dev_status)
{
    if (!k_pool || !v_pool || !k_new || !v_new || !positions) return PKV_ERR_INVALID_ARG;
    if (num_blocks <= 0 || num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq < 0)
        return PKV_ERR_INVALID_ARG;
    if (!block_tables && num_seqs > 0 && max_blocks_per_seq > 0) return PKV_ERR_INVALID_ARG;
    if (block_size != 16 || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * 16 > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(positions, 4) ||
        (block_tables && !aligned(block_tables, 4)) || (dev_status && !aligned(dev_status, 4)))
        return PKV_ERR_MISALIGNED;
    return PKV_OK;
}

template <typename Kernel, typename... Args>
pkv_status launch_pdl(Kernel kernel, int64_t grid, int threads, void *stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_append_fp16(void *k_cache, void *v_cache, int num_blocks,
                                      const void *k_new, const void *v_new,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *positions, int num_seqs, int num_kv_heads,
                                      int head_dim, int block_size, int32_t *dev_status,
                                      void *stream)
{
    using namespace pkv;
    const pkv_status st =
        check_append(k_cache, v_cache, k_new, v_new, num_blocks, block_tables,
                     max_blocks_per_seq, positions, num_seqs, num_kv_heads, head_dim,
                     block_size, dev_status);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    DeviceInfo di;
    if (!current_device_info(&di)) return PKV_ERR_CUDA;
    const int row_chunks = head_dim / 8;
    const int64_t threads = static_cast<int64_t>(num_seqs) * 2 * num_kv_heads * row_chunks;
    int64_t grid = (threads + kAppendThreads - 1) / kAppendThreads;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * 8;
    if (grid > cap) grid = cap;
    return launch_pdl(append_fp16_kernel, grid, kAppendThreads, stream,
                      static_cast<__half *>(k_cache), static_cast<__half *>(v_cache),
                      static_cast<const __half *>(k_new), static_cast<const __half *>(v_new),
                      block_tables, max_blocks_per_seq, positions, num_seqs, num_kv_heads,
                      row_chunks, num_blocks, dev_status);
}

namespace pkv {
namespace {

pkv_status append_codes(void *k_cache, void *v_cache, void *k_codes, void *v_codes,
                        float *k_scales, float *v_scales, int num_blocks, const void *k_new,
                        const void *v_new, const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *positions, int num_seqs, int num_kv_heads, int head_dim,
                        int block_size, int32_t *dev_status, void *stream, bool fp8)
{
    const pkv_status st =
        check_append(k_cache, v_cache, k_new, v_new, num_blocks, block_tables,
                     max_blocks_per_seq, positions, num_seqs, num_kv_heads, head_dim,
                     block_size, dev_status);
    if (st != PKV_OK) return st;
    if (!k_codes || !v_codes || !k_scales || !v_scales) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_codes, 16) || !aligned(v_codes, 16) || !aligned(k_scales, 4) ||
        !aligned(v_scales, 4))
        return PKV_ERR_MISALIGNED;
    if (num_seqs == 0) return PKV_OK;
    DeviceInfo di;
    if (!current_device_info(&di)) return PKV_ERR_CUDA;
    int64_t grid = static_cast<int64_t>(num_seqs) * num_kv_heads * 2;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * 16;
    if (grid > cap) grid = cap;
    __half *kp = static_cast<__half *>(k_cache), *vp = static_cast<__half *>(v_cache);
    const __half *kn = static_cast<const __half *>(k_new), *vn = static_cast<const __half *>(v_new);
    uint8_t *kc = static_cast<uint8_t *>(k_codes), *vc = static_cast<uint8_t *>(v_codes);
    if (head_dim == 128)
        return fp8 ? launch_pdl(append_int8_kernel<128, true>, grid, tile_threads<128>(), stream, kp,
                                vp, kc, vc, k_scales, v_scales, kn, vn, block_tables,
                                max_blocks_per_seq, positions, num_seqs, num_kv_heads,
                                num_blocks, dev_status)
                   : launch_pdl(append_int8_kernel<128, false>, grid, tile_threads<128>(), stream, kp,
                                vp, kc, vc, k_scales, v_scales, kn, vn, block_tables,
                                max_blocks_per_seq, positions, num_seqs, num_kv_heads,
                                num_blocks, dev_status);
    return fp8 ? launch_pdl(append_int8_kernel<64, true>, grid, tile_threads<64>(), stream, kp, vp,
                            kc, vc, k_scales, v_scales, kn, vn, block_tables,
                            max_blocks_per_seq, positions, num_seqs, num_kv_heads, num_blocks,
                            dev_status)
               : launch_pdl(append_int8_kernel<64, false>, grid, tile_threads<64>(), stream, kp, vp,
                            kc, vc, k_scales, v_scales, kn, vn, block_tables,
                            max_blocks_per_seq, positions, num_seqs, num_kv_heads, num_blocks,
                            dev_status);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_append_int8(void *k_cache, void *v_cache, int8_t *k_codes,
                                      int8_t *v_codes, float *k_scales, float *v_scales,
                                      int num_blocks, const void *k_new, const void *v_new,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *positions, int num_seqs, int num_kv_heads,
                                      int head_dim, int block_size, int32_t *dev_status,
                                      void *stream)
{
    return pkv::append_codes(k_cache, v_cache, k_codes, v_codes, k_scales, v_scales, num_blocks,
                             k_new, v_new, block_tables, max_blocks_per_seq, positions,
                             num_seqs, num_kv_heads, head_dim, block_size, dev_status, stream,
                             false);
}

extern "C" pkv_status pkv_append_fp8(void *k_cache, void *v_cache, uint8_t *k_codes,
                                     uint8_t *v_codes, float *k_scales, float *v_scales,
                                     int num_blocks, const void *k_new, const void *v_new,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *positions, int num_seqs, int num_kv_heads,
                                     int head_dim, int block_size, int32_t *dev_status,
                                     void *stream)
{
    return pkv::append_codes(k_cache, v_cache, k_codes, v_codes, k_scales, v_scales, num_blocks,
                             k_new, v_new, block_tables, max_blocks_per_seq, positions,
                             num_seqs, num_kv_heads, head_dim, block_size, dev_status, stream,
                             true);
}

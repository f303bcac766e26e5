// pkv_copy.cu -- batched block copy for copy-on-write: for every (source,
// destination) pair, every pool's bytes of the source block are copied to the
// destination block ("PagedAttention & KV-Cache Memory Management", section
// 4.1.1: on divergence a fresh page is acquired and the shared page copied
// into it).  One launch copies all pairs of all pools of a cache (K and V, and
// for an INT8 cache also codes and scales): a block's data in a pool
// [num_blocks][...] is one contiguous run of bytes.
//
// One CTA per (pair, pool) copies that run with 16-byte loads and stores
// (4-byte words for pools whose block size or base is not a multiple of 16).
// HBM-bound for large batches: every byte is read once and written once.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_host.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kMaxPools = 8;

struct PoolSet {
    unsigned char *base[kMaxPools];
    long long block_bytes[kMaxPools];
    int wide[kMaxPools];  // 1: 16-byte units, 0: 4-byte units
};

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(const PoolSet ps, int num_blocks, const int32_t *__restrict__ pairs,
                       int num_pairs, int32_t *dev_status)
{
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int pool = blockIdx.y;
    for (int i = blockIdx.x; i < num_pairs; i += gridDim.x) {
        const int src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (pool == 0 && threadIdx.x == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_BLOCK);
            continue;
        }
        if (src == dst) continue;
        const long long nb = ps.block_bytes[pool];
        if (ps.wide[pool]) {
            const uint4 *s = reinterpret_cast<const uint4 *>(ps.base[pool] + src * nb);
            uint4 *d = reinterpret_cast<uint4 *>(ps.base[pool] + dst * nb);
            const long long n = nb >> 4;
            for (long long j = threadIdx.x; j < n; j += kCopyThreads) d[j] = __ldcs(s + j);
        } else {
            const uint32_t *s = reinterpret_cast<const uint32_t *>(ps.base[pool] + src * nb);
            uint32_t *d = reinterpret_cast<uint32_t *>(ps.base[pool] + dst * nb);
            const long long n = nb >> 2;
            for (long long j = threadIdx.x; j < n; j += kCopyThreads) d[j] = __ldcs(s + j);
        }
    }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_copy_blocks(void *const *pools, const int64_t *block_bytes,
                                      int num_pools, int num_blocks, const int32_t *pairs,
                                      int num_pairs, int32_t *dev_status, void *stream)
{
    using namespace pkv;
    if (!pools || !block_bytes || num_pools <= 0 || num_blocks <= 0 || num_pairs < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_pools > kMaxPools) return PKV_ERR_UNSUPPORTED;
    if (num_pairs > 0 && !pairs) return PKV_ERR_INVALID_ARG;
    if ((pairs && !aligned(pairs, 4)) || (dev_status && !aligned(dev_status, 4)))
        return PKV_ERR_MISALIGNED;
    PoolSet ps = {};
    for (int p = 0; p < num_pools; ++p) {
        if (!pools[p] || block_bytes[p] <= 0) return PKV_ERR_INVALID_ARG;
        if (block_bytes[p] % 4 != 0 || !aligned(pools[p], 4)) return PKV_ERR_MISALIGNED;
        ps.base[p] = static_cast<unsigned char *>(pools[p]);
        ps.block_bytes[p] = block_bytes[p];
        ps.wide[p] = block_bytes[p] % 16 == 0 && aligned(pools[p], 16);
    }
    if (num_pairs == 0) return PKV_OK;
    DeviceInfo di;
    if (!current_device_info(&di)) return PKV_ERR_CUDA;
    int64_t gx = num_pairs;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * 8;
    if (gx > cap) gx = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(num_pools));
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, copy_blocks_kernel, ps, num_blocks, pairs, num_pairs,
                           dev_status) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

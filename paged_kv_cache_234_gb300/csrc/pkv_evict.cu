// pkv_evict.cu -- eviction scoring of the physical KV blocks and the choice
// of the k blocks to evict, in one launch.
//
// Score: the least-reference-count + age heuristic ("PagedAttention &
// KV-Cache Memory Management", section 4.3.1):
//   score = alpha * (max_refcnt - refcnt) + beta * (current_tick - last_used)
// in fp32 with one rounding per operation; a larger score is more evictable.
// Every physical block is scored and the eviction ids are returned
// (PagedKV-Fusion README: component A "fused scoring + top-k over paged KV
// blocks" and the sequence diagram's "score all physical blocks" / "eviction
// ids").  Blocks with refcnt <= 0 are free and are never chosen; max_refcnt is
// the largest refcnt of the pool; equal scores go to the smaller block id.
//
// GB300 design: one thread-block cluster (up to 16 CTAs of 1024 threads) owns
// the whole pool; each CTA keeps its slice of 32-bit order keys in shared
// memory, so the pool is read from HBM once.  The k-th largest key is found by
// a four-pass MSB radix select (8-bit digits): every CTA counts its slice into
// a shared-memory histogram (warp-aggregated atomics), one cluster barrier,
// then every CTA sums the cluster's histograms through distributed shared
// memory and picks the same digit.  A final CTA scan plus one more exchange of
// per-CTA counts places the chosen ids, in ascending block-id order.  No
// global atomics, no second launch, no spin-waits: the cluster barrier is the
// hardware's and every CTA of a cluster is resident together.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pkv_host.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kEvThreads = 1024;
constexpr int kEvWarps = kEvThreads / 32;
constexpr int kEvBins = 256;
constexpr int kEvMaxSlice = 49152;    // keys per CTA in shared memory (192 KiB)
constexpr int kEvTargetSlice = 4096;  // keys per CTA that sets the cluster size
constexpr uint32_t kNoBin = 0xffffffffu;

struct EvictParams {
    const int32_t *refcnt;
    const int64_t *last_used;
    float *scores;
    int32_t *ids;
    int32_t *num_evicted;
    long long tick;
    float alpha, beta;
    int num_blocks;
    int slice;  // blocks per CTA
    int k;
};

// Order-preserving map of a (non-NaN) fp32 score to a uint32; -0 maps with
// +0.  The result is never 0, which marks blocks that are not candidates.
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive scan of one value per thread in thread order; *total gets the
// CTA sum.  warp_sums: kEvWarps words of shared memory.
__device__ __forceinline__ uint32_t cta_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const uint32_t before = warp ? warp_sums[warp - 1] : 0u;
    *total = warp_sums[kEvWarps - 1];
    __syncthreads();  // warp_sums is reused by the next scan
    return v + before;
}

__global__ void __launch_bounds__(kEvThreads, 1) evict_kernel(EvictParams p)
{
    extern __shared__ uint32_t keys[];  // this CTA's slice
    __shared__ uint32_t hist[2][kEvBins];
    __shared__ uint32_t warp_sums[kEvWarps];
    __shared__ uint32_t x_ref[2];  // this CTA's max refcnt and candidate count
    __shared__ uint32_t x_sel;     // this CTA's (eq << 16 | gt) selection counts
    __shared__ uint32_t bcast[4];

    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const uint32_t rank = ptx::cluster_ctarank(), csize = ptx::cluster_nctarank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lo = static_cast<int64_t>(rank) * p.slice;
    const int64_t left = static_cast<int64_t>(p.num_blocks) - lo;
    const int n_local = static_cast<int>(left < 0 ? 0 : (left < p.slice ? left : p.slice));

    // 1. reference counts: max and candidates over the pool
    int32_t rmax = 0;
    uint32_t cand = 0;
    for (int j = tid; j < n_local; j += kEvThreads) {
        const int32_t r = __ldg(p.refcnt + lo + j);
        keys[j] = static_cast<uint32_t>(r);
        rmax = max(rmax, r);
        cand += r > 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        rmax = max(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
        cand += __shfl_xor_sync(0xffffffffu, cand, o);
    }
    if (lane == 0) {
        hist[0][warp] = static_cast<uint32_t>(rmax);
        hist[1][warp] = cand;
    }
    __syncthreads();
    if (warp == 0) {
        int32_t m = static_cast<int32_t>(hist[0][lane]);
        uint32_t c = hist[1][lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            c += __shfl_xor_sync(0xffffffffu, c, o);
        }
        if (lane == 0) {
            x_ref[0] = static_cast<uint32_t>(m);
            x_ref[1] = c;
        }
    }
    ptx::cluster_sync();
    if (warp == 0) {
        int32_t m = 0;
        uint32_t c = 0;
        if (static_cast<uint32_t>(lane) < csize) {
            m = static_cast<int32_t>(ptx::ld_cluster_u32(ptx::smem_addr(&x_ref[0]), lane));
            c = ptx::ld_cluster_u32(ptx::smem_addr(&x_ref[1]), lane);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            c += __shfl_xor_sync(0xffffffffu, c, o);
        }
        if (lane == 0) {
            bcast[0] = static_cast<uint32_t>(m);
            bcast[1] = c;
        }
    }
    __syncthreads();
    const int32_t max_ref = static_cast<int32_t>(bcast[0]);
    const uint32_t n_cand = bcast[1];

    // 2. scores (written out) and order keys (kept in shared memory)
    for (int j = tid; j < n_local; j += kEvThreads) {
        const int32_t r = static_cast<int32_t>(keys[j]);
        const long long used = __ldg(reinterpret_cast<const long long *>(p.last_used) + lo + j);
        float sc = -INFINITY;
        uint32_t key = 0;
        if (r > 0) {
            const float d_ref = __int2float_rn(max_ref - r);
            const float d_age = __ll2float_rn(p.tick - used);
            sc = __fadd_rn(__fmul_rn(p.alpha, d_ref), __fmul_rn(p.beta, d_age));
            if (isnan(sc)) sc = -INFINITY;
            key = score_key(sc);
        }
        if (p.scores) p.scores[lo + j] = sc;
        keys[j] = key;
    }
    __syncthreads();

    // 3. threshold: choose every key > thresh and the first kk keys == thresh
    const uint32_t k = static_cast<uint32_t>(p.k);
    uint32_t thresh, kk;
    if (k == 0) {
        thresh = 0xffffffffu;  // no key reaches it
        kk = 0;
    } else if (k >= n_cand) {
        thresh = 0;            // every candidate
        kk = 0;
    } else {
        uint32_t prefix = 0, mask = 0;
        kk = k;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            uint32_t *h = hist[pass & 1];
            if (tid < kEvBins) h[tid] = 0;
            __syncthreads();
            for (int j0 = 0; j0 < n_local; j0 += kEvThreads) {
                const int j = j0 + tid;
                uint32_t bin = kNoBin;
                if (j < n_local) {
                    const uint32_t key = keys[j];
                    if (key != 0 && (key & mask) == prefix) bin = (key >> shift) & 0xffu;
                }
                const uint32_t peers = __match_any_sync(0xffffffffu, bin);
                if (bin != kNoBin && lane == __ffs(peers) - 1) atomicAdd(&h[bin], __popc(peers));
            }
            // every CTA's histogram of this pass is complete past the barrier;
            // the other buffer is the one the next pass clears, and all reads
            // of it (two passes back) finished before this barrier
            ptx::cluster_sync();
            uint32_t cnt = 0;
            if (tid < kEvBins) {
                const uint32_t addr = ptx::smem_addr(&h[kEvBins - 1 - tid]);  // top bin first
                for (uint32_t c = 0; c < csize; ++c) cnt += ptx::ld_cluster_u32(addr, c);
            }
            uint32_t total;
            const uint32_t incl = cta_scan(cnt, warp_sums, &total);
            if (tid < kEvBins && incl - cnt < kk && kk <= incl) {
                bcast[2] = kEvBins - 1 - tid;
                bcast[3] = incl - cnt;  // keys in higher bins
            }
            __syncthreads();
            prefix |= bcast[2] << shift;
            mask |= 0xffu << shift;
            kk -= bcast[3];
            __syncthreads();
        }
        thresh = prefix;
    }

    // 4. place the chosen ids in ascending block-id order: each thread owns a
    // contiguous run of the slice; counts are < 2^16 per CTA, packed in one word
    const int per = (n_local + kEvThreads - 1) / kEvThreads;
    const int j0 = min(tid * per, n_local), j1 = min(j0 + per, n_local);
    uint32_t gt = 0, eq = 0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t key = keys[j];
        gt += key > thresh;
        eq += key == thresh;
    }
    const uint32_t mine = gt | (eq << 16);
    uint32_t cta_total;
    const uint32_t before = cta_scan(mine, warp_sums, &cta_total) - mine;
    if (tid == 0) x_sel = cta_total;
    ptx::cluster_sync();
    if (warp == 0) {
        uint32_t g = 0, e = 0;
        if (static_cast<uint32_t>(lane) < rank) {
            const uint32_t v = ptx::ld_cluster_u32(ptx::smem_addr(&x_sel), lane);
            g = v & 0xffffu;
            e = v >> 16;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (lane == 0) {
            bcast[0] = g;
            bcast[1] = e;
        }
    }
    __syncthreads();
    uint32_t gt_b = bcast[0] + (before & 0xffffu), eq_b = bcast[1] + (before >> 16);
    for (int j = j0; j < j1; ++j) {
        const uint32_t key = keys[j];
        // an output slot is below k by construction; the check keeps every
        // store inside the caller's k-entry buffer regardless
        if (key > thresh) {
            const uint32_t at = gt_b + min(eq_b, kk);
            if (at < k) p.ids[at] = static_cast<int32_t>(lo + j);
            ++gt_b;
        } else if (key == thresh) {
            if (eq_b < kk && gt_b + eq_b < k) p.ids[gt_b + eq_b] = static_cast<int32_t>(lo + j);
            ++eq_b;
        }
    }

    // 5. the count, and -1 in the unused tail of the id buffer
    const uint32_t n_sel = k < n_cand ? k : n_cand;
    if (rank == 0 && tid == 0) *p.num_evicted = static_cast<int32_t>(n_sel);
    for (int64_t i = n_sel + static_cast<int64_t>(rank) * kEvThreads + tid; i < p.k;
         i += static_cast<int64_t>(csize) * kEvThreads)
        p.ids[i] = -1;
    ptx::cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

// One-time set-up per device: allow the full shared-memory slice, and find
// the largest cluster size the device schedules for this kernel (16 if the
// non-portable size fits, else the portable 8).  Returns 0 on a CUDA error.
int evict_setup(int device)
{
    static std::atomic<int> cache[64];
    if (device < 0 || device >= 64) return 0;
    int c = cache[device].load(std::memory_order_relaxed);
    if (c) return c;
    if (cudaFuncSetAttribute(evict_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kEvMaxSlice * sizeof(uint32_t))) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    c = 8;
    if (cudaFuncSetAttribute(evict_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(kEvThreads);
        cfg.dynamicSmemBytes = kEvMaxSlice * sizeof(uint32_t);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, evict_kernel, &cfg) == cudaSuccess &&
            clusters >= 1)
            c = 16;
    }
    cudaGetLastError();
    cache[device].store(c, std::memory_order_relaxed);
    return c;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_evict_select(const int32_t *refcnt, const int64_t *last_used,
                                       int num_blocks, int64_t current_tick, float alpha,
                                       float beta, int k, float *scores, int32_t *evict_ids,
                                       int32_t *num_evicted, void *stream)
{
    using namespace pkv;
    if (num_blocks < 0 || k < 0 || !num_evicted) return PKV_ERR_INVALID_ARG;
    if (num_blocks > 0 && (!refcnt || !last_used)) return PKV_ERR_INVALID_ARG;
    if (k > 0 && !evict_ids) return PKV_ERR_INVALID_ARG;
    if (!isfinite(alpha) || !isfinite(beta)) return PKV_ERR_INVALID_ARG;
    if ((refcnt && !aligned(refcnt, 4)) || (last_used && !aligned(last_used, 8)) ||
        (scores && !aligned(scores, 4)) || (evict_ids && !aligned(evict_ids, 4)) ||
        !aligned(num_evicted, 4))
        return PKV_ERR_MISALIGNED;
    DeviceInfo di;
    if (!current_device_info(&di)) return PKV_ERR_CUDA;
    const int cmax = evict_setup(di.device);
    if (!cmax) return PKV_ERR_CUDA;
    int64_t csize = (static_cast<int64_t>(num_blocks) + kEvTargetSlice - 1) / kEvTargetSlice;
    if (csize < 1) csize = 1;
    if (csize > cmax) csize = cmax;
    const int64_t slice = (static_cast<int64_t>(num_blocks) + csize - 1) / csize;
    if (slice > kEvMaxSlice) return PKV_ERR_UNSUPPORTED;
    const size_t smem = static_cast<size_t>(slice > 0 ? slice : 1) * sizeof(uint32_t);
    EvictParams prm;
    prm.refcnt = refcnt;
    prm.last_used = last_used;
    prm.scores = scores;
    prm.ids = evict_ids;
    prm.num_evicted = num_evicted;
    prm.tick = current_tick;
    prm.alpha = alpha;
    prm.beta = beta;
    prm.num_blocks = num_blocks;
    prm.slice = static_cast<int>(slice);
    prm.k = k;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(csize));
    cfg.blockDim = dim3(kEvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, evict_kernel, prm) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

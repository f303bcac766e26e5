// pkv_evict.cu -- eviction scoring of the physical KV blocks and the choice
// of the k blocks to evict, in one launch.
//
// Score: the least-reference-count + age heuristic ("PagedAttention &
// KV-Cache Memory Management", section 4.3.1):
//   score = alpha * (max_refcnt - refcnt) + beta * (current_tick - last_used)
// in fp32 with one rounding per operation; a larger score is more evictable.
// Every physical block is scored and the eviction ids are returned
// (PagedKV-Fusion README: Overview, component A, a CUDA kernel that scores
// the blocks and selects k of them in one pass, and the Architecture
// sequence diagram, where the eviction kernel scores every physical block
// and returns the ids of the k blocks to evict to its caller).  Blocks with
// refcnt <= 0 are free and are never chosen; max_refcnt is
// the largest refcnt of the pool; equal scores go to the smaller block id.
//
// GB300 design: one thread-block cluster (up to 16 CTAs of 512 threads) owns
// the whole pool; each CTA copies its slice of reference counts and ages into
// shared memory with 16-byte cp.async (all copies in flight at once) and keeps
// its 32-bit order keys there, so the pool is read from HBM once.  The k-th
// largest key is found by a four-pass MSB radix select (8-bit digits): every
// CTA counts its slice into a local histogram (warp-aggregated shared-memory
// atomics), then adds its nonzero bins into every CTA's merged histogram with
// red.shared::cluster through distributed shared memory; after one cluster
// barrier each CTA scans the merged counts in its own shared memory and picks
// the same digit.  The chosen ids are placed in ascending block-id order by a
// CTA scan plus one more exchange of per-CTA counts.  Data only ever moves by
// pushes into peers before a barrier, so no CTA reads a peer after the last
// barrier and CTAs leave independently.  No global atomics, no second launch,
// no spin-waits (the barriers are the hardware's; a cluster's CTAs are resident
// together); a one-CTA cluster uses plain CTA barriers.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pkv_host.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

// Block shape and cluster sizing; the defaults are the measured best on GB300.
#ifndef PKV_EVICT_THREADS
#define PKV_EVICT_THREADS 512
#endif
#ifndef PKV_EVICT_SLICE
#define PKV_EVICT_SLICE 2048
#endif
constexpr int kEvThreads = PKV_EVICT_THREADS;
constexpr int kEvWarps = kEvThreads / 32;
constexpr int kEvBins = 256;          // 8-bit digits: four passes from the top byte
constexpr int kEvMaxCluster = 16;
constexpr int kEvMaxSlice = 49152;    // keys per CTA in shared memory (192 KiB)
constexpr int kEvStageSlice = 16384;  // slices up to this also stage the ages (12 B per block)
constexpr int kEvTargetSlice = PKV_EVICT_SLICE;  // keys per CTA that sets the cluster size
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
    int slice;   // blocks per CTA, a multiple of 4
    int k;
    int staged;  // 1: refcnt and last_used are copied to shared memory with
                 // 16-byte cp.async (16-byte aligned inputs, slice <= kEvStageSlice)
};

// Order-preserving map of a (non-NaN) fp32 score to a uint32; -0 maps with
// +0.  The result is never 0, which marks blocks that are not candidates.
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Barrier over the CTAs that exchange data: the whole cluster (release /
// acquire, so shared-memory writes into peers before it are visible after
// it), or just this CTA when the cluster has one.
__device__ __forceinline__ void group_sync(uint32_t csize)
{
    if (csize > 1)
        ptx::cluster_sync();
    else
        __syncthreads();
}

// Exclusive scan, over the first 256 threads (8 warps), of one value each,
// top bin first; the others pass 0.  *total gets the sum.  part: 8 words.
__device__ __forceinline__ uint32_t bins_exclusive_scan(uint32_t v, uint32_t *part,
                                                        uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += n;
    }
    if (lane == 31 && warp < kEvBins / 32) part[warp] = x;
    __syncthreads();
    uint32_t before = 0, sum = 0;
#pragma unroll
    for (int w = 0; w < kEvBins / 32; ++w) {
        const uint32_t pw = part[w];
        before += w < warp ? pw : 0u;
        sum += pw;
    }
    *total = sum;
    return before + x - v;
}

// Built with PKV_DEBUG: the slice this CTA stages must fit its dynamic shared
// memory, the cluster must fit the per-CTA peer arrays, and every 16-byte
// copy destination must lie inside the slice buffers; a failed check sets a
// bit in g_ev_debug_flags (read by pkv_debug_evict_flags) and the CTA takes
// an empty slice / skips the copy instead.  Release builds compile it away.
#ifdef PKV_DEBUG
__device__ unsigned int g_ev_debug_flags;
__device__ __forceinline__ bool ev_dbg_ok(bool ok, unsigned bit)
{
    if (!ok) atomicOr(&g_ev_debug_flags, bit);
    return ok;
}
__device__ __forceinline__ uint32_t ev_dyn_smem_size()
{
    uint32_t r;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}
#define PKV_EV_CHECK(cond, bit) ev_dbg_ok((cond), (bit))
#else
#define PKV_EV_CHECK(cond, bit) true
#endif

__global__ void __launch_bounds__(kEvThreads, 1) evict_kernel(EvictParams p)
{
    extern __shared__ __align__(16) unsigned char ev_smem[];
    uint32_t *keys = reinterpret_cast<uint32_t *>(ev_smem);  // this CTA's slice
    long long *ages = reinterpret_cast<long long *>(ev_smem + 4 * p.slice);  // when staged
    __shared__ uint32_t warp_hist[kEvWarps][kEvBins];  // each warp's counts of one pass
    __shared__ uint32_t merged[2][kEvBins];      // the cluster's counts, alternate passes
    __shared__ uint32_t peer_ref[kEvMaxCluster][2];  // every CTA's max refcnt, candidates
    __shared__ uint32_t peer_sel[kEvMaxCluster];     // every CTA's (eq << 16 | gt) counts
    __shared__ uint32_t warp_a[kEvWarps], warp_b[kEvWarps];
    __shared__ uint32_t part[kEvBins / 32];
    __shared__ uint32_t bcast[2];

    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const uint32_t rank = ptx::cluster_ctarank(), csize = ptx::cluster_nctarank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lo = static_cast<int64_t>(rank) * p.slice;
    const int64_t left = static_cast<int64_t>(p.num_blocks) - lo;
    int n_local = static_cast<int>(left < 0 ? 0 : (left < p.slice ? left : p.slice));
#ifdef PKV_DEBUG
    // the slice buffers (keys; ages when staged) inside the dynamic shared
    // memory, the cluster within the peer arrays
    if (!PKV_EV_CHECK(static_cast<uint64_t>(p.slice) * (p.staged ? 12u : 4u) <= ev_dyn_smem_size(), 1u) ||
        !PKV_EV_CHECK(csize <= static_cast<uint32_t>(kEvMaxCluster) && rank < csize, 2u))
        n_local = 0;
#endif
    const long long *last_used = reinterpret_cast<const long long *>(p.last_used) + lo;
    for (int b = tid; b < kEvWarps * kEvBins; b += kEvThreads) (&warp_hist[0][0])[b] = 0;
    if (tid < kEvBins) {
        merged[0][tid] = 0;  // peers add into it only after the first group barrier
        merged[1][tid] = 0;
    }

    // 1. reference counts (max and candidates over the pool).  Staged: both
    // input slices are copied to shared memory at once (all copies in
    // flight together), so the ages cost no second round trip to DRAM.
    const int32_t *refcnt = p.refcnt + lo;
    if (p.staged) {
        const int nr = n_local >> 2, na = n_local >> 1;  // 16-byte chunks
        for (int c = tid; c < nr; c += kEvThreads)
            if (PKV_EV_CHECK(4 * c + 4 <= p.slice, 4u))
                ptx::cp_async_16(ptx::smem_addr(keys + 4 * c), refcnt + 4 * c);
        for (int c = tid; c < na; c += kEvThreads)
            if (PKV_EV_CHECK(2 * c + 2 <= p.slice, 4u))
                ptx::cp_async_16(ptx::smem_addr(ages + 2 * c), last_used + 2 * c);
        if (tid == 0) {
            for (int j = 4 * nr; j < n_local; ++j) keys[j] = static_cast<uint32_t>(__ldg(refcnt + j));
            for (int j = 2 * na; j < n_local; ++j) ages[j] = __ldg(last_used + j);
        }
        ptx::cp_async_wait_all();
    } else {
#pragma unroll 4
        for (int j = tid; j < n_local; j += kEvThreads) keys[j] = static_cast<uint32_t>(__ldg(refcnt + j));
    }
    __syncthreads();
    int32_t rmax = 0;
    uint32_t cand = 0;
    for (int j = tid; j < n_local; j += kEvThreads) {
        const int32_t r = static_cast<int32_t>(keys[j]);
        rmax = max(rmax, r);
        cand += r > 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        rmax = max(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
        cand += __shfl_xor_sync(0xffffffffu, cand, o);
    }
    if (lane == 0) {
        warp_a[warp] = static_cast<uint32_t>(rmax);
        warp_b[warp] = cand;
    }
    __syncthreads();
    if (warp == 0) {
        int32_t m = lane < kEvWarps ? static_cast<int32_t>(warp_a[lane]) : 0;
        uint32_t c = lane < kEvWarps ? warp_b[lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            c += __shfl_xor_sync(0xffffffffu, c, o);
        }
        // push this CTA's figures into slot `rank` of every CTA of the cluster
        if (static_cast<uint32_t>(lane) < csize) {
            ptx::st_cluster_addr(ptx::map_cluster(ptx::smem_addr(&peer_ref[rank][0]), lane),
                                 static_cast<uint32_t>(m));
            ptx::st_cluster_addr(ptx::map_cluster(ptx::smem_addr(&peer_ref[rank][1]), lane), c);
        }
    }
    group_sync(csize);
    int32_t max_ref = 0;
    uint32_t n_cand = 0;
    for (uint32_t c = 0; c < csize; ++c) {
        max_ref = max(max_ref, static_cast<int32_t>(peer_ref[c][0]));
        n_cand += peer_ref[c][1];
    }

    // 2. scores (written out) and order keys (kept in shared memory)
#pragma unroll 4
    for (int j = tid; j < n_local; j += kEvThreads) {
        const long long used = p.staged ? ages[j] : __ldg(last_used + j);
        const int32_t r = static_cast<int32_t>(keys[j]);
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
        // MSB radix select of the k-th largest key, one byte per pass.  Each
        // CTA counts its slice locally, then adds its nonzero bins into the
        // merged histogram of every CTA of the cluster; one group barrier,
        // and every CTA holds the cluster's counts in its own shared memory.
        uint32_t prefix = 0, mask = 0;
        kk = k;
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int j0 = 0; j0 < n_local; j0 += kEvThreads) {
                const int j = j0 + tid;
                uint32_t bin = kNoBin;
                if (j < n_local) {
                    const uint32_t key = keys[j];
                    if (key != 0 && (key & mask) == prefix) bin = (key >> shift) & 0xffu;
                }
                const uint32_t peers = __match_any_sync(0xffffffffu, bin);
                if (bin != kNoBin && lane == __ffs(peers) - 1)
                    warp_hist[warp][bin] += __popc(peers);  // this warp's own row
            }
            __syncthreads();
            uint32_t *m = merged[pass & 1];
            if (tid < kEvBins) {
                uint32_t v = 0;
#pragma unroll
                for (int w = 0; w < kEvWarps; ++w) {
                    v += warp_hist[w][tid];
                    warp_hist[w][tid] = 0;
                }
                if (v) {
                    const uint32_t addr = ptx::smem_addr(&m[tid]);
                    for (uint32_t c = 0; c < csize; ++c)
                        ptx::red_add_cluster(ptx::map_cluster(addr, c), v);
                }
                // the other buffer was read in the previous pass (before the
                // barrier below, in every CTA): clear it for the next pass
                merged[(pass + 1) & 1][tid] = 0;
            }
            group_sync(csize);
            const uint32_t cnt = tid < kEvBins ? m[kEvBins - 1 - tid] : 0u;  // top bin first
            uint32_t total;
            const uint32_t above = bins_exclusive_scan(cnt, part, &total);
            if (tid < kEvBins && above < kk && kk <= above + cnt) {
                bcast[0] = kEvBins - 1 - tid;
                bcast[1] = above;  // keys in higher bins
            }
            __syncthreads();
            prefix |= bcast[0] << shift;
            mask |= 0xffu << shift;
            kk -= bcast[1];
        }
        thresh = prefix;
    }

    // 4. place the chosen ids in ascending block-id order.  Each warp owns a
    // contiguous segment of the slice and walks it in 32-key chunks (lane l
    // reads key base + l: no bank conflicts); ballots give each key's rank.
    const int seg = ((n_local + kEvWarps * 32 - 1) / (kEvWarps * 32)) * 32;
    const int s0 = min(warp * seg, n_local), s1 = min(s0 + seg, n_local);
    uint32_t gt = 0, eq = 0;  // warp-uniform counts over the segment
    for (int base = s0; base < s1; base += 32) {
        const int j = base + lane;
        const uint32_t key = j < s1 ? keys[j] : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, j < s1 && key > thresh));
        eq += __popc(__ballot_sync(0xffffffffu, j < s1 && key == thresh));
    }
    if (lane == 0) {
        warp_a[warp] = gt;
        warp_b[warp] = eq;
    }
    __syncthreads();
    uint32_t gt_b = 0, eq_b = 0, cta_gt = 0, cta_eq = 0;
    for (int w = 0; w < kEvWarps; ++w) {
        gt_b += w < warp ? warp_a[w] : 0u;
        eq_b += w < warp ? warp_b[w] : 0u;
        cta_gt += warp_a[w];
        cta_eq += warp_b[w];
    }
    if (tid < static_cast<int>(csize))
        ptx::st_cluster_addr(ptx::map_cluster(ptx::smem_addr(&peer_sel[rank]), tid),
                             cta_gt | (cta_eq << 16));
    // after this barrier no CTA touches another's shared memory: CTAs may
    // leave in any order
    group_sync(csize);
    for (uint32_t c = 0; c < rank; ++c) {
        gt_b += peer_sel[c] & 0xffffu;
        eq_b += peer_sel[c] >> 16;
    }
    const uint32_t below = (1u << lane) - 1u;  // lanes before this one
    for (int base = s0; base < s1; base += 32) {
        const int j = base + lane;
        const uint32_t key = j < s1 ? keys[j] : 0u;
        const uint32_t gm = __ballot_sync(0xffffffffu, j < s1 && key > thresh);
        const uint32_t em = __ballot_sync(0xffffffffu, j < s1 && key == thresh);
        const uint32_t g = gt_b + __popc(gm & below), e = eq_b + __popc(em & below);
        // an output slot is below k by construction; the checks keep every
        // store inside the caller's k-entry buffer regardless
        if (j < s1 && key > thresh) {
            const uint32_t at = g + min(e, kk);
            if (at < k) p.ids[at] = static_cast<int32_t>(lo + j);
        } else if (j < s1 && key == thresh && e < kk && g + e < k) {
            p.ids[g + e] = static_cast<int32_t>(lo + j);
        }
        gt_b += __popc(gm);
        eq_b += __popc(em);
    }

    // 5. the count, and -1 in the unused tail of the id buffer
    const uint32_t n_sel = k < n_cand ? k : n_cand;
    if (rank == 0 && tid == 0) *p.num_evicted = static_cast<int32_t>(n_sel);
    for (int64_t i = n_sel + static_cast<int64_t>(rank) * kEvThreads + tid; i < p.k;
         i += static_cast<int64_t>(csize) * kEvThreads)
        p.ids[i] = -1;
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
    int64_t slice = (static_cast<int64_t>(num_blocks) + csize - 1) / csize;
    slice = (slice + 3) & ~static_cast<int64_t>(3);
    if (slice > kEvMaxSlice) return PKV_ERR_UNSUPPORTED;
    const bool staged = num_blocks > 0 && slice <= kEvStageSlice && aligned(refcnt, 16) &&
                        aligned(last_used, 16);
    const size_t smem = static_cast<size_t>(slice > 0 ? slice : 4) * (staged ? 12 : 4);
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
    prm.staged = staged ? 1 : 0;
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

#ifdef PKV_DEBUG
// Debug builds only (not part of the C ABI header): the eviction kernel's
// check bits set since the last reset (1: slice larger than the dynamic
// shared memory, 2: cluster larger than the peer arrays, 4: a copy outside
// the slice); reset nonzero clears them.  Synchronises with the device.
extern "C" __attribute__((visibility("default"))) unsigned int pkv_debug_evict_flags(int reset)
{
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, pkv::g_ev_debug_flags, sizeof(v)) != cudaSuccess)
        return 0xffffffffu;
    if (reset) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(pkv::g_ev_debug_flags, &z, sizeof(z)) != cudaSuccess) return 0xffffffffu;
    }
    return v;
}
#endif

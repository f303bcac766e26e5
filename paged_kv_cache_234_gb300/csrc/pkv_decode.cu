// pkv_decode.cu -- decode-step paged attention over a block-table-indexed KV
// cache, fp16 or INT8 KV, for sm_103a.
//
// What is computed (PagedKV-Fusion README, "Architecture": online softmax,
// GQA, per-(block, head) INT8; paged-attention-runtime summary, CORE
// CAPABILITIES 2: block-table indirection, online single-pass softmax, FP32
// accumulation; "PagedAttention & KV-Cache Memory Management" section 2.1:
// block = table[t / 16], slot = t % 16):
//   out[s][h] = sum_t softmax_t(scale * <q[s][h], K_t>) V_t,  t < ctx[s],
// with query head h reading kv head h / (Hq / Hkv).
//
// Work decomposition.  A work item is (sequence, kv head, up to 8 query heads
// of that kv head, or up to 16 as two groups of 8 when the kv head has more
// than 8); its pages are the sequence's 16-token blocks.  All items' pages
// form one stream of T pages, and every warp of a persistent grid (one worker
// per resident warp -- seven per SM for fp16 at head_dim 128, ten at 64 --
// and no more than the larger of four per item and one per eight pages)
// streams one contiguous, equal share of it, so every SM moves the same
// number of bytes whatever the mix of context lengths.  A worker's share is a
// run of "pieces": at most one partial item at each end and whole items in
// between.  Whole items are finished in place; a partial piece leaves
// (running max, running sum, unnormalised accumulator) in the workspace, and
// a split-context reduce kernel, launched as a programmatic dependent of the
// decode grid, merges the pieces of every split item (a warp per item and
// query head, or, for items cut into many pieces, several CTAs each).
// Small batches run one item per thread-block cluster instead, merged in
// distributed shared memory.
//
// Per worker (warp), pages flow through a private ring of S shared-memory
// stages of one or two pages each.  Lane 0 issues TMA tile loads (16 rows x
// head_dim, 128- or 64-byte swizzled) for the K and V tiles of the stage's
// pages, plus 4-byte cp.async copies of the INT8 scales, all completing on
// the stage's mbarrier; the ring keeps the next stages in flight while the
// warp computes on the oldest one.
//
// Per page, the item's query heads share one read of K and V, per group of 8:
//   S^T[16 tok][8 heads] = K_page[16 x d] . Q^T      (m16n8k16, f16 -> f32)
//   online softmax in base 2, one update per stage
//   O^T[d][8 heads]     += V_page^T[d x 16] . P^T    (m16n8k16, f16 -> f32)
// (with two groups, each K and V fragment is loaded and widened once and
// enters both groups' mma).
// FP8 (OCP E4M3) codes are widened to f16 exactly by cvt.rn.f16x2.e4m3x2; the
// K and V scales apply as for INT8.
// INT8 codes are widened to f16 exactly by byte permutes: a code c placed
// under the exponent byte 0x64 reads as 1152 + c.  For K the constant 1152
// is left in and removed from the scores as 1152 * sum(q); for V it is
// subtracted before the product.  The K scale multiplies the scores.  The V
// scale enters as a ratio to the piece's largest V scale so far (<= 1, the
// accumulators move to a new reference with the softmax rescale), and the
// reference multiplies the accumulators when they leave the registers, so
// the result does not depend on the magnitude of V.
//
// The probabilities (times 2^15, times the V scale ratio) reach the PV mma as
// fp32 values: an f16 high part plus an f16 low part (the next 11 bits),
// either in the spare mma columns (groups of up to four query heads) or as a
// second mma into the same accumulators.  So P is not rounded to f16
// precision, and differently split batches agree to float rounding.
#include <cuda_fp16.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "pkv_host.cuh"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 4;  // workers per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kPage = 16;              // tokens per block
constexpr int kItemHeads = 8;          // query heads per group (mma N); an item has 1 or 2
constexpr int kMaxWorkers = 4096;      // workspace is sized for at most this many
constexpr int kMaxWorkersPerItem = 4;  // measured on GB300: 8 x 512, 32 x 1024 and Qwen2-
                                       // shape batches run 10-30 % faster than with one
                                       // worker per resident warp
constexpr int kMaxSeqs = 8192;         // per-sequence tables live in shared memory
constexpr int kMaxCluster = 8;         // CTAs per cluster in the one-item-per-cluster mode
constexpr int kMaxClusterStages = 2;   // the cluster mode only while a warp has at most this
                                       // many stages of its item at the largest cluster
constexpr int kMinPagesPerWorker = 8;  // persistent workers: at least this many pages each
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s
constexpr float kPScale = 32768.f;     // probabilities enter PV as 2^15 p (see the main loop)
constexpr float kPScaleInv = 1.f / 32768.f;

int g_worker_cap = 0;  // pkv_set_decode_workers
std::mutex g_cfg_mu;

struct DecodeArgs {
    float *out;
    const __half *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const float *k_scales;
    const float *v_scales;
    float *partials;     // [num_workers * 2][rec_heads][head_dim + 4]: m, l, 0, -, acc
    int32_t *dev_status;
    int num_seqs, num_heads, num_kv_heads;
    int group;           // query heads per kv head
    int item_heads;      // query heads per work item: 8, or 16 when group > 8
    int qgroups;         // ceil(group / item_heads)
    int items_per_seq;   // num_kv_heads * qgroups
    int rec_heads;       // min(item_heads, group): heads per partial record
    int max_blocks_per_seq;
    int num_blocks;
    int ctx_cap;         // largest valid context length
    int num_workers;
    int clust;           // 0: persistent workers; else one item per cluster of this many CTAs
    float scale_log2;    // softmax_scale * log2(e)
};

// ------------------------------------------------------ debug build checks
// Built with PKV_DEBUG, the decode kernel checks every shared-memory address
// it forms (range inside the CTA's dynamic shared memory, alignment of the
// access) and every index into its per-sequence tables and the block tables.
// A failed check sets a bit in g_debug_flags (read by pkv_debug_flags) and the
// access is redirected to the start of the buffer or to index 0, so nothing
// outside the buffers is touched.  Release builds compile the checks away.
#ifdef PKV_DEBUG
__device__ unsigned int g_debug_flags;
constexpr unsigned kDbgSmemRange = 1u, kDbgSmemAlign = 2u, kDbgIndex = 4u;

__device__ __forceinline__ uint32_t dbg_smem(uint32_t addr, uint32_t bytes, uint32_t align)
{
    extern __shared__ __align__(16) uint8_t dbg_dyn_smem[];
    const uint32_t lo = static_cast<uint32_t>(__cvta_generic_to_shared(dbg_dyn_smem));
    uint32_t size;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
    unsigned bad = 0;
    if (addr < lo || addr + bytes > lo + size) bad |= kDbgSmemRange;
    if (addr & (align - 1)) bad |= kDbgSmemAlign;
    if (!bad) return addr;
    atomicOr(&g_debug_flags, bad);
    return (lo + align - 1) & ~(align - 1);
}

__device__ __forceinline__ int64_t dbg_index(int64_t i, int64_t n)
{
    if (i >= 0 && i < n) return i;
    atomicOr(&g_debug_flags, kDbgIndex);
    return 0;
}
// Limit of the main loop's waits for a stage (the drain after a timeout keeps
// kWaitLimitNs).  Settable through pkv_debug_set_stage_wait_ns so that a test
// can make a wait run out on a copy that does land: 0 means a wait that gives
// up at once, as if its limit had run out.
__device__ unsigned long long g_debug_stage_wait_ns = kWaitLimitNs;
#define PKV_STAGE_WAIT_NS g_debug_stage_wait_ns
#define PKV_SMEM(addr, bytes, align) dbg_smem((addr), (bytes), (align))
// a shared-memory record reached through a generic pointer (one item per
// cluster): its range inside the CTA's dynamic shared memory
#define PKV_REC(ptr, bytes)                                                              \
    reinterpret_cast<float *>(__cvta_shared_to_generic(                                  \
        dbg_smem(static_cast<uint32_t>(__cvta_generic_to_shared(ptr)), (bytes), 16)))
#define PKV_IDX(i, n) dbg_index((i), (n))
#define PKV_TABLE_AT(p, seq, page, u, mb) \
    ((p).block_tables + dbg_index((seq), (p).num_seqs) * (mb) + dbg_index((page) + (u), (mb)))
#else
#define PKV_STAGE_WAIT_NS kWaitLimitNs
#define PKV_SMEM(addr, bytes, align) (addr)
#define PKV_REC(ptr, bytes) (ptr)
#define PKV_IDX(i, n) (i)
#define PKV_TABLE_AT(p, seq, page, u, mb) ((p).block_tables + (seq) * (mb) + (page) + (u))
#endif

// Pipeline shape per variant: pages per stage, stages per warp, CTAs (of
// four warps) per SM.  Shared memory per CTA is 4 * stages * pages * (K + V
// tile) bytes; the register budget follows from the CTA count.
#ifndef PKV_F16_D128_PPS
#define PKV_F16_D128_PPS 1
#endif
#ifndef PKV_F16_D128_STAGES
#define PKV_F16_D128_STAGES 2
#endif
#ifndef PKV_F16_D128_CTAS
#define PKV_F16_D128_CTAS 3
#endif
#ifndef PKV_I8_D128_PPS
#define PKV_I8_D128_PPS 2
#endif
#ifndef PKV_I8_D128_STAGES
#define PKV_I8_D128_STAGES 2
#endif
#ifndef PKV_I8_D128_CTAS
#define PKV_I8_D128_CTAS 3
#endif
// fp16 d128: workers per SM (0: every resident warp).  Measured on GB300: the
// fp16 kernel moves its pages faster with ~7 streaming warps per SM than with
// all 12 (64 x 2048: 93.6 against 101.4 us per call; 256 ragged sequences:
// 322.7 against 339.8 us), while the INT8 and FP8 kernels need every warp.
#ifndef PKV_F16_D128_WARPS_PER_SM
#define PKV_F16_D128_WARPS_PER_SM 7
#endif
// fp16 d64: the same with 16 resident warps; measured on GB300 with 512 x 2048
// in the Qwen2-0.5B shape (14 / 2 heads) and 128 x 2048 with 32 / 8 heads:
// 92.0 and 87.3 us per call at 10 streaming warps per SM against 96.0 and
// 91.2 us with all 16 (12: 94.7 / 90.1 us; 8: 99.8 / 91.9 us).
#ifndef PKV_F16_D64_WARPS_PER_SM
#define PKV_F16_D64_WARPS_PER_SM 10
#endif

template <int kPPS_, int kStages_, int kMinCtas_>
struct Tune {
    static constexpr int kPPS = kPPS_;
    static constexpr int kStages = kStages_;
    static constexpr int kMinCtas = kMinCtas_;
};

// KV kinds: 0 fp16 values; 1 INT8 codes, 2 FP8 (E4M3) codes, both one byte
// per value with an fp32 K and V scale per (block, kv head).
constexpr int kKvF16 = 0, kKvI8 = 1, kKvF8 = 2;

template <int kKv, int kD>
struct TuneOf;
template <>
struct TuneOf<kKvF16, 128> : Tune<PKV_F16_D128_PPS, PKV_F16_D128_STAGES, PKV_F16_D128_CTAS> {};
template <>
struct TuneOf<kKvI8, 128> : Tune<PKV_I8_D128_PPS, PKV_I8_D128_STAGES, PKV_I8_D128_CTAS> {};
template <>
struct TuneOf<kKvF8, 128> : Tune<PKV_I8_D128_PPS, PKV_I8_D128_STAGES, PKV_I8_D128_CTAS> {};
template <>
struct TuneOf<kKvF16, 64> : Tune<1, 3, 4> {};
template <>
struct TuneOf<kKvI8, 64> : Tune<2, 3, 4> {};
template <>
struct TuneOf<kKvF8, 64> : Tune<2, 3, 4> {};

template <int kKv, int kD>
struct Cfg {
    static constexpr bool kInt8 = kKv != kKvF16;  // one-byte codes with scales
    static constexpr int kElem = kInt8 ? 1 : 2;
    static constexpr int kRowBytes = kD * kElem;                 // 256 / 128 / 64
    static constexpr int kTileBytes = kPage * kRowBytes;         // one (block, kv head) tile
    static constexpr int kPageBytes = 2 * kTileBytes;            // K tile + V tile
    static constexpr int kPPS = TuneOf<kKv, kD>::kPPS;           // pages per stage
    static constexpr int kStageBytes = kPPS * kPageBytes;
    static constexpr int kBoxInner = kRowBytes > 128 ? 128 / kElem : kD;  // elements
    static constexpr int kBoxes = kD / kBoxInner;
    static constexpr int kBoxBytes = kPage * kBoxInner * kElem;
    static constexpr int kSwizzle = kRowBytes >= 128 ? 128 : 64;
    static constexpr int kStages = TuneOf<kKv, kD>::kStages;
    static constexpr int kMinCtas = TuneOf<kKv, kD>::kMinCtas;
    static constexpr int kWarpsPerSm =
        kKv != kKvF16 ? 0 : kD == 128 ? PKV_F16_D128_WARPS_PER_SM : PKV_F16_D64_WARPS_PER_SM;
    static_assert(kPPS == 1 || kPPS == 2, "one or two pages per stage");
    static constexpr int kHdrBytes = 32;  // per stage: bad[2], k scale[2], v scale[2]
    static constexpr int kStageRegion = kWarps * kStages * kStageBytes;
    static constexpr int kHdrOffset = kStageRegion;
    static constexpr int kBarOffset = kHdrOffset + kWarps * kStages * kHdrBytes;
    static constexpr int kTabOffset = kBarOffset + kWarps * kStages * 8;
    static size_t smem_bytes(int num_seqs)
    {
        return 1024 + kTabOffset + static_cast<size_t>(2 * num_seqs + 1) * sizeof(int32_t);
    }
    // One item per cluster: the records pushed to this CTA, after the tables.
    __host__ __device__ static size_t crec_offset(int num_seqs)
    {
        return (kTabOffset + static_cast<size_t>(2 * num_seqs + 1) * sizeof(int32_t) + 15) & ~size_t(15);
    }
    static size_t crec_bytes(int warps, int heads_per_cta)
    {
        return static_cast<size_t>(warps) * heads_per_cta * (kD + 4) * sizeof(float);
    }
};

// Byte offset of 16-byte chunk `ch` of row `t` inside a TMA-written tile.
// Rows wider than 128 bytes arrive as 128-byte-wide boxes of 16 rows each.
template <int kRowBytes>
__device__ __forceinline__ uint32_t swz(int t, int ch)
{
    if constexpr (kRowBytes == 256) {
        return ((ch >> 3) << 11) + (t << 7) + (((ch & 7) ^ (t & 7)) << 4);
    } else if constexpr (kRowBytes == 128) {
        return (t << 7) + (((ch) ^ (t & 7)) << 4);
    } else {
        return (t << 6) + (((ch) ^ ((t >> 1) & 3)) << 4);
    }
}

// ------------------------------------------------------ per-sequence tables
// ctxs[s]   = context length, or -1 if it is outside [0, ctx_cap]
// prefix[s] = pages of all sequences before s (exclusive prefix sum)
// Computed by a CTA of kNT threads from context_lens alone.
template <int kNT = kThreads>
__device__ void build_page_tables(const DecodeArgs &p, int32_t *prefix, int32_t *ctxs)
{
    constexpr int kNW = kNT / 32;
    __shared__ int32_t warp_sums[kNW];
    __shared__ int32_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        prefix[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += kNT) {
        const int s = base + threadIdx.x;
        int np = 0;
        if (s < p.num_seqs) {
            const int c = p.context_lens[s];
            const bool ok = c >= 0 && c <= p.ctx_cap;
            ctxs[s] = ok ? c : -1;
            np = ok ? (c + kPage - 1) / kPage : 0;
        }
        int v = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) warp_sums[warp] = v;
        __syncthreads();
        int before = carry;
        for (int j = 0; j < warp; ++j) before += warp_sums[j];
        const int incl = before + v;
        if (s < p.num_seqs) prefix[s + 1] = incl;
        __syncthreads();
        if (threadIdx.x == kNT - 1) carry = incl;
        __syncthreads();
    }
}

// floor(x * k / d) for x, k >= 0 and d > 0; a 32-bit division when the
// operands fit (the usual case), else a 64-bit one.
__device__ __forceinline__ int64_t muldiv(int64_t x, int64_t k, int64_t d)
{
    const uint64_t num = static_cast<uint64_t>(x) * static_cast<uint64_t>(k);
    if (num <= 0xffffffffull && static_cast<uint64_t>(d) <= 0xffffffffull)
        return static_cast<uint32_t>(num) / static_cast<uint32_t>(d);
    return static_cast<int64_t>(num / static_cast<uint64_t>(d));
}

// Position of one page in the stream of all items' pages.
struct PageCursor {
    int seq;     // sequence
    int item;    // kv head * qgroups + query-head group
    int kvh;     // kv head of the item
    int qg;      // query-head group of the item (8 heads each)
    int page;    // page (16-token block) within the sequence
    int npages;  // pages of the sequence

    // All 32 lanes of a warp, with the same x.  The sequence is the largest s
    // with items_per_seq * prefix[s] <= x (prefix is nondecreasing, so the
    // s that pass form a run from 0): each round tests 32 evenly spaced
    // candidates of the remaining range with one ballot and keeps the span
    // after the last one that passes, down to 32 candidates, then counts.
    // The item within the sequence is counted the same way when a sequence
    // has at most 32 items.
    __device__ void seek(const DecodeArgs &p, const int32_t *prefix, int64_t x, int lane)
    {
        const int64_t ips = p.items_per_seq;
        int lo = 0, span = p.num_seqs;  // prefix[lo] * ips <= x throughout
        while (span > 32) {
            const int step = (span + 31) >> 5;
            const int sc = lo + lane * step;
            const bool le = lane * step < span &&
                            ips * prefix[PKV_IDX(sc, p.num_seqs + 1)] <= x;
            const int c = __popc(__ballot_sync(0xffffffffu, le));
            lo += (c - 1) * step;
            span = min(step, span - (c - 1) * step);
        }
        {
            const bool le = lane < span && ips * prefix[PKV_IDX(lo + lane, p.num_seqs + 1)] <= x;
            seq = lo + __popc(__ballot_sync(0xffffffffu, le)) - 1;
        }
        npages = prefix[PKV_IDX(seq + 1, p.num_seqs + 1)] - prefix[seq];
        const int64_t r = x - ips * prefix[seq];
        if (ips <= 32) {
            const bool le = lane < ips && static_cast<int64_t>(lane) * npages <= r;
            item = __popc(__ballot_sync(0xffffffffu, le)) - 1;
            page = static_cast<int>(r - static_cast<int64_t>(item) * npages);
        } else if (r <= 0xffffffffll) {
            const uint32_t r32 = static_cast<uint32_t>(r);
            item = static_cast<int>(r32 / static_cast<uint32_t>(npages));
            page = static_cast<int>(r32 - static_cast<uint32_t>(item) * static_cast<uint32_t>(npages));
        } else {
            item = static_cast<int>(r / npages);
            page = static_cast<int>(r % npages);
        }
        if (p.qgroups == 1) {
            kvh = item;
            qg = 0;
        } else {
            kvh = item / p.qgroups;
            qg = item - kvh * p.qgroups;
        }
    }

    // pages of the next stage: up to pps, never past the item's end or `left`
    __device__ __forceinline__ int unit(int pps, int left) const
    {
        int u = npages - page;
        u = u < pps ? u : pps;
        return u < left ? u : left;
    }

    __device__ void advance(const DecodeArgs &p, const int32_t *prefix, int k)
    {
        page += k;
        if (page < npages) return;
        page = 0;
        if (++qg == p.qgroups) {
            qg = 0;
            ++kvh;
        }
        if (++item < p.items_per_seq) return;
        item = kvh = qg = 0;
        do {
            ++seq;
        } while (seq < p.num_seqs && prefix[seq + 1] == prefix[seq]);
        npages = seq < p.num_seqs ? prefix[seq + 1] - prefix[seq] : 0;
    }
};

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_half2(uint32_t w)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

// two int8 codes (bytes picked by sel from a word already XOR-ed with 0x80)
// as an f16 pair 1152 + c, exact
__device__ __forceinline__ uint32_t i8pair_biased(uint32_t xw, uint32_t sel)
{
    return ptx::prmt(xw, 0x64646464u, sel);
}

// the same pair with the bias removed: exactly c
__device__ __forceinline__ uint32_t i8pair_exact(uint32_t xw, uint32_t sel)
{
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(i8pair_biased(xw, sel)), "r"(0x64806480u));
    return r;
}

// Which worker's page range holds stream page x (largest w with a_w <= x).
__device__ __forceinline__ int64_t worker_of(int64_t x, int64_t total, int workers)
{
    const uint64_t num = static_cast<uint64_t>(x + 1) * static_cast<uint64_t>(workers) - 1;
    if (num <= 0xffffffffull && static_cast<uint64_t>(total) <= 0xffffffffull)
        return static_cast<uint32_t>(num) / static_cast<uint32_t>(total);
    return static_cast<int64_t>(num / static_cast<uint64_t>(total));
}

// S^T fragments (rows: tokens g, g+8; cols: heads 2c, 2c+1 of each of kG
// groups of 8 query heads) of one page: every K fragment is loaded and
// widened once and multiplied with each group's query fragments.
template <int kKv, int kD, int kG>
__device__ __forceinline__ void page_scores(uint32_t kt, const uint32_t (&qf)[kG][kD / 16][2],
                                            int lane, float (&s)[kG][4])
{
    using C = Cfg<kKv, kD>;
    constexpr bool kInt8 = C::kInt8;
    constexpr int KS = kD / 16;
    float sa[kG][4], sb[kG][4];
#pragma unroll
    for (int gi = 0; gi < kG; ++gi)
#pragma unroll
        for (int i = 0; i < 4; ++i) sa[gi][i] = sb[gi][i] = 0.f;
    if constexpr (!kInt8) {
        const int lt = (lane & 7) + 8 * ((lane >> 3) & 1);
        const int lch = lane >> 4;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a0, a1, a2, a3;
            ptx::ldsm_x4(PKV_SMEM(kt + swz<C::kRowBytes>(lt, 2 * ks + lch), 16, 16), a0, a1, a2, a3);
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                if (ks & 1)
                    ptx::mma_16816(sb[gi], a0, a1, a2, a3, qf[gi][ks][0], qf[gi][ks][1]);
                else
                    ptx::mma_16816(sa[gi], a0, a1, a2, a3, qf[gi][ks][0], qf[gi][ks][1]);
            }
        }
    } else {
        // lane (g, c): rows g and g+8, bytes [DG*c, DG*c + DG), DG = kD/4; the
        // head_dim order matches the query fragments
        const int g = lane >> 2, c = lane & 3;
        constexpr int CH = kD / 64;  // 16-byte chunks per row per lane
        uint32_t kw[2][4 * CH];
        // INT8: flip the sign bit for the biased widening; FP8: as stored
        constexpr uint32_t kFlip = kKv == kKvI8 ? 0x80808080u : 0u;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                const uint4 v =
                    ptx::lds128(PKV_SMEM(kt + swz<C::kRowBytes>(g + 8 * r, CH * c + j), 16, 16));
                kw[r][4 * j + 0] = v.x ^ kFlip;
                kw[r][4 * j + 1] = v.y ^ kFlip;
                kw[r][4 * j + 2] = v.z ^ kFlip;
                kw[r][4 * j + 3] = v.w ^ kFlip;
            }
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a0, a1, a2, a3;
            if constexpr (kKv == kKvI8) {
                a0 = i8pair_biased(kw[0][ks], 0x4140u);
                a2 = i8pair_biased(kw[0][ks], 0x4342u);
                a1 = i8pair_biased(kw[1][ks], 0x4140u);
                a3 = i8pair_biased(kw[1][ks], 0x4342u);
            } else {
                a0 = ptx::e4m3x2_to_f16x2(kw[0][ks]);
                a2 = ptx::e4m3x2_to_f16x2(kw[0][ks] >> 16);
                a1 = ptx::e4m3x2_to_f16x2(kw[1][ks]);
                a3 = ptx::e4m3x2_to_f16x2(kw[1][ks] >> 16);
            }
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                if (ks & 1)
                    ptx::mma_16816(sb[gi], a0, a1, a2, a3, qf[gi][ks][0], qf[gi][ks][1]);
                else
                    ptx::mma_16816(sa[gi], a0, a1, a2, a3, qf[gi][ks][0], qf[gi][ks][1]);
            }
        }
    }
#pragma unroll
    for (int gi = 0; gi < kG; ++gi)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[gi][i] = sa[gi][i] + sb[gi][i];
}

// O^T += V_page^T . P^T for one page; tokens >= ntok contribute nothing.
// kLoCols: P^T (pb0, pb1) holds the high f16 parts of the probabilities in
// columns 0-3 and the low parts in columns 4-7, one mma per k-step.
// Otherwise P^T arrives as two f16 operands whose sum is the fp32
// probabilities (high part pb0/pb1, low part pl0/pl1) and both products go
// into the same fp32 accumulators.  Either way P is not rounded to f16
// precision.  Every V fragment is loaded and widened once and multiplied
// with each of the kG groups' probabilities.
template <int kKv, int kD, bool kLoCols, int kG>
__device__ __forceinline__ void page_pv(uint32_t vt, const uint32_t (&pb0)[kG],
                                        const uint32_t (&pb1)[kG], const uint32_t (&pl0)[kG],
                                        const uint32_t (&pl1)[kG], int ntok, int lane,
                                        float (&o)[kG][kD / 16][4])
{
    using C = Cfg<kKv, kD>;
    constexpr bool kInt8 = C::kInt8;
    constexpr int KS = kD / 16;
    const int g = lane >> 2, c = lane & 3;
    if constexpr (!kInt8) {
        const int lt = (lane & 7) + 8 * (lane >> 4);
        const int lch = (lane >> 3) & 1;
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (ntok < kPage) {  // zero V rows of tokens past the end (they may hold NaN)
            mlo = (2 * c < ntok ? 0x0000ffffu : 0u) | (2 * c + 1 < ntok ? 0xffff0000u : 0u);
            mhi = (2 * c + 8 < ntok ? 0x0000ffffu : 0u) | (2 * c + 9 < ntok ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int i = 0; i < KS; ++i) {
            uint32_t a0, a1, a2, a3;
            ptx::ldsm_x4_t(PKV_SMEM(vt + swz<C::kRowBytes>(lt, 2 * i + lch), 16, 16), a0, a1, a2, a3);
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                ptx::mma_16816(o[gi][i], a0, a1, a2, a3, pb0[gi], pb1[gi]);
                if constexpr (!kLoCols) ptx::mma_16816(o[gi][i], a0, a1, a2, a3, pl0[gi], pl1[gi]);
            }
        }
    } else {
        // lane (g, c): tokens 2c, 2c+1, 2c+8, 2c+9; bytes [DG*g, DG*g + DG), DG = kD/8
        constexpr int NW = kD / 32;  // words per token per lane
        constexpr uint32_t kFlip = kKv == kKvI8 ? 0x80808080u : 0u;
        uint32_t vw[4][NW];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 2 * c + (r & 1) + 8 * (r >> 1);
            if constexpr (kD == 128) {
                const uint4 v = ptx::lds128(PKV_SMEM(vt + swz<C::kRowBytes>(t, g), 16, 16));
                vw[r][0] = v.x ^ kFlip;
                vw[r][1] = v.y ^ kFlip;
                vw[r][2] = v.z ^ kFlip;
                vw[r][3] = v.w ^ kFlip;
            } else {
                const uint2 v =
                    ptx::lds64(PKV_SMEM(vt + swz<C::kRowBytes>(t, g >> 1) + (g & 1) * 8, 8, 8));
                vw[r][0] = v.x ^ kFlip;
                vw[r][1] = v.y ^ kFlip;
            }
        }
        // FP8: rows of tokens past the end are zeroed (a NaN byte there
        // would survive a zero probability); INT8 codes are always finite
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (kKv == kKvF8 && ntok < kPage) {
            mlo = (2 * c < ntok ? 0x0000ffffu : 0u) | (2 * c + 1 < ntok ? 0xffff0000u : 0u);
            mhi = (2 * c + 8 < ntok ? 0x0000ffffu : 0u) | (2 * c + 9 < ntok ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int i = 0; i < KS; ++i) {
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
            const uint32_t il01 = ptx::prmt(vw[0][i >> 1], vw[1][i >> 1], sel);
            const uint32_t il23 = ptx::prmt(vw[2][i >> 1], vw[3][i >> 1], sel);
            uint32_t a0, a1, a2, a3;
            if constexpr (kKv == kKvI8) {
                a0 = i8pair_exact(il01, 0x4140u);
                a1 = i8pair_exact(il01, 0x4342u);
                a2 = i8pair_exact(il23, 0x4140u);
                a3 = i8pair_exact(il23, 0x4342u);
            } else {
                a0 = ptx::e4m3x2_to_f16x2(il01) & mlo;
                a1 = ptx::e4m3x2_to_f16x2(il01 >> 16) & mlo;
                a2 = ptx::e4m3x2_to_f16x2(il23) & mhi;
                a3 = ptx::e4m3x2_to_f16x2(il23 >> 16) & mhi;
            }
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                ptx::mma_16816(o[gi][i], a0, a1, a2, a3, pb0[gi], pb1[gi]);
                if constexpr (!kLoCols) ptx::mma_16816(o[gi][i], a0, a1, a2, a3, pl0[gi], pl1[gi]);
            }
        }
    }
}

// kLoCols (groups of at most four query heads): mma columns 4-7 repeat the
// query heads of columns 0-3, so their scores, maxima and probabilities are
// the same numbers; lanes holding columns 0-3 pass the high f16 part of each
// probability to PV and lanes holding columns 4-7 the low part, and the two
// column halves of O^T are added when a piece ends.  Larger groups use all
// eight columns and a second PV mma for the low parts.
// kClust: one item per thread-block cluster of p.clust CTAs (small batches);
// otherwise persistent workers over the whole page stream.
template <int kKv, int kD, bool kLoCols, bool kClust, int kG>
__global__ void __launch_bounds__(kThreads, kG == 1 ? Cfg<kKv, kD>::kMinCtas : (kD == 128 ? 2 : 3))
    decode_kernel(const DecodeArgs p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv)
{
    using C = Cfg<kKv, kD>;
    static_assert(kG == 1 || !kLoCols, "several groups per item use all eight mma columns");
    constexpr int kGH = kItemHeads * kG;  // query heads per work item
    constexpr bool kInt8 = C::kInt8;
    constexpr int S = C::kStages;
    constexpr int PPS = C::kPPS;
    constexpr int KS = kD / 16;  // mma k-steps over head_dim, also m-tiles of O^T
    [[maybe_unused]] constexpr uint32_t kTmaAlign = C::kSwizzle == 128 ? 1024 : 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + C::kTabOffset);
    int32_t *ctxs = prefix + p.num_seqs + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;  // mma fragment row group / column pair
    [[maybe_unused]] const float lo_sel = c >= 2 ? 1.f : 0.f;  // kLoCols: low-part lanes

    if (threadIdx.x == 0) {
        ptx::prefetch_tmap(&tmk);
        ptx::prefetch_tmap(&tmv);
    }
    // This warp's stage barriers, set up before anything else (shared memory
    // only) so that the fence making them visible to the copy engine is done
    // by the time the first copies are issued.
    const uint32_t bar0 = ptx::smem_addr(smem + C::kBarOffset) + warp * S * 8;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) ptx::mbar_init(PKV_SMEM(bar0 + 8 * s, 8, 8), kInt8 ? 2 : 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    // Launched as a programmatic dependent of the previous kernel on the
    // stream: wait until its writes are visible before reading any input.
    ptx::griddep_wait();
    // The next kernel on the stream may begin its own launch now; it waits
    // for this grid's completion before reading anything this grid writes.
    ptx::griddep_launch_dependents();
    const int64_t mb = p.max_blocks_per_seq;

    int n = 0;       // pages of this worker
    PageCursor ci;   // its first page
    int w = 0;       // persistent workers: the worker's index
    // One item per cluster: the item's pages of the longest possible context
    // (cP) are split evenly over the cluster's cW warps, this warp being cw;
    // the item's actual pages are cnp, its sequence's context length cctx.
    int cP = 0, cW = 0, cw = 0, cnp = 0, cctx = 0;
    int32_t pre_blk = 0;  // block id of page (first page + lane), cluster mode
    // cluster mode: the record of head h of this warp's piece, in the shared
    // memory of the CTA that merges head h (rank h mod clust), slot
    // (h / clust) * cW + cw; the layout of a partial record (m, l, -, -, acc)
    float *crec = reinterpret_cast<float *>(smem + C::crec_offset(p.num_seqs));
    auto crec_of = [&](int h) -> float * {
        const int slot = (h / p.clust) * cW + cw;
        float *local = PKV_REC(crec + slot * (kD + 4), (kD + 4) * 4);
        return static_cast<float *>(ptx::map_generic(local, h % p.clust));
    };
    if constexpr (kClust) {
        const int r = static_cast<int>(ptx::cluster_ctarank());
        const int gi = blockIdx.x / p.clust;  // the cluster's item
        const int seq = gi / p.items_per_seq, item = gi - seq * p.items_per_seq;
        cP = (p.ctx_cap + kPage - 1) / kPage;
        cW = p.clust * kWarps;
        cw = r * kWarps + warp;
        const int lo = static_cast<int>(static_cast<int64_t>(cw) * cP / cW);
        const int hi = static_cast<int>(static_cast<int64_t>(cw + 1) * cP / cW);
        // the block ids of this warp's first stages (pages below cP are in
        // the table row) and the context length, in one round trip
        if (lane < S * PPS && lo + lane < hi)
            pre_blk = __ldg(PKV_TABLE_AT(p, seq, lo, lane, mb));
        const int cx = __ldg(p.context_lens + seq);
        const bool ok = cx >= 0 && cx <= p.ctx_cap;
        cctx = ok ? cx : -1;
        cnp = ok ? (cx + kPage - 1) / kPage : 0;
        n = max(0, min(hi, cnp) - lo);
        ci.seq = seq;
        ci.item = item;
        ci.kvh = item / p.qgroups;
        ci.qg = item - ci.kvh * p.qgroups;
        ci.page = lo;
        ci.npages = cnp;
        if (!ok && cw == 0 && lane == 0 && p.dev_status) atomicOr(p.dev_status, PKV_DEV_BAD_CTX);
    } else {
        build_page_tables(p, prefix, ctxs);
        const int64_t total = static_cast<int64_t>(p.items_per_seq) * prefix[p.num_seqs];

        // Sequences with no pages: zero output (bad lengths are also reported).
        for (int s = blockIdx.x; s < p.num_seqs; s += gridDim.x) {
            if (prefix[s + 1] != prefix[s]) continue;
            if (ctxs[s] < 0 && threadIdx.x == 0 && p.dev_status)
                atomicOr(p.dev_status, PKV_DEV_BAD_CTX);
            float4 *o =
                reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(s) * p.num_heads * kD);
            for (int i = threadIdx.x; i < p.num_heads * kD / 4; i += kThreads)
                o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }

        w = blockIdx.x * kWarps + warp;
        if (w >= p.num_workers) return;
        if (total == 0) return;
        const int64_t a = muldiv(w, total, p.num_workers);
        const int64_t b = muldiv(w + 1, total, p.num_workers);
        if (a >= b) return;
        n = static_cast<int>(b - a);
        ci.seek(p, prefix, a, lane);
    }

    const uint32_t stage0 = ptx::smem_addr(smem) + warp * S * C::kStageBytes;
    uint8_t *hdr_base = smem + C::kHdrOffset + warp * S * C::kHdrBytes;
    const uint32_t hdr0 = ptx::smem_addr(hdr_base);
    const uint64_t policy = ptx::policy_evict_first();
    const uint64_t stage_wait_ns = PKV_STAGE_WAIT_NS;

    // Lane 0: start the copies of the `cnt` pages of one stage; blk[u] are
    // their block ids, kvh the kv head of the item.
    auto issue = [&](int slot, int cnt, const int32_t (&blk)[PPS], int kvh) {
        const uint32_t bar = bar0 + 8 * slot;
        int32_t *hb = reinterpret_cast<int32_t *>(hdr_base + slot * C::kHdrBytes);
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < PPS; ++u) {
            const bool ok = u < cnt && blk[u] >= 0 && blk[u] < p.num_blocks;
            hb[u] = ok ? 0 : 1;
            if (u < cnt && !ok && p.dev_status) atomicOr(p.dev_status, PKV_DEV_BAD_BLOCK);
            bytes += ok ? C::kPageBytes : 0;
        }
        ptx::mbar_arrive_expect_tx(PKV_SMEM(bar, 8, 8), bytes);
#pragma unroll
        for (int u = 0; u < PPS; ++u) {
            if (hb[u]) continue;
            const int row = (blk[u] * p.num_kv_heads + kvh) * kPage;
            const uint32_t kdst = stage0 + slot * C::kStageBytes + u * C::kPageBytes;
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx) {
                ptx::tma_load_2d(PKV_SMEM(kdst + bx * C::kBoxBytes, C::kBoxBytes, kTmaAlign), &tmk,
                                 bx * C::kBoxInner, row, bar,
                                 policy);
                ptx::tma_load_2d(PKV_SMEM(kdst + C::kTileBytes + bx * C::kBoxBytes, C::kBoxBytes,
                                          kTmaAlign),
                                 &tmv,
                                 bx * C::kBoxInner, row, bar, policy);
            }
            if constexpr (kInt8) {
                const int64_t si = static_cast<int64_t>(blk[u]) * p.num_kv_heads + kvh;
                ptx::cp_async_4(PKV_SMEM(hdr0 + slot * C::kHdrBytes + 8 + 4 * u, 4, 4),
                                p.k_scales + si);
                ptx::cp_async_4(PKV_SMEM(hdr0 + slot * C::kHdrBytes + 16 + 4 * u, 4, 4),
                                p.v_scales + si);
            }
        }
        if constexpr (kInt8) ptx::cp_async_arrive_noinc(PKV_SMEM(bar, 8, 8));
    };

    // ---- prologue: block ids of the first stages (one lane per page), issue
    PageCursor cc = ci;
    int ipos = 0;          // pages issued so far
    uint32_t issued = 0;   // stages issued so far
    {
        // lane j*PPS + u holds page u of stage j
        PageCursor cj = ci;
        int pos = 0;
        const int my_stage = lane / PPS, my_u = lane % PPS;
        int32_t myblk = 0;
        int mykvh = 0, mycnt = 0;
        for (int j = 0; j < S && pos < n; ++j) {
            const int cnt = cj.unit(PPS, n - pos);
            if (j == my_stage) {
                mycnt = cnt;
                mykvh = cj.kvh;
                // cluster mode: one item, pages in order, ids loaded above
                if (my_u < cnt)
                    myblk = kClust ? pre_blk : __ldg(PKV_TABLE_AT(p, cj.seq, cj.page, my_u, mb));
            }
            cj.advance(p, prefix, cnt);
            pos += cnt;
        }
        for (int j = 0; j < S && ipos < n; ++j) {
            const int cnt = __shfl_sync(0xffffffffu, mycnt, j * PPS);
            const int kvh = __shfl_sync(0xffffffffu, mykvh, j * PPS);
            int32_t blk[PPS];
#pragma unroll
            for (int u = 0; u < PPS; ++u) blk[u] = __shfl_sync(0xffffffffu, myblk, j * PPS + u);
            if (lane == 0) issue(j, cnt, blk, kvh);
            ci.advance(p, prefix, cnt);
            ipos += cnt;
            ++issued;
        }
    }
    // lanes u < PPS: block id of page u of the next stage to issue
    int32_t nblk = 0;
    if (ipos < n && lane < ci.unit(PPS, n - ipos))
        nblk = __ldg(PKV_TABLE_AT(p, ci.seq, ci.page, lane, mb));

    // ---- per-piece state, per group of 8 query heads (the item's kG groups
    // share every page)
    float m0[kG], m1[kG];    // running max (log2 units), heads 2c and 2c+1 of the group
    float l0[kG], l1[kG];    // lane-partial running sums
    float o[kG][KS][4];      // O^T accumulators (see the output mapping)
    uint32_t qf[kG][KS][2];  // Q^T B-fragments
    float qb0[kG], qb1[kG];  // INT8: 1152 * sum(q) of heads 2c, 2c+1
#pragma unroll
    for (int gi = 0; gi < kG; ++gi) {
        m0[gi] = m1[gi] = -INFINITY;
        l0[gi] = l1[gi] = 0.f;
        qb0[gi] = qb1[gi] = 0.f;
    }
    // Codes: V scale reference of the piece (the largest V scale of its pages
    // so far) and its reciprocal.  A page enters PV with its probabilities
    // times sv / vref <= 1, so the f16 operand keeps its full precision
    // whatever the magnitude of V; vref multiplies the accumulators only
    // when they leave the registers.
    float vref = 0.f, vinv = 0.f;
    bool piece_bad = false;
    bool piece_has_a = true;
    int piece_first_page = 0;
    int piece_pages = 0;

    bool timed_out = false;
    int pos = 0;
    for (uint32_t k = 0; pos < n; ++k) {
        const int slot = static_cast<int>(k % S);
        const uint32_t parity = (k / S) & 1u;
        const int cnt = cc.unit(PPS, n - pos);
        const bool first = pos == 0 || cc.page == 0;
        const bool last = pos + cnt == n || cc.page + cnt == cc.npages;
        const int h0 = cc.kvh * p.group + cc.qg * kGH;
        const int gh = min(kGH, p.group - cc.qg * kGH);

        if (first) {
            // query fragments of the item's heads (group gi, column g: head
            // 8 gi + g, or g mod 4 with kLoCols); heads past gh are zero
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                const int hq = kItemHeads * gi + (kLoCols ? (g & 3) : g);
                const __half *qrow =
                    p.query + (static_cast<int64_t>(cc.seq) * p.num_heads + h0 + hq) * kD;
                const bool live = hq < gh;
                if constexpr (kInt8) {
                    // lane (g, c) holds q[g][DG*c .. DG*c + DG), DG = kD / 4
                    constexpr int DG = kD / 4;
                    uint4 qv[DG / 8];
#pragma unroll
                    for (int j = 0; j < DG / 8; ++j)
                        qv[j] = live ? __ldg(reinterpret_cast<const uint4 *>(qrow + DG * c) + j)
                                     : make_uint4(0, 0, 0, 0);
                    const uint32_t *qw = reinterpret_cast<const uint32_t *>(qv);
                    float qs = 0.f;
#pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        qf[gi][s][0] = qw[2 * s];
                        qf[gi][s][1] = qw[2 * s + 1];
                        const float2 f0 =
                            __half22float2(*reinterpret_cast<const __half2 *>(&qw[2 * s]));
                        const float2 f1 =
                            __half22float2(*reinterpret_cast<const __half2 *>(&qw[2 * s + 1]));
                        qs += (f0.x + f0.y) + (f1.x + f1.y);
                    }
                    // sum over the head's four lanes, then fetch heads 2c and 2c+1
                    qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                    qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                    if constexpr (kKv == kKvI8) {  // FP8 codes carry no bias
                        qb0[gi] = 1152.f * __shfl_sync(0xffffffffu, qs, 8 * c);
                        qb1[gi] = 1152.f * __shfl_sync(0xffffffffu, qs, 8 * c + 4);
                    }
                } else {
                    const uint32_t *qw = reinterpret_cast<const uint32_t *>(qrow);
#pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        qf[gi][s][0] = live ? __ldg(qw + 8 * s + c) : 0u;
                        qf[gi][s][1] = live ? __ldg(qw + 8 * s + 4 + c) : 0u;
                    }
                }
            }
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                m0[gi] = m1[gi] = -INFINITY;
                l0[gi] = l1[gi] = 0.f;
            }
            vref = vinv = 0.f;
#pragma unroll
            for (int gi = 0; gi < kG; ++gi)
#pragma unroll
                for (int i = 0; i < KS; ++i)
                    o[gi][i][0] = o[gi][i][1] = o[gi][i][2] = o[gi][i][3] = 0.f;
            piece_bad = false;
            piece_has_a = pos == 0;
            piece_first_page = cc.page;
            piece_pages = 0;
        }
        piece_pages += cnt;

        // every lane waits (acquire); the outcome is made warp-uniform
        const bool landed =
            stage_wait_ns != 0 &&
            ptx::mbar_wait_bounded(PKV_SMEM(bar0 + 8 * slot, 8, 8), parity, stage_wait_ns);
        if (!__all_sync(0xffffffffu, landed)) {
            // The copy did not land in time: report, let every copy this
            // worker issued land (bounded; the stage just waited on
            // included), so that none still writes into this CTA's shared
            // memory, and stop this worker.
            if (lane == 0 && p.dev_status) atomicOr(p.dev_status, PKV_DEV_TIMEOUT);
            for (uint32_t r = k; r < issued; ++r)
                ptx::mbar_wait_bounded(PKV_SMEM(bar0 + 8 * (r % S), 8, 8), (r / S) & 1u,
                                       kWaitLimitNs);
            if constexpr (!kClust) return;
            timed_out = true;  // the cluster's merge still needs this warp
            break;
        }

        const int32_t *hb = reinterpret_cast<const int32_t *>(hdr_base + slot * C::kHdrBytes);
        const float *hf = reinterpret_cast<const float *>(hb);
        bool good[PPS];
        bool any_good = false;
#pragma unroll
        for (int u = 0; u < PPS; ++u) {
            good[u] = u < cnt && hb[u] == 0;
            piece_bad |= u < cnt && !good[u];
            any_good |= good[u];
        }
        if (any_good) {
            const uint32_t st = stage0 + slot * C::kStageBytes;
            const int ctx = kClust ? cctx : ctxs[PKV_IDX(cc.seq, p.num_seqs)];
            // ---- scores of the stage's pages, base-2 logits
            float x[kG][PPS][4];
#pragma unroll
            for (int u = 0; u < PPS; ++u) {
                if (good[u]) {
                    float sc[kG][4];
                    page_scores<kKv, kD, kG>(st + u * C::kPageBytes, qf, lane, sc);
                    float sl = p.scale_log2;
                    if constexpr (kInt8) sl *= hf[2 + u];
                    const int ntok = ctx - (cc.page + u) * kPage;
#pragma unroll
                    for (int gi = 0; gi < kG; ++gi) {
                        if constexpr (kInt8) {
                            x[gi][u][0] = (sc[gi][0] - qb0[gi]) * sl;
                            x[gi][u][1] = (sc[gi][1] - qb1[gi]) * sl;
                            x[gi][u][2] = (sc[gi][2] - qb0[gi]) * sl;
                            x[gi][u][3] = (sc[gi][3] - qb1[gi]) * sl;
                        } else {
                            x[gi][u][0] = sc[gi][0] * sl;
                            x[gi][u][1] = sc[gi][1] * sl;
                            x[gi][u][2] = sc[gi][2] * sl;
                            x[gi][u][3] = sc[gi][3] * sl;
                        }
                        if (ntok < kPage) {
                            if (g >= ntok) x[gi][u][0] = x[gi][u][1] = -INFINITY;
                            if (g + 8 >= ntok) x[gi][u][2] = x[gi][u][3] = -INFINITY;
                        }
                    }
                } else {
#pragma unroll
                    for (int gi = 0; gi < kG; ++gi)
                        x[gi][u][0] = x[gi][u][1] = x[gi][u][2] = x[gi][u][3] = -INFINITY;
                }
            }
            // ---- online softmax, one update for the whole stage, per group
            float mn0[kG], mn1[kG], al0[kG], al1[kG];
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                float mx0 = fmaxf(x[gi][0][0], x[gi][0][2]), mx1 = fmaxf(x[gi][0][1], x[gi][0][3]);
#pragma unroll
                for (int u = 1; u < PPS; ++u) {
                    mx0 = fmaxf(mx0, fmaxf(x[gi][u][0], x[gi][u][2]));
                    mx1 = fmaxf(mx1, fmaxf(x[gi][u][1], x[gi][u][3]));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                mn0[gi] = fmaxf(m0[gi], mx0);
                mn1[gi] = fmaxf(m1[gi], mx1);
                al0[gi] = ptx::ex2(m0[gi] - mn0[gi]);
                al1[gi] = ptx::ex2(m1[gi] - mn1[gi]);
                m0[gi] = mn0[gi];
                m1[gi] = mn1[gi];
            }
            float oa0[kG], oa1[kG];  // rescale of the accumulators
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                oa0[gi] = al0[gi];
                oa1[gi] = al1[gi];
            }
            [[maybe_unused]] float vr[PPS];
            if constexpr (kInt8) {
                // a page with a larger V scale becomes the reference: the
                // accumulators move to the new reference with the rescale
                float smax = vref;
#pragma unroll
                for (int u = 0; u < PPS; ++u)
                    if (good[u]) smax = fmaxf(smax, hf[4 + u]);
                if (smax > vref) {
                    vinv = __frcp_rn(smax);
                    const float ratio = vref * vinv;
                    vinv *= kPScale;
#pragma unroll
                    for (int gi = 0; gi < kG; ++gi) {
                        oa0[gi] *= ratio;
                        oa1[gi] *= ratio;
                    }
                    vref = smax;
                }
#pragma unroll
                for (int u = 0; u < PPS; ++u) vr[u] = hf[4 + u] * vinv;
            }
            float pr[kG][PPS][4];
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int u = 0; u < PPS; ++u) {
                    pr[gi][u][0] = ptx::ex2(x[gi][u][0] - mn0[gi]);
                    pr[gi][u][1] = ptx::ex2(x[gi][u][1] - mn1[gi]);
                    pr[gi][u][2] = ptx::ex2(x[gi][u][2] - mn0[gi]);
                    pr[gi][u][3] = ptx::ex2(x[gi][u][3] - mn1[gi]);
                    ps0 += pr[gi][u][0] + pr[gi][u][2];
                    ps1 += pr[gi][u][1] + pr[gi][u][3];
                }
                l0[gi] = l0[gi] * al0[gi] + ps0;
                l1[gi] = l1[gi] * al1[gi] + ps1;
                if (__any_sync(0xffffffffu, oa0[gi] != 1.f || oa1[gi] != 1.f)) {
#pragma unroll
                    for (int i = 0; i < KS; ++i) {
                        o[gi][i][0] *= oa0[gi];
                        o[gi][i][1] *= oa1[gi];
                        o[gi][i][2] *= oa0[gi];
                        o[gi][i][3] *= oa1[gi];
                    }
                }
            }
            // ---- O^T += V^T . P^T per page (P^T: transposed 8x8 halves of P)
#pragma unroll
            for (int u = 0; u < PPS; ++u) {
                if (good[u]) {
                    // P' = 2^15 p (codes: 2^15 p sv / vref) <= 2^15, exact
                    // scaling by a power of two; its f16 high part is a normal
                    // number down to p = 2^-29 and the low part adds the
                    // next 11 bits
                    const float sc = kInt8 ? vr[u] : kPScale;
                    uint32_t pb0[kG], pb1[kG], pl0[kG], pl1[kG];
#pragma unroll
                    for (int gi = 0; gi < kG; ++gi) {
                        const float pa = pr[gi][u][0] * sc, pb = pr[gi][u][1] * sc;
                        const float pc = pr[gi][u][2] * sc, pd = pr[gi][u][3] * sc;
                        const uint32_t h01 = pack_half2(pa, pb), h23 = pack_half2(pc, pd);
                        const float2 f01 = unpack_half2(h01), f23 = unpack_half2(h23);
                        pl0[gi] = pl1[gi] = 0;
                        if constexpr (kLoCols) {
                            // columns 0-3 (c < 2): high parts; 4-7: low parts
                            pb0[gi] = ptx::movmatrix_t(
                                pack_half2(fmaf(-lo_sel, f01.x, pa), fmaf(-lo_sel, f01.y, pb)));
                            pb1[gi] = ptx::movmatrix_t(
                                pack_half2(fmaf(-lo_sel, f23.x, pc), fmaf(-lo_sel, f23.y, pd)));
                        } else {
                            pb0[gi] = ptx::movmatrix_t(h01);
                            pb1[gi] = ptx::movmatrix_t(h23);
                            pl0[gi] = ptx::movmatrix_t(pack_half2(pa - f01.x, pb - f01.y));
                            pl1[gi] = ptx::movmatrix_t(pack_half2(pc - f23.x, pd - f23.y));
                        }
                    }
                    const int ntok = min(kPage, ctx - (cc.page + u) * kPage);
                    page_pv<kKv, kD, kLoCols, kG>(st + u * C::kPageBytes + C::kTileBytes, pb0,
                                                  pb1, pl0, pl1, ntok, lane, o);
                }
            }
        }
        __syncwarp();

        // ---- refill this stage with the next pages
        if (ipos < n) {
            const int icnt = ci.unit(PPS, n - ipos);
            int32_t blk[PPS];
#pragma unroll
            for (int u = 0; u < PPS; ++u) blk[u] = __shfl_sync(0xffffffffu, nblk, u);
            if (lane == 0) {
                ptx::fence_proxy_async_smem();
                issue(slot, icnt, blk, ci.kvh);
            }
            ci.advance(p, prefix, icnt);
            ipos += icnt;
            ++issued;
            if (ipos < n && lane < ci.unit(PPS, n - ipos))
                nblk = __ldg(PKV_TABLE_AT(p, ci.seq, ci.page, lane, mb));
        }

        // ---- piece finished: final output, or a partial for the reduce
        if (last) {
            const bool whole =
                !kClust && piece_first_page == 0 && cc.page + cnt == cc.npages;
#pragma unroll
            for (int gi = 0; gi < kG; ++gi) {
                if constexpr (kLoCols) {
                    // add the low-part columns (lanes c + 2) to the high-part ones
#pragma unroll
                    for (int i = 0; i < KS; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[gi][i][j] += __shfl_xor_sync(0xffffffffu, o[gi][i][j], 2);
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l0[gi] += __shfl_xor_sync(0xffffffffu, l0[gi], off);
                    l1[gi] += __shfl_xor_sync(0xffffffffu, l1[gi], off);
                }
                const int hA = kItemHeads * gi + 2 * c, hB = hA + 1;  // heads of the item
                float *dstA, *dstB;
                float fA, fB;
                if (whole) {
                    const int64_t orow = (static_cast<int64_t>(cc.seq) * p.num_heads + h0) * kD;
                    dstA = p.out + orow + static_cast<int64_t>(hA) * kD;
                    dstB = p.out + orow + static_cast<int64_t>(hB) * kD;
                    const float vs = (kInt8 ? vref : 1.f) * kPScaleInv;
                    fA = piece_bad ? 0.f : vs / l0[gi];
                    fB = piece_bad ? 0.f : vs / l1[gi];
                } else {
                    if constexpr (kClust) {
                        // pushed to the shared memory of the CTAs merging hA, hB
                        dstA = hA < gh ? crec_of(hA) + 4 : nullptr;
                        dstB = hB < gh ? crec_of(hB) + 4 : nullptr;
                    } else {
                        const int slotp = piece_has_a ? 0 : 1;
                        float *rec = p.partials + (static_cast<int64_t>(w) * 2 + slotp) *
                                                      p.rec_heads * (kD + 4);
                        dstA = rec + hA * (kD + 4) + 4;
                        dstB = rec + hB * (kD + 4) + 4;
                    }
                    fA = fB = (kInt8 ? vref : 1.f) * kPScaleInv;  // accumulators in V units
                    if (g == 0) {
                        // m, l, and a zero word (the many-piece reduce counts
                        // its CTAs in the first piece's)
                        if (hA < gh) {
                            dstA[-4] = m0[gi];
                            dstA[-3] = piece_bad ? -1.f : l0[gi];
                            if constexpr (!kClust) dstA[-2] = 0.f;
                        }
                        if (hB < gh) {
                            dstB[-4] = m1[gi];
                            dstB[-3] = piece_bad ? -1.f : l1[gi];
                            if constexpr (!kClust) dstB[-2] = 0.f;
                        }
                    }
                }
                if (piece_bad) {
#pragma unroll
                    for (int i = 0; i < KS; ++i)
                        o[gi][i][0] = o[gi][i][1] = o[gi][i][2] = o[gi][i][3] = 0.f;
                }
                if constexpr (!kInt8) {
#pragma unroll
                    for (int i = 0; i < KS; ++i) {
                        if (hA < gh) {
                            dstA[16 * i + g] = o[gi][i][0] * fA;
                            dstA[16 * i + 8 + g] = o[gi][i][2] * fA;
                        }
                        if (hB < gh) {
                            dstB[16 * i + g] = o[gi][i][1] * fB;
                            dstB[16 * i + 8 + g] = o[gi][i][3] * fB;
                        }
                    }
                } else {
                    constexpr int DG = kD / 8;  // lane (g, c) owns d in [DG*g, DG*g + DG)
#pragma unroll
                    for (int i = 0; i < KS; i += 2) {
                        if (hA < gh)
                            *reinterpret_cast<float4 *>(dstA + DG * g + 2 * i) =
                                make_float4(o[gi][i][0] * fA, o[gi][i][2] * fA,
                                            o[gi][i + 1][0] * fA, o[gi][i + 1][2] * fA);
                        if (hB < gh)
                            *reinterpret_cast<float4 *>(dstB + DG * g + 2 * i) =
                                make_float4(o[gi][i][1] * fB, o[gi][i][3] * fB,
                                            o[gi][i + 1][1] * fB, o[gi][i + 1][3] * fB);
                    }
                }
            }
        }
        cc.advance(p, prefix, cnt);
        pos += cnt;
    }
    if constexpr (!kClust) return;
    else {

    // ---- one item per cluster: merge the cluster's pieces of the item
    // Every warp with pages has pushed its (m, l, acc) record of each head h
    // into the shared memory of CTA h mod clust (one that timed out pushes a
    // bad mark).  After one cluster barrier every CTA merges its heads from
    // its own shared memory, in piece order:
    //   out = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j
    // and nothing reads another CTA's memory after the barrier.
    const int gi = blockIdx.x / p.clust;
    const int seq = gi / p.items_per_seq, item = gi - seq * p.items_per_seq;
    const int kvh = item / p.qgroups, qg = item - kvh * p.qgroups;
    const int gh = min(kGH, p.group - qg * kGH);
    const int h0 = kvh * p.group + qg * kGH;
    if (timed_out && lane < gh) crec_of(lane)[1] = -1.f;
    __syncwarp();
    ptx::cluster_sync();
    const int rank = static_cast<int>(ptx::cluster_ctarank());
    constexpr int kChunks = kD / 32;
    const int my_heads = gh > rank ? (gh - rank + p.clust - 1) / p.clust : 0;
    for (int t = warp; t < my_heads * kChunks; t += kWarps) {
        const int hl = t / kChunks, ch = t - hl * kChunks;
        const int h = rank + hl * p.clust;
        const float *rb = crec + hl * cW * (kD + 4);  // records of head h, piece 0
        float res = 0.f;
        if (cnp > 0) {
            // lane j: piece j's running max and sum
            const int j = lane;
            bool has = false;
            float mj = -INFINITY, lj = 0.f;
            if (j < cW) {
                const int lo_j = static_cast<int>(static_cast<int64_t>(j) * cP / cW);
                const int hi_j = min(static_cast<int>(static_cast<int64_t>(j + 1) * cP / cW), cnp);
                has = lo_j < hi_j;
                if (has) {
                    const float *rj = PKV_REC(const_cast<float *>(rb) + j * (kD + 4), (kD + 4) * 4);
                    mj = rj[0];
                    lj = rj[1];
                }
            }
            float M = mj;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            const bool bad = __any_sync(0xffffffffu, has && lj < 0.f);
            const float fj = has ? ptx::ex2(mj - M) : 0.f;
            float L = fj * lj;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
            // accumulators: every piece's value at this lane's head_dim
            // index, eight pieces' loads in flight at a time
            float acc = 0.f;
            const float *vp = rb + 4 + 32 * ch + lane;
            for (int jb = 0; jb < cW; jb += 8) {
                float v[8], f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    f[u] = __shfl_sync(0xffffffffu, fj, (jb + u) & 31);
                    v[u] = jb + u < cW && f[u] != 0.f ? vp[(jb + u) * (kD + 4)] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) acc += f[u] * v[u];
            }
            res = bad ? 0.f : acc / L;
        }
        p.out[(static_cast<int64_t>(seq) * p.num_heads + h0 + h) * kD + 32 * ch + lane] = res;
    }
    }
}

// Split-context reduce.  Tasks are (item, query head); a warp takes tasks
// gw, gw + warps, ... and merges those whose item is split across workers:
//   out = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w,  M = max_w m_w
// over the pieces of the workers holding the item's first .. last page.  A
// piece flagged bad (l < 0) zeroes the item.  Which items are split, which
// workers hold their pieces and where those records are depend only on the
// partition of the page stream, i.e. on context_lens, an input of the call:
// all of it is worked out before the kernel waits for the decode grid, so
// that after the wait only the records are read (every load of up to eight
// pieces at once; beyond that the (m, l) of 32 pieces per round, one lane per
// piece, then the accumulators four pieces per batch).  Lanes run across
// head_dim; pieces are combined in a fixed order.
constexpr int kRedThreads = 128;

template <int kD>
__global__ void __launch_bounds__(kRedThreads) reduce_kernel(const DecodeArgs p)
{
    extern __shared__ __align__(16) uint8_t rsmem[];
    int32_t *prefix = reinterpret_cast<int32_t *>(rsmem);
    int32_t *ctxs = prefix + p.num_seqs + 1;
    build_page_tables<kRedThreads>(p, prefix, ctxs);
    const int lane = threadIdx.x & 31;
    const int W = p.num_workers;
    const int64_t total = static_cast<int64_t>(p.items_per_seq) * prefix[p.num_seqs];
    const int64_t per_seq = static_cast<int64_t>(p.items_per_seq) * p.rec_heads;
    const int64_t ntasks = per_seq * p.num_seqs;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kRedThreads / 32);
    bool waited = false;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * (kRedThreads / 32) + (threadIdx.x >> 5);
         t < ntasks; t += nwarps) {
        const int seq = static_cast<int>(t / per_seq);
        const int rem = static_cast<int>(t - seq * per_seq);
        const int item = rem / p.rec_heads;
        const int h = rem - item * p.rec_heads;
        const int kvh = item / p.qgroups, qg = item - kvh * p.qgroups;
        const int gh = min(p.item_heads, p.group - qg * p.item_heads);
        const int npages = prefix[seq + 1] - prefix[seq];
        if (h >= gh || npages == 0) continue;
        const int64_t s0 = static_cast<int64_t>(p.items_per_seq) * prefix[seq] +
                           static_cast<int64_t>(item) * npages;  // the item's first page
        const int64_t last = s0 + npages - 1;
        const int wf = static_cast<int>(worker_of(s0, total, W));
        const int nw = static_cast<int>(worker_of(last, total, W)) - wf + 1;
        if (nw == 1) continue;  // whole inside one worker: finished by the decode
        const int slot0 = s0 == muldiv(wf, total, W) ? 0 : 1;

        // the record of piece j of this item (null: a worker with no pages)
        auto rec_of = [&](int j) -> const float * {
            const int64_t w = wf + j;
            if (j > 0 && muldiv(w, total, W) == muldiv(w + 1, total, W)) return nullptr;
            const int slot = j == 0 ? slot0 : 0;
            return p.partials + ((w * 2 + slot) * p.rec_heads + h) * (kD + 4);
        };
        constexpr int kFast = 8;  // pieces whose loads are all issued at once
        const float *rp[kFast];
#pragma unroll
        for (int j = 0; j < kFast; ++j) rp[j] = j < nw ? rec_of(j) : nullptr;
        if (!waited) {
            ptx::griddep_wait();  // the decode grid's records are complete and visible
            waited = true;
        }

        float acc[kD / 32];
#pragma unroll
        for (int i = 0; i < kD / 32; ++i) acc[i] = 0.f;
        float L = 0.f;
        bool bad = false;
        if (nw <= kFast) {
            float m[kFast], l[kFast], v[kFast][kD / 32];
#pragma unroll
            for (int j = 0; j < kFast; ++j) {
                const float *r = rp[j];
                if (r) {
                    m[j] = __ldcg(r);
                    l[j] = __ldcg(r + 1);
#pragma unroll
                    for (int i = 0; i < kD / 32; ++i) v[j][i] = __ldcg(r + 4 + lane + 32 * i);
                } else {
                    m[j] = -INFINITY;
                    l[j] = 0.f;
#pragma unroll
                    for (int i = 0; i < kD / 32; ++i) v[j][i] = 0.f;
                }
            }
            float M = m[0];
#pragma unroll
            for (int j = 1; j < kFast; ++j) M = fmaxf(M, m[j]);
#pragma unroll
            for (int j = 0; j < kFast; ++j) {
                const float f = m[j] == -INFINITY ? 0.f : ptx::ex2(m[j] - M);
                bad |= l[j] < 0.f;
                L += f * l[j];
#pragma unroll
                for (int i = 0; i < kD / 32; ++i) acc[i] += f * v[j][i];
            }
        } else {
            float M = -INFINITY;
            for (int base = 0; base < nw; base += 32) {
                const float *r = base + lane < nw ? rec_of(base + lane) : nullptr;
                if (r) {
                    M = fmaxf(M, __ldcg(r));
                    bad |= __ldcg(r + 1) < 0.f;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            bad = __any_sync(0xffffffffu, bad);
            for (int base = 0; base < nw; base += 32) {
                const float *mine = base + lane < nw ? rec_of(base + lane) : nullptr;
                const float f_lane = mine ? ptx::ex2(__ldcg(mine) - M) : 0.f;
                float Lp = mine ? f_lane * __ldcg(mine + 1) : 0.f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) Lp += __shfl_xor_sync(0xffffffffu, Lp, off);
                L += Lp;
                const uint64_t mbits = reinterpret_cast<uint64_t>(mine);
                const uint32_t mlo = static_cast<uint32_t>(mbits);
                const uint32_t mhi = static_cast<uint32_t>(mbits >> 32);
                const int cnt = min(32, nw - base);
                for (int j0 = 0; j0 < cnt; j0 += 4) {
                    float v[4][kD / 32], f[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int src = min(j0 + u, 31);
                        const uint64_t bits =
                            (static_cast<uint64_t>(__shfl_sync(0xffffffffu, mhi, src)) << 32) |
                            __shfl_sync(0xffffffffu, mlo, src);
                        f[u] = __shfl_sync(0xffffffffu, f_lane, src);
                        const float *r = reinterpret_cast<const float *>(bits);
                        const bool use = j0 + u < cnt && r != nullptr;
                        if (!use) f[u] = 0.f;
#pragma unroll
                        for (int i = 0; i < kD / 32; ++i)
                            v[u][i] = use ? __ldcg(r + 4 + lane + 32 * i) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int i = 0; i < kD / 32; ++i) acc[i] += f[u] * v[u][i];
                }
            }
        }
        const int h0 = kvh * p.group + qg * p.item_heads;
        float *dst = p.out + (static_cast<int64_t>(seq) * p.num_heads + h0 + h) * kD;
        const float inv = bad ? 0.f : 1.f / L;
#pragma unroll
        for (int i = 0; i < kD / 32; ++i) dst[lane + 32 * i] = bad ? 0.f : acc[i] * inv;
    }
}

// Split-context reduce for items cut into many pieces (a few long contexts
// spread over the whole grid).  S CTAs (1-8) of kManyWarps warps share each
// (item, query head) task: warp k of CTA r merges the chunks of eight pieces
// numbered r * kManyWarps + k, then that plus A * kManyWarps, ... (A: the
// task's active CTAs, those with pieces; each chunk's loads all in flight,
// merged online into a running max, sum and accumulator), and the CTA
// combines its warps' partials in shared memory.  With one active CTA that
// is the output.  Otherwise CTA r stores its partial in the record of piece
// 64 r (read by this CTA alone, already consumed), and counts itself in the
// zero word of piece 0's record; the CTA that arrives last combines the A
// partials in rank order, so the bits do not depend on the arrival order:
//   out = sum_r 2^(M_r - M) acc_r / sum_r 2^(M_r - M) L_r,  M = max_r M_r
// No CTA waits for another.  Used instead of reduce_kernel when the grid has
// more than eight workers per item on average.
constexpr int kManyWarps = 8;
constexpr int kManyThreads = kManyWarps * 32;
constexpr int kManyChunk = kManyWarps * 8;  // pieces one CTA takes per round

template <int kD>
__global__ void __launch_bounds__(kManyThreads) reduce_many_kernel(const DecodeArgs p, int S)
{
    constexpr int kC = kD / 32;  // accumulator floats per lane
    extern __shared__ __align__(16) uint8_t msmem[];
    int32_t *prefix = reinterpret_cast<int32_t *>(msmem);
    int32_t *ctxs = prefix + p.num_seqs + 1;
    __shared__ float sm_m[kManyWarps], sm_l[kManyWarps];
    __shared__ int sm_bad[kManyWarps];
    __shared__ __align__(16) float sm_acc[kManyWarps][kD];
    build_page_tables<kManyThreads>(p, prefix, ctxs);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = static_cast<int>(blockIdx.x % S);
    const int W = p.num_workers;
    const int64_t total = static_cast<int64_t>(p.items_per_seq) * prefix[p.num_seqs];
    const int64_t per_seq = static_cast<int64_t>(p.items_per_seq) * p.rec_heads;
    const int64_t ntasks = per_seq * p.num_seqs;
    const int64_t ngroups = gridDim.x / S;
    ptx::griddep_wait();  // the decode grid's records are complete and visible
    for (int64_t t = blockIdx.x / S; t < ntasks; t += ngroups) {
        const int seq = static_cast<int>(t / per_seq);
        const int rem = static_cast<int>(t - seq * per_seq);
        const int item = rem / p.rec_heads;
        const int h = rem - item * p.rec_heads;
        const int kvh = item / p.qgroups, qg = item - kvh * p.qgroups;
        const int gh = min(p.item_heads, p.group - qg * p.item_heads);
        const int npages = prefix[seq + 1] - prefix[seq];
        if (h >= gh || npages == 0) continue;
        const int64_t s0 = static_cast<int64_t>(p.items_per_seq) * prefix[seq] +
                           static_cast<int64_t>(item) * npages;  // the item's first page
        const int64_t last = s0 + npages - 1;
        const int wf = static_cast<int>(worker_of(s0, total, W));
        const int nw = static_cast<int>(worker_of(last, total, W)) - wf + 1;
        if (nw == 1) continue;  // whole inside one worker: finished by the decode
        const int active = min(S, (nw + kManyChunk - 1) / kManyChunk);
        if (r >= active) continue;
        const int slot0 = s0 == muldiv(wf, total, W) ? 0 : 1;
        // the record slot of piece j of this item (that of a worker with no
        // pages is never written by the decode)
        auto rec_at = [&](int j) -> float * {
            const int64_t w = wf + j;
            const int slot = j == 0 ? slot0 : 0;
            return p.partials + ((w * 2 + slot) * p.rec_heads + h) * (kD + 4);
        };
        // the record of piece j (null: a worker with no pages)
        auto rec_of = [&](int j) -> const float * {
            const int64_t w = wf + j;
            if (j > 0 && muldiv(w, total, W) == muldiv(w + 1, total, W)) return nullptr;
            return rec_at(j);
        };
        float M = -INFINITY, L = 0.f, acc[kC];
#pragma unroll
        for (int i = 0; i < kC; ++i) acc[i] = 0.f;
        bool bad = false;
        for (int c0 = (r * kManyWarps + warp) * 8; c0 < nw; c0 += active * kManyChunk) {
            float m[8], l[8], v[8][kC];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float *rp = c0 + u < nw ? rec_of(c0 + u) : nullptr;
                if (rp) {
                    m[u] = __ldcg(rp);
                    l[u] = __ldcg(rp + 1);
#pragma unroll
                    for (int i = 0; i < kC; ++i) v[u][i] = __ldcg(rp + 4 + lane + 32 * i);
                } else {
                    m[u] = -INFINITY;
                    l[u] = 0.f;
#pragma unroll
                    for (int i = 0; i < kC; ++i) v[u][i] = 0.f;
                }
            }
            float Mn = M;
#pragma unroll
            for (int u = 0; u < 8; ++u) Mn = fmaxf(Mn, m[u]);
            const float fo = M == -INFINITY ? 0.f : ptx::ex2(M - Mn);
            L *= fo;
#pragma unroll
            for (int i = 0; i < kC; ++i) acc[i] *= fo;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float f = m[u] == -INFINITY ? 0.f : ptx::ex2(m[u] - Mn);
                bad |= l[u] < 0.f;
                L += f * l[u];
#pragma unroll
                for (int i = 0; i < kC; ++i) acc[i] += f * v[u][i];
            }
            M = Mn;
        }
        if (lane == 0) {
            sm_m[warp] = M;
            sm_l[warp] = L;
            sm_bad[warp] = bad ? 1 : 0;
        }
#pragma unroll
        for (int i = 0; i < kC; ++i) sm_acc[warp][lane + 32 * i] = acc[i];
        __syncthreads();
        if (warp == 0) {
            // this CTA's warps, in warp order (L < 0: a bad piece)
            float Mt = -INFINITY;
            bool anybad = false;
#pragma unroll
            for (int k = 0; k < kManyWarps; ++k) {
                Mt = fmaxf(Mt, sm_m[k]);
                anybad |= sm_bad[k] != 0;
            }
            float Lt = 0.f, o[kC];
#pragma unroll
            for (int i = 0; i < kC; ++i) o[i] = 0.f;
#pragma unroll
            for (int k = 0; k < kManyWarps; ++k) {
                const float f = sm_m[k] == -INFINITY ? 0.f : ptx::ex2(sm_m[k] - Mt);
                Lt += f * sm_l[k];
#pragma unroll
                for (int i = 0; i < kC; ++i) o[i] += f * sm_acc[k][lane + 32 * i];
            }
            bool write = true;
            if (active > 1) {
                float *part = rec_at(r * kManyChunk);
                if (lane == 0) {
                    part[0] = Mt;
                    part[1] = anybad ? -1.f : Lt;
                }
#pragma unroll
                for (int i = 0; i < kC; ++i) part[4 + lane + 32 * i] = o[i];
                __threadfence();  // the partial is visible before the count
                __syncwarp();
                int prior = 0;
                if (lane == 0)
                    prior = atomicAdd(reinterpret_cast<int *>(rec_at(0) + 2), 1);
                write = __shfl_sync(0xffffffffu, prior, 0) == active - 1;
                if (write) {
                    __threadfence();  // every other CTA's partial is visible
                    // all partials' loads in flight at once, then the merge
                    float mq[8], lq[8], vq[8][kC];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        mq[q] = -INFINITY;
                        lq[q] = 0.f;
#pragma unroll
                        for (int i = 0; i < kC; ++i) vq[q][i] = 0.f;
                        if (q < active) {
                            const float *pq = rec_at(q * kManyChunk);
                            mq[q] = __ldcg(pq);
                            lq[q] = __ldcg(pq + 1);
#pragma unroll
                            for (int i = 0; i < kC; ++i) vq[q][i] = __ldcg(pq + 4 + lane + 32 * i);
                        }
                    }
                    Mt = -INFINITY;
                    anybad = false;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        Mt = fmaxf(Mt, mq[q]);
                        anybad |= lq[q] < 0.f;
                    }
                    Lt = 0.f;
#pragma unroll
                    for (int i = 0; i < kC; ++i) o[i] = 0.f;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float f = mq[q] == -INFINITY ? 0.f : ptx::ex2(mq[q] - Mt);
                        Lt += f * lq[q];
#pragma unroll
                        for (int i = 0; i < kC; ++i) o[i] += f * vq[q][i];
                    }
                }
            }
            if (write) {
                const int h0 = kvh * p.group + qg * p.item_heads;
                float *dst = p.out + (static_cast<int64_t>(seq) * p.num_heads + h0 + h) * kD;
                const float inv = anybad ? 0.f : 1.f / Lt;
#pragma unroll
                for (int i = 0; i < kC; ++i) dst[lane + 32 * i] = anybad ? 0.f : o[i] * inv;
            }
        }
        __syncthreads();  // the shared partials are free for the next task
    }
}

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel on the stream drains; it calls griddepcontrol.wait
// before touching that kernel's results.
// cluster > 0: thread-block clusters of that many CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t st, int cluster, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster > 0 ? cluster : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 0 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// How many clusters of `cluster` CTAs of kern can be resident at once.
template <typename... KArgs>
int cluster_capacity(void (*kern)(KArgs...), size_t smem, int cluster)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// ------------------------------------------------------------------- host
struct DecodeCall {
    float *out;
    const void *query;
    const void *kpool;
    const void *vpool;
    const float *k_scales;
    const float *v_scales;
    int num_blocks;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    int max_context_len;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size;
    float softmax_scale;
    void *workspace;
    size_t workspace_bytes;
    int32_t *dev_status;
    void *stream;
};

struct Shape {
    int group, item_heads, qgroups, items_per_seq, rec_heads, ctx_cap;
    int64_t max_pages;  // upper bound of the page stream length
};

pkv_status check_shape(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                       int max_context_len, int max_blocks_per_seq, Shape *sh)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_context_len < 0 || max_blocks_per_seq < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    sh->group = num_heads / num_kv_heads;
    // a work item serves 8 query heads, or 16 (two groups of 8 sharing every
    // staged page) when a kv head has more than 8
    sh->item_heads = sh->group > kItemHeads ? 2 * kItemHeads : kItemHeads;
    sh->qgroups = (sh->group + sh->item_heads - 1) / sh->item_heads;
    const int64_t ips = static_cast<int64_t>(num_kv_heads) * sh->qgroups;
    if (ips > (1 << 20)) return PKV_ERR_UNSUPPORTED;
    sh->items_per_seq = static_cast<int>(ips);
    sh->rec_heads = sh->group < sh->item_heads ? sh->group : sh->item_heads;
    const int64_t cap_tab = static_cast<int64_t>(max_blocks_per_seq) * kPage;
    sh->ctx_cap = static_cast<int>(max_context_len < cap_tab ? max_context_len : cap_tab);
    const int64_t pages_per_seq = (sh->ctx_cap + kPage - 1) / kPage;
    if (static_cast<int64_t>(num_seqs) * pages_per_seq > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    sh->max_pages = static_cast<int64_t>(num_seqs) * pages_per_seq * ips;
    return PKV_OK;
}

// workspace: two partial records (first and last piece) for each of up to
// min(4096, pages) workers
size_t workspace_bytes_for(const Shape &sh, int head_dim)
{
    const int64_t workers = sh.max_pages < kMaxWorkers ? sh.max_pages : kMaxWorkers;
    return static_cast<size_t>(workers) * 2 * sh.rec_heads * (head_dim + 4) * sizeof(float);
}

struct OccCache {
    int device = -1;
    size_t smem = 0;
    int per_sm = 0;
};

// Resident clusters of `cl` CTAs with `smem` bytes each, recently asked.
struct ClusterCache {
    int device = -1;
    size_t smem = 0;
    int cl = 0;
    int clusters = 0;
};

template <int kKv, int kD, bool kLoCols, int kG>
pkv_status launch(const DecodeCall &call, const Shape &sh)
{
    using C = Cfg<kKv, kD>;
    DeviceInfo di;
    if (!current_device_info(&di)) return PKV_ERR_CUDA;
    const size_t smem = C::smem_bytes(call.num_seqs);
    if (smem > di.max_smem_optin) return PKV_ERR_UNSUPPORTED;
    auto kern = decode_kernel<kKv, kD, kLoCols, false, kG>;
    auto kern_cl = decode_kernel<kKv, kD, kLoCols, true, kG>;
    static OccCache occ[64];
    static size_t smem_attr[2][64] = {};  // dynamic shared memory each kernel may use, per device
    static ClusterCache ccache[8];
    static int ccache_next = 0;
    size_t smem_launch = smem;
    int per_sm = 0;
    int cap = 0;
    int clust = 0;
    {
        std::lock_guard<std::mutex> lock(g_cfg_mu);
        OccCache &oc = occ[di.device & 63];
        // raise a kernel's dynamic shared memory limit to what a launch needs
        auto allow = [&](auto k, int which, size_t bytes) -> bool {
            if (bytes <= smem_attr[which][di.device & 63]) return true;
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(bytes)) != cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            smem_attr[which][di.device & 63] = bytes;
            return true;
        };
        if (!allow(kern, 0, smem)) return PKV_ERR_CUDA;
        if (oc.device != di.device || oc.smem != smem) {
            int v = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kThreads, smem) !=
                cudaSuccess)
                return PKV_ERR_CUDA;
            oc.device = di.device;
            oc.smem = smem;
            oc.per_sm = v;
        }
        per_sm = oc.per_sm;
        cap = g_worker_cap;
        // One item per cluster when every item's cluster fits in one wave
        // (and no worker cap asks for the persistent partition): the
        // cluster's warps split the item's pages, about one stage each as
        // far as the wave allows, and merge through distributed shared
        // memory, with no reduce launch.
        const int64_t items = static_cast<int64_t>(call.num_seqs) * sh.items_per_seq;
        const int64_t resident = static_cast<int64_t>(per_sm) * di.num_sms;
        const int64_t stage_pages = static_cast<int64_t>(kWarps) * C::kPPS;
        const int64_t pages = (sh.ctx_cap + kPage - 1) / kPage;
        int64_t cl = (pages + stage_pages - 1) / stage_pages;
        // long items stream faster over the persistent workers, whose number
        // follows the pages rather than the items
        const bool cluster_ok = cl <= static_cast<int64_t>(kMaxClusterStages) * kMaxCluster;
        if (cl > kMaxCluster) cl = kMaxCluster;
        if (items > 0 && cl > resident / items) cl = resident / items;
        // the records pushed to a CTA take shared memory, so a smaller
        // cluster may be what fits in one wave: halve until it does
        for (; cap == 0 && cluster_ok && cl >= 1 && items * cl <= resident;
             cl = cl > 1 ? cl / 2 : 0) {
            const int hpc = static_cast<int>((sh.rec_heads + cl - 1) / cl);
            const size_t smem_cl = 1024 + C::crec_offset(call.num_seqs) +
                                   C::crec_bytes(static_cast<int>(cl) * kWarps, hpc);
            if (smem_cl > di.max_smem_optin || !allow(kern_cl, 1, smem_cl)) continue;
            int fit = -1;
            for (const ClusterCache &e : ccache)
                if (e.device == di.device && e.smem == smem_cl && e.cl == cl) fit = e.clusters;
            if (fit < 0) {
                fit = cluster_capacity(kern_cl, smem_cl, static_cast<int>(cl));
                ClusterCache &e = ccache[ccache_next];
                ccache_next = (ccache_next + 1) % 8;
                e.device = di.device;
                e.smem = smem_cl;
                e.cl = static_cast<int>(cl);
                e.clusters = fit;
            }
            if (fit >= items) {
                clust = static_cast<int>(cl);
                smem_launch = smem_cl;
                break;
            }
        }
    }
    if (per_sm <= 0) return PKV_ERR_UNSUPPORTED;
    int64_t workers = static_cast<int64_t>(per_sm) * di.num_sms * kWarps;
    if (C::kWarpsPerSm > 0 && workers > static_cast<int64_t>(C::kWarpsPerSm) * di.num_sms)
        workers = static_cast<int64_t>(C::kWarpsPerSm) * di.num_sms;
    if (workers > kMaxWorkers) workers = kMaxWorkers;
    if (cap > 0 && workers > cap) workers = cap;
    if (workers > sh.max_pages) workers = sh.max_pages;
    // at most kMaxWorkersPerItem workers per item, or one per
    // kMinPagesPerWorker pages if that is more: short items then split into a
    // few pieces (the reduce's fast path) rather than one page per warp, and
    // long items still spread over the whole grid
    const int64_t by_items =
        static_cast<int64_t>(kMaxWorkersPerItem) * call.num_seqs * sh.items_per_seq;
    const int64_t by_pages = sh.max_pages / kMinPagesPerWorker;
    const int64_t limit = by_items > by_pages ? by_items : by_pages;
    if (workers > limit) workers = limit;
    if (workers < 1) workers = 1;

    CUtensorMap tmk, tmv;
    const uint64_t rows = static_cast<uint64_t>(call.num_blocks) * call.num_kv_heads * kPage;
    if (!encode_tmap_2d(&tmk, call.kpool, C::kElem, kD, rows, C::kBoxInner, kPage, C::kSwizzle) ||
        !encode_tmap_2d(&tmv, call.vpool, C::kElem, kD, rows, C::kBoxInner, kPage, C::kSwizzle))
        return PKV_ERR_CUDA;

    DecodeArgs args;
    args.out = call.out;
    args.query = static_cast<const __half *>(call.query);
    args.block_tables = call.block_tables;
    args.context_lens = call.context_lens;
    args.k_scales = call.k_scales;
    args.v_scales = call.v_scales;
    args.partials = static_cast<float *>(call.workspace);
    args.dev_status = call.dev_status;
    args.num_seqs = call.num_seqs;
    args.num_heads = call.num_heads;
    args.num_kv_heads = call.num_kv_heads;
    args.group = sh.group;
    args.item_heads = sh.item_heads;
    args.qgroups = sh.qgroups;
    args.items_per_seq = sh.items_per_seq;
    args.rec_heads = sh.rec_heads;
    args.max_blocks_per_seq = call.max_blocks_per_seq;
    args.num_blocks = call.num_blocks;
    args.ctx_cap = sh.ctx_cap;
    args.num_workers = static_cast<int>(workers);
    args.clust = clust;
    args.scale_log2 = call.softmax_scale * 1.4426950408889634f;

    cudaStream_t st = static_cast<cudaStream_t>(call.stream);
    if (clust) {
        const int64_t items = static_cast<int64_t>(call.num_seqs) * sh.items_per_seq;
        args.num_workers = static_cast<int>(items * clust * kWarps);
        if (launch_pdl(kern_cl, static_cast<unsigned>(items * clust), kThreads, smem_launch, st, clust,
                       args, tmk, tmv) != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        return PKV_OK;
    }
    const unsigned grid = static_cast<unsigned>((workers + kWarps - 1) / kWarps);
    if (launch_pdl(kern, grid, kThreads, smem, st, 0, args, tmk, tmv) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (workers > 1) {
        const int64_t items = static_cast<int64_t>(call.num_seqs) * sh.items_per_seq;
        const int64_t tasks = items * sh.rec_heads;
        // items cut into more than eight pieces on average: CTAs per task
        // (their warps share the pieces); else a warp per task
        const int many = workers > 8 * items ? 1 : 0;
        const int rthreads = many ? kManyThreads : kRedThreads;
        int64_t rgrid = (tasks + kRedThreads / 32 - 1) / (kRedThreads / 32);
        const size_t rsmem = static_cast<size_t>(2 * call.num_seqs + 1) * sizeof(int32_t);
        const void *rk = many ? reinterpret_cast<const void *>(reduce_many_kernel<kD>)
                              : reinterpret_cast<const void *>(reduce_kernel<kD>);
        int red_per_sm = 0;
        {
            // the per-sequence tables of the largest batch, once per device
            // and kernel; a grid of at most one wave (tasks then loop)
            static int red_ready[64][2] = {};
            static size_t red_smem[64][2] = {};
            static int red_occ[64][2] = {};
            std::lock_guard<std::mutex> lock(g_cfg_mu);
            const int dv = di.device & 63;
            if (!red_ready[dv][many]) {
                if (cudaFuncSetAttribute(rk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>((2 * kMaxSeqs + 1) * sizeof(int32_t))) !=
                    cudaSuccess)
                    return PKV_ERR_CUDA;
                red_ready[dv][many] = 1;
                red_smem[dv][many] = ~size_t(0);
            }
            if (red_smem[dv][many] != rsmem) {
                int v = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, rk, rthreads, rsmem) !=
                    cudaSuccess)
                    return PKV_ERR_CUDA;
                red_smem[dv][many] = rsmem;
                red_occ[dv][many] = v;
            }
            red_per_sm = red_occ[dv][many];
        }
        const int64_t wave = static_cast<int64_t>(red_per_sm > 0 ? red_per_sm : 1) * di.num_sms;
        cudaError_t le;
        if (many) {
            // up to 8 CTAs per task, as many as one wave allows
            int split = 8;
            while (split > 1 && tasks * split > wave) split /= 2;
            int64_t groups = wave / split;
            if (groups > tasks) groups = tasks;
            if (groups < 1) groups = 1;
            le = launch_pdl(reduce_many_kernel<kD>, static_cast<unsigned>(groups * split),
                            kManyThreads, rsmem, st, 0, args, split);
        } else {
            if (rgrid > wave) rgrid = wave;
            le = launch_pdl(reduce_kernel<kD>, static_cast<unsigned>(rgrid), kRedThreads, rsmem, st,
                            0, args);
        }
        if (le != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
    }
    return PKV_OK;
}

pkv_status decode_entry(const DecodeCall &call, int kv)
{
    const bool int8 = kv != kKvF16;
    if (!call.out || !call.query || !call.kpool || !call.vpool || !call.block_tables ||
        !call.context_lens)
        return PKV_ERR_INVALID_ARG;
    if (int8 && (!call.k_scales || !call.v_scales)) return PKV_ERR_INVALID_ARG;
    if (call.num_blocks <= 0 || call.block_size <= 0) return PKV_ERR_INVALID_ARG;
    if (!(call.softmax_scale == call.softmax_scale) || call.softmax_scale > 3.0e38f ||
        call.softmax_scale < -3.0e38f)
        return PKV_ERR_INVALID_ARG;
    Shape sh;
    const pkv_status st = check_shape(call.num_seqs, call.num_heads, call.num_kv_heads,
                                      call.head_dim, call.max_context_len,
                                      call.max_blocks_per_seq, &sh);
    if (st != PKV_OK) return st;
    if (call.block_size != kPage) return PKV_ERR_UNSUPPORTED;
    if (call.num_seqs > kMaxSeqs) return PKV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(call.num_blocks) * call.num_kv_heads * kPage > 0x7fffffffLL)
        return PKV_ERR_UNSUPPORTED;
    if (!aligned(call.out, 16) || !aligned(call.query, 16) || !aligned(call.kpool, 16) ||
        !aligned(call.vpool, 16) || !aligned(call.block_tables, 4) ||
        !aligned(call.context_lens, 4) || (call.dev_status && !aligned(call.dev_status, 4)) ||
        (int8 && (!aligned(call.k_scales, 4) || !aligned(call.v_scales, 4))))
        return PKV_ERR_MISALIGNED;
    if (call.num_seqs == 0) return PKV_OK;
    const size_t need = workspace_bytes_for(sh, call.head_dim);
    if (need > 0 && (!call.workspace || call.workspace_bytes < need)) return PKV_ERR_WORKSPACE;
    if (call.workspace && !aligned(call.workspace, 16)) return PKV_ERR_MISALIGNED;
    // groups of at most four query heads carry the low parts of the
    // probabilities in the spare mma columns; above eight, a work item
    // serves two groups of eight from every staged page
    const int variant = sh.group <= 4 ? 0 : sh.item_heads > kItemHeads ? 2 : 1;
    auto pick = [&](auto lo, auto mid, auto two) -> pkv_status {
        return variant == 0 ? lo(call, sh) : variant == 1 ? mid(call, sh) : two(call, sh);
    };
    if (kv == kKvF8) {
        if (call.head_dim == 128)
            return pick(launch<kKvF8, 128, true, 1>, launch<kKvF8, 128, false, 1>,
                        launch<kKvF8, 128, false, 2>);
        return pick(launch<kKvF8, 64, true, 1>, launch<kKvF8, 64, false, 1>,
                    launch<kKvF8, 64, false, 2>);
    }
    if (kv == kKvI8) {
        if (call.head_dim == 128)
            return pick(launch<kKvI8, 128, true, 1>, launch<kKvI8, 128, false, 1>,
                        launch<kKvI8, 128, false, 2>);
        return pick(launch<kKvI8, 64, true, 1>, launch<kKvI8, 64, false, 1>,
                    launch<kKvI8, 64, false, 2>);
    }
    if (call.head_dim == 128)
        return pick(launch<kKvF16, 128, true, 1>, launch<kKvF16, 128, false, 1>,
                    launch<kKvF16, 128, false, 2>);
    return pick(launch<kKvF16, 64, true, 1>, launch<kKvF16, 64, false, 1>,
                launch<kKvF16, 64, false, 2>);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_decode_fp16(float *out, const void *query, const void *k_cache,
                                            const void *v_cache, int num_blocks,
                                            const int32_t *block_tables, int max_blocks_per_seq,
                                            const int32_t *context_lens, int max_context_len,
                                            int num_seqs, int num_heads, int num_kv_heads,
                                            int head_dim, int block_size, float softmax_scale,
                                            void *workspace, size_t workspace_bytes,
                                            int32_t *dev_status, void *stream)
{
    const pkv::DecodeCall call{out, query, k_cache, v_cache, nullptr, nullptr, num_blocks,
                               block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                               softmax_scale, workspace, workspace_bytes, dev_status, stream};
    return pkv::decode_entry(call, pkv::kKvF16);
}

extern "C" pkv_status pkv_paged_decode_int8(float *out, const void *query, const int8_t *k_codes,
                                            const int8_t *v_codes, const float *k_scales,
                                            const float *v_scales, int num_blocks,
                                            const int32_t *block_tables, int max_blocks_per_seq,
                                            const int32_t *context_lens, int max_context_len,
                                            int num_seqs, int num_heads, int num_kv_heads,
                                            int head_dim, int block_size, float softmax_scale,
                                            void *workspace, size_t workspace_bytes,
                                            int32_t *dev_status, void *stream)
{
    const pkv::DecodeCall call{out, query, k_codes, v_codes, k_scales, v_scales, num_blocks,
                               block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                               softmax_scale, workspace, workspace_bytes, dev_status, stream};
    return pkv::decode_entry(call, pkv::kKvI8);
}

extern "C" pkv_status pkv_paged_decode_fp8(float *out, const void *query, const uint8_t *k_codes,
                                           const uint8_t *v_codes, const float *k_scales,
                                           const float *v_scales, int num_blocks,
                                           const int32_t *block_tables, int max_blocks_per_seq,
                                           const int32_t *context_lens, int max_context_len,
                                           int num_seqs, int num_heads, int num_kv_heads,
                                           int head_dim, int block_size, float softmax_scale,
                                           void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, void *stream)
{
    const pkv::DecodeCall call{out, query, k_codes, v_codes, k_scales, v_scales, num_blocks,
                               block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                               softmax_scale, workspace, workspace_bytes, dev_status, stream};
    return pkv::decode_entry(call, pkv::kKvF8);
}

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                            int head_dim, int max_context_len)
{
    pkv::Shape sh;
    // the block table can hold any context up to max_context_len here
    const int mbps = (max_context_len + 15) / 16;
    if (pkv::check_shape(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len, mbps,
                         &sh) != PKV_OK)
        return 0;
    return pkv::workspace_bytes_for(sh, head_dim);
}

extern "C" pkv_status pkv_set_decode_workers(int max_workers)
{
    if (max_workers < 0) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(pkv::g_cfg_mu);
    pkv::g_worker_cap = max_workers;
    return PKV_OK;
}

// ------------------------------------------------- decode without allocation
// Scratch for pkv_paged_decode_int8_static_workspace: a fixed device array
// that every GPU loading this library holds until the process exits.  Only
// the partial records and split descriptors of the decode live here; they are
// fully rewritten by every call before they are read, so nothing needs to
// start at zero.  Host code must not pass `g_static_ws` itself to a kernel:
// on the host that name is a stand-in, not a device address.
static __device__ __align__(256) unsigned char g_static_ws[PKV_STATIC_WORKSPACE_BYTES];

namespace pkv {
namespace {
std::mutex g_static_mu;
void *g_static_ptr[64] = {};  // device address of g_static_ws, per device
}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_decode_int8_static_workspace(
    float *out, const void *query, const int8_t *k_codes, const int8_t *v_codes,
    const float *k_scales, const float *v_scales, int num_blocks, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, float softmax_scale,
    int32_t *dev_status, void *stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    void *ws = nullptr;
    {
        // set-up, once per device, with that device current
        std::lock_guard<std::mutex> lock(pkv::g_static_mu);
        if (!pkv::g_static_ptr[dev]) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) {
                cudaGetLastError();
                return PKV_ERR_CUDA;
            }
            pkv::g_static_ptr[dev] = ptr;
        }
        ws = pkv::g_static_ptr[dev];
    }
    const pkv::DecodeCall call{out, query, k_codes, v_codes, k_scales, v_scales, num_blocks,
                               block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                               softmax_scale, ws, PKV_STATIC_WORKSPACE_BYTES, dev_status, stream};
    // a call needing more than PKV_STATIC_WORKSPACE_BYTES of scratch is
    // rejected with PKV_ERR_WORKSPACE before anything is launched
    return pkv::decode_entry(call, pkv::kKvI8);
}

#ifdef PKV_DEBUG
// Debug builds only (not part of the C ABI header): the OR of the check bits
// set since the last reset (1: a shared-memory address outside the dynamic
// shared memory, 2: a misaligned one, 4: a table index out of range); reset
// nonzero clears them.  Synchronises with the device.
extern "C" __attribute__((visibility("default"))) unsigned int pkv_debug_flags(int reset)
{
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, pkv::g_debug_flags, sizeof(v)) != cudaSuccess)
        return 0xffffffffu;
    if (reset) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(pkv::g_debug_flags, &z, sizeof(z)) != cudaSuccess) return 0xffffffffu;
    }
    return v;
}

// Debug builds only: the limit of the decode kernel's waits for a stage, in
// ns, on the current device (0: a wait gives up at once, as if its limit had
// run out, while its copies are still in flight; the drain that follows a
// timeout keeps its 1 s limit).  Negative restores the default of 1 s.  Synchronises with the
// device; returns 0, or -1 if the CUDA runtime fails.
extern "C" __attribute__((visibility("default"))) int pkv_debug_set_stage_wait_ns(long long ns)
{
    const unsigned long long v =
        ns < 0 ? pkv::kWaitLimitNs : static_cast<unsigned long long>(ns);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyToSymbol(pkv::g_debug_stage_wait_ns, &v, sizeof(v)) != cudaSuccess)
        return -1;
    return 0;
}
#endif

/*
 * pkv.h -- C ABI of libpkv: decode-step paged attention over a
 * block-table-indexed KV cache, fp16, INT8 or FP8 (E4M3) KV, for NVIDIA GB300
 * (sm_103a), with the per-(block, kv head) INT8 and FP8 quantizers, the token
 * append that precedes a decode step, eviction scoring with the choice of the
 * blocks to evict, and a host block manager (free list, reference counts,
 * prefix sharing, copy-on-write) whose page copies run on the GPU.
 *
 * Sources for what each call computes:
 *  [PKF]  "PagedKV-Fusion" README (INT8 per-(block, head) quantized decode
 *         attention): Overview, component B; Architecture, the flowchart
 *         (symmetric INT8 per block and head; online softmax with GQA) and
 *         the sequence diagram (INT8 codes handed on with their scales; the
 *         decode step through the block table); Results, Memory footprint
 *         table.
 *  [PAR]  "paged-attention-runtime" summary: CORE CAPABILITIES 1 (16-token
 *         blocks) and 2 (block-table indirection, online softmax, FP32
 *         accumulation), 4 (GQA).
 *  [GLO]  "PagedAttention & KV-Cache Memory Management": section 2.1 (block
 *         table: block = table[t / B], slot = t % B; "Kernel Mechanics":
 *         token writes), 3.3.2 (appending tokens), 4.3.1 (least-reference-
 *         count + age eviction score), 4.1.1 (copy-on-write), 5.1 (per-block
 *         scaled FP8 KV).
 *
 * Layouts (all row-major, all pointers are DEVICE pointers owned by the
 * caller; the library never allocates, frees or synchronises).  A decode
 * call's query, block_tables, context_lens and out, and the quantizers'
 * block_ids, may also be pinned host memory (page-locked, e.g. from
 * cudaHostAlloc: one address for the host and the GPU), which the kernels
 * then read or write in place over the GPU's link to the host; KV pools,
 * scales and workspaces must be device memory:
 *   K/V pools      [num_blocks][num_kv_heads][block_size][head_dim]
 *                  (one contiguous tile per (block, kv head))
 *   scales         [num_blocks][num_kv_heads]  fp32, one for K, one for V
 *   query          [num_seqs][num_heads][head_dim]  fp16
 *   block_tables   [num_seqs][max_blocks_per_seq]   int32 physical ids
 *   context_lens   [num_seqs]                        int32
 *   out            [num_seqs][num_heads][head_dim]  fp32
 * Query head h attends with kv head h / (num_heads / num_kv_heads).
 * Supported: block_size 16; head_dim 64 or 128; any group size; decode
 * batches of up to 8192 sequences (PKV_ERR_UNSUPPORTED beyond).
 *
 * Errors.  Host-side argument errors are returned before anything is
 * launched.  Device-side data errors never trap: the affected outputs are
 * written as zeros and a bit is OR-ed into the optional caller-owned int32
 * *dev_status (device memory; the caller zeroes it).  Every wait inside a
 * kernel is bounded (about one second); a wait that runs out sets
 * PKV_DEV_TIMEOUT and the kernel returns.  Calls are asynchronous on the
 * given stream (NULL = the legacy default stream); a launch failure is
 * reported as PKV_ERR_CUDA.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* null pointer, negative size, heads not divisible, ... */
    PKV_ERR_UNSUPPORTED = 2, /* block_size != 16, head_dim not 64/128, size limits */
    PKV_ERR_MISALIGNED = 3,  /* a pointer misses its required alignment */
    PKV_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    PKV_ERR_EXHAUSTED = 6    /* block manager: not enough free blocks (or host
                                memory); nothing was changed */
} pkv_status;

/* Bits of *dev_status. */
#define PKV_DEV_BAD_BLOCK 1u /* a block id outside [0, num_blocks) was needed */
#define PKV_DEV_BAD_CTX 2u   /* context_lens[s] outside [0, max_context_len] or
                                beyond max_blocks_per_seq * block_size */
#define PKV_DEV_TIMEOUT 4u   /* a bounded wait for an asynchronous copy ran out */

/*
 * pkv_quantize_blocks -- symmetric per-(block, kv head) INT8 quantization
 * of fp16 K and V tiles ([PKF] Overview, component B; Architecture, sequence
 * diagram: INT8 codes handed on with their scales).
 *
 * For every listed block b and kv head h, separately for K and V, over all
 * block_size * head_dim values x of the tile (padding slots included):
 *   amax  = max |x| in fp32 (NaN values ignored)
 *   scale = amax / 127            (IEEE fp32 division)
 *   code  = round-half-to-even(x / scale) clamped to [-127, 127]
 *           (x / scale rounded to fp32 first; a NaN quotient -- 0/0, inf/inf,
 *           NaN input -- gives code 0)
 * Codes go to the same (b, h) tile of k_codes / v_codes, scales to
 * k_scales[b][h] / v_scales[b][h].  Results are bit-identical to the CPU
 * oracle of this repository.
 *
 *   k_fp16, v_fp16     const fp16 pools, 16-byte aligned
 *   k_codes, v_codes   int8 pools of the same shape, 16-byte aligned
 *   k_scales, v_scales fp32 [num_blocks][num_kv_heads], 4-byte aligned
 *   block_ids          device int32 [num_ids] or NULL for all blocks;
 *                      duplicates allowed (same result); ids outside
 *                      [0, num_blocks) are skipped and set PKV_DEV_BAD_BLOCK
 *   dev_status         optional device int32 (may be NULL)
 *   stream             cudaStream_t as void*
 */
PKV_API pkv_status pkv_quantize_blocks(const void *k_fp16, const void *v_fp16,
                               int8_t *k_codes, int8_t *v_codes,
                               float *k_scales, float *v_scales,
                               const int32_t *block_ids, int num_ids,
                               int num_blocks, int num_kv_heads, int head_dim,
                               int block_size, int32_t *dev_status,
                               void *stream);

/*
 * pkv_paged_decode_fp16 -- one decode step of paged attention over fp16 KV
 * ([PKF] Architecture, sequence diagram: the decode step through the block
 * table; [PAR] CORE CAPABILITIES 2 and 4; [GLO] section 2.1).
 *
 * For every sequence s (ctx = context_lens[s]) and query head h with kv head
 * kvh = h / (num_heads / num_kv_heads):
 *   K_t = k_cache[block_tables[s][t / 16]][kvh][t % 16][:]   (t < ctx)
 *   z_t = softmax_scale * <query[s][h], K_t>
 *   out[s][h] = sum_t softmax(z)_t * V_t      (FP32 accumulation)
 * ctx == 0 gives zeros.  Slots t >= ctx of the last block are never used
 * (they may hold anything, NaN included).  Table entries past the context
 * are never read.
 *
 *   out            fp32 [num_seqs][num_heads][head_dim], 16-byte aligned
 *   query          fp16, 16-byte aligned
 *   k_cache/v_cache fp16 pools, 16-byte aligned, num_blocks blocks
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   int32 [num_seqs]
 *   max_context_len host bound on every context_lens[s] (sizes the launch;
 *                  a larger length on the device is PKV_DEV_BAD_CTX)
 *   workspace      device scratch of at least pkv_decode_workspace_size()
 *                  bytes, 16-byte aligned; contents need no initialisation
 *                  and are overwritten
 *   dev_status     optional device int32 (may be NULL)
 * Two calls sharing a workspace must not overlap on the GPU.
 * num_seqs == 0 returns PKV_OK without launching.
 */
PKV_API pkv_status pkv_paged_decode_fp16(float *out, const void *query,
                                 const void *k_cache, const void *v_cache,
                                 int num_blocks, const int32_t *block_tables,
                                 int max_blocks_per_seq,
                                 const int32_t *context_lens,
                                 int max_context_len, int num_seqs,
                                 int num_heads, int num_kv_heads, int head_dim,
                                 int block_size, float softmax_scale,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream);

/*
 * pkv_paged_decode_int8 -- the same decode step over INT8 KV with one fp32
 * scale per (block, kv head) for K and one for V ([PKF] Overview component
 * B; Architecture, flowchart): K_t = k_codes[...] * k_scales[blk][kvh],
 * V_t = v_codes[...] * v_scales[blk][kvh], as produced by
 * pkv_quantize_blocks.  Arguments as for pkv_paged_decode_fp16, with
 *   k_codes/v_codes  int8 pools, 16-byte aligned
 *   k_scales/v_scales fp32 [num_blocks][num_kv_heads], 4-byte aligned
 */
PKV_API pkv_status pkv_paged_decode_int8(float *out, const void *query,
                                 const int8_t *k_codes, const int8_t *v_codes,
                                 const float *k_scales, const float *v_scales,
                                 int num_blocks, const int32_t *block_tables,
                                 int max_blocks_per_seq,
                                 const int32_t *context_lens,
                                 int max_context_len, int num_seqs,
                                 int num_heads, int num_kv_heads, int head_dim,
                                 int block_size, float softmax_scale,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream);

/*
 * pkv_quantize_blocks_fp8 -- pkv_quantize_blocks with FP8 codes: OCP E4M3
 * bytes (sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite 448) with one fp32 scale per (block, kv head)
 * for K and one for V ([GLO] section 5.1: per-block scaled FP8 keys and
 * values).  For every value x of the tile:
 *   scale = amax / 448 (IEEE fp32 division; amax = max |x|, NaN ignored)
 *   code  = the E4M3 value nearest to the fp32 quotient x / scale (ties to
 *           even), saturated to +-448; a NaN quotient gives code 0
 * Arguments as pkv_quantize_blocks, with uint8 code pools.  Bit-identical to
 * the CPU oracle of this repository.
 */
PKV_API pkv_status pkv_quantize_blocks_fp8(const void *k_fp16, const void *v_fp16,
                                           uint8_t *k_codes, uint8_t *v_codes,
                                           float *k_scales, float *v_scales,
                                           const int32_t *block_ids, int num_ids,
                                           int num_blocks, int num_kv_heads, int head_dim,
                                           int block_size, int32_t *dev_status, void *stream);

/*
 * pkv_paged_decode_fp8 -- the decode step over FP8 (E4M3) codes with per-
 * (block, kv head) scales, as produced by pkv_quantize_blocks_fp8:
 * K_t = e4m3(k_codes[...]) * k_scales[blk][kvh], V_t likewise.  Arguments as
 * pkv_paged_decode_int8 with uint8 code pools.
 */
PKV_API pkv_status pkv_paged_decode_fp8(float *out, const void *query,
                                        const uint8_t *k_codes, const uint8_t *v_codes,
                                        const float *k_scales, const float *v_scales,
                                        int num_blocks, const int32_t *block_tables,
                                        int max_blocks_per_seq, const int32_t *context_lens,
                                        int max_context_len, int num_seqs, int num_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        float softmax_scale, void *workspace,
                                        size_t workspace_bytes, int32_t *dev_status,
                                        void *stream);

/*
 * pkv_paged_decode_int8_static_workspace -- pkv_paged_decode_int8 for
 * callers that cannot allocate device memory.  This call has no counterpart
 * in the source pages: it serves code whose device memory is owned by some
 * other allocator (a framework pool that must see every allocation), and
 * code that cannot afford the implicit device synchronisation that
 * cudaMalloc / cudaFree may perform.  Such callers cannot provide the
 * workspace argument, so this variant uses a fixed scratch array of
 * PKV_STATIC_WORKSPACE_BYTES compiled into the library instead.
 *
 * Everything else -- arguments, layouts, results, error codes -- is as for
 * pkv_paged_decode_int8, without workspace / workspace_bytes.  The library
 * allocates nothing here (no cudaMalloc, no cudaFree, no allocating
 * library routine):
 *  - the scratch array is part of the library's device image, so every GPU
 *    that loads the library holds PKV_STATIC_WORKSPACE_BYTES until exit;
 *  - the first call on each device looks up the array's device address
 *    (with that device current); make that first call before any stream
 *    capture begins.  The address is kept for the life of the process, so
 *    resetting the device (cudaDeviceReset, or anything else that destroys
 *    its primary context) after that first call is not supported while the
 *    library stays loaded;
 *  - a call whose workspace requirement (pkv_decode_workspace_size) exceeds
 *    PKV_STATIC_WORKSPACE_BYTES returns PKV_ERR_WORKSPACE without launching;
 *  - all calls on a device share the one array: calls that can overlap on
 *    the GPU (different streams, no ordering between them) race and give
 *    wrong results.  The array needs no clearing: each call rewrites what it
 *    reads.
 */
#define PKV_STATIC_WORKSPACE_BYTES (32u << 20)

PKV_API pkv_status pkv_paged_decode_int8_static_workspace(
    float *out, const void *query, const int8_t *k_codes, const int8_t *v_codes,
    const float *k_scales, const float *v_scales, int num_blocks,
    const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size,
    float softmax_scale, int32_t *dev_status, void *stream);

/*
 * pkv_append_fp16 -- the KV write that precedes a decode step: for every
 * sequence s with t = positions[s] >= 0, row t % 16 of tile
 * (block_tables[s][t / 16], kv head h) of each pool is set to
 * k_new[s][h][:] / v_new[s][h][:], for every kv head h
 * ([GLO] section 2.1, Logical Token Blocks & Page Tables: block = table[t /
 * B], slot = t % B, and under Kernel Mechanics the write of a token to slot
 * phys_block_id * B + token_offset; section 3.3.2: new tokens are appended
 * to the cache).  A decode over context_lens[s] = t + 1 then attends to the
 * new token.
 *
 *   k_cache, v_cache  fp16 pools [num_blocks][num_kv_heads][16][head_dim],
 *                     written in place, 16-byte aligned
 *   k_new, v_new      fp16 [num_seqs][num_kv_heads][head_dim], 16-byte aligned
 *   block_tables      int32 [num_seqs][max_blocks_per_seq] (may be NULL when
 *                     max_blocks_per_seq is 0)
 *   positions         int32 [num_seqs]: token index of the new token; a
 *                     negative value means "no token for this sequence"
 * A position >= max_blocks_per_seq * 16 sets PKV_DEV_BAD_CTX, a table entry
 * outside [0, num_blocks) sets PKV_DEV_BAD_BLOCK; such a sequence writes
 * nothing.  The caller guarantees that no two appended tokens of one call
 * fall in the same physical block (a block shared by several sequences is
 * copied before it is written); otherwise the result is undefined.
 */
PKV_API pkv_status pkv_append_fp16(void *k_cache, void *v_cache, int num_blocks,
                                   const void *k_new, const void *v_new,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *positions, int num_seqs, int num_kv_heads,
                                   int head_dim, int block_size, int32_t *dev_status,
                                   void *stream);

/*
 * pkv_append_int8 -- pkv_append_fp16 for a cache kept as INT8 codes + scales
 * next to its fp16 pools: the new rows are written to the fp16 pools, and
 * every (block, kv head) tile that received a row is re-quantized into
 * k_codes/v_codes and k_scales/v_scales, bit-identical to
 * pkv_quantize_blocks on that block after the fp16 append (one fused kernel;
 * [PKF] Architecture, sequence diagram: INT8 codes with their scales).  All 16 slots of the
 * tile are quantized, as pkv_quantize_blocks does.  Extra arguments:
 *   k_codes, v_codes   int8 pools, 16-byte aligned
 *   k_scales, v_scales fp32 [num_blocks][num_kv_heads], 4-byte aligned
 */
PKV_API pkv_status pkv_append_int8(void *k_cache, void *v_cache, int8_t *k_codes,
                                   int8_t *v_codes, float *k_scales, float *v_scales,
                                   int num_blocks, const void *k_new, const void *v_new,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *positions, int num_seqs, int num_kv_heads,
                                   int head_dim, int block_size, int32_t *dev_status,
                                   void *stream);

/*
 * pkv_append_fp8 -- pkv_append_int8 for an FP8 (E4M3) cache: the written
 * tiles are re-quantized as pkv_quantize_blocks_fp8 would (bit-identical).
 * uint8 code pools; otherwise as pkv_append_int8.
 */
PKV_API pkv_status pkv_append_fp8(void *k_cache, void *v_cache, uint8_t *k_codes,
                                  uint8_t *v_codes, float *k_scales, float *v_scales,
                                  int num_blocks, const void *k_new, const void *v_new,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *positions, int num_seqs, int num_kv_heads,
                                  int head_dim, int block_size, int32_t *dev_status,
                                  void *stream);

/*
 * pkv_evict_select -- score every physical block for eviction and choose
 * the k most evictable ones, in one launch ([PKF] Overview, component A:
 * eviction scoring of the paged KV blocks fused with the top-k choice;
 * Architecture, sequence diagram: every physical block scored, the ids to
 * evict handed back).  The score is the
 * least-reference-count + age heuristic of [GLO] section 4.3.1:
 *   score[b] = alpha * (max_refcnt - refcnt[b]) + beta * (current_tick - last_used[b])
 * evaluated in fp32, one rounding per operation, each difference formed
 * exactly in integers and rounded to fp32; max_refcnt = max over b of
 * refcnt[b].  A block with refcnt[b] <= 0 is free: it gets score -inf and is
 * never chosen.  A NaN score (inf - inf with extreme weights) counts as -inf.
 * The chosen blocks are the min(k, number of candidates) with the largest
 * scores, equal scores going to the smaller block id; they are written to
 * evict_ids[0 .. n) in ascending block-id order, n to *num_evicted, and -1
 * to evict_ids[n .. k).  The [GLO] page gives alpha = 0.7, beta = 0.3.
 *
 *   refcnt       int32 [num_blocks], device; 4-byte aligned
 *   last_used    int64 [num_blocks], device (ticks); 8-byte aligned
 *   current_tick the present tick; every current_tick - last_used[b] must
 *                fit in int64
 *   alpha, beta  finite weights (else PKV_ERR_INVALID_ARG)
 *   k            >= 0, blocks to choose
 *   scores       optional fp32 [num_blocks] output (NULL: not written)
 *   evict_ids    int32 [k] output (may be NULL when k == 0)
 *   num_evicted  int32 device output
 * num_blocks may be at most 16 * 49152 (786432) on a device that schedules
 * 16-CTA clusters, else 8 * 49152; larger pools give PKV_ERR_UNSUPPORTED.
 */
PKV_API pkv_status pkv_evict_select(const int32_t *refcnt, const int64_t *last_used,
                                    int num_blocks, int64_t current_tick, float alpha,
                                    float beta, int k, float *scores, int32_t *evict_ids,
                                    int32_t *num_evicted, void *stream);

/*
 * Block manager -- host-side bookkeeping of the physical KV blocks
 * ([PAR] CORE CAPABILITIES 1: fixed 16-token blocks, free-list allocator,
 * reference counting, prefix sharing, copy-on-write, fragmentation metrics;
 * [GLO] the prefix-sharing block allocator and section 4.1.1: page-level
 * reference counts; a shared page that diverges gets a fresh page and a
 * copy).  Host memory only; the handle is opaque and every call locks it, so
 * one manager may be used from several threads.  A failing call changes
 * nothing.
 *
 *  - Blocks are numbered 0 .. num_blocks-1.  The free list is a stack: a
 *    fresh manager hands out 0, 1, 2, ...; a freed block is handed out next.
 *  - pkv_bm_allocate: one block per entry of hashes[0..n) (hashes NULL: all
 *    0).  A nonzero hash already registered shares that block (its count + 1);
 *    any other entry takes a free block with count 1, fill 0, and registers a
 *    nonzero hash.  PKV_ERR_EXHAUSTED if the free list cannot serve every
 *    entry that needs a fresh block.  Ids go to out_ids[0..n).
 *  - pkv_bm_free: one reference dropped per entry; a block reaching count 0
 *    loses its hash and fill and returns to the free list.
 *    PKV_ERR_INVALID_ARG if an id is not in use or listed more often than
 *    its count.
 *  - pkv_bm_fork: one reference added per entry (another sequence or beam
 *    now points at the block).
 *  - pkv_bm_cow: for each id in order, the block to write into: the block
 *    itself if its count is 1 (it loses any hash registration, its contents
 *    are about to change), else a fresh block that takes one reference from
 *    the shared one, with its fill; out_ids[i] gets it, and each
 *    (source, fresh) pair is appended to copy_pairs (int32 [n][2], may be
 *    NULL) for pkv_copy_blocks; *num_copies gets their number.
 *    PKV_ERR_EXHAUSTED if not enough free blocks.
 *  - pkv_bm_set_fill: tokens held by each block (0 .. block_size).
 *  - pkv_bm_stats: free, used (count > 0), shared (count > 1) and logical
 *    (sum of counts) blocks, tokens in used blocks, internal fragmentation
 *    1 - tokens / (used * block_size), sharing saving 1 - used / logical.
 *  - pkv_bm_refcounts: every block's count (host int32 [num_blocks]), the
 *    refcnt input of pkv_evict_select.
 */
typedef struct pkv_block_manager pkv_block_manager;

typedef struct pkv_bm_stats_t {
    int64_t free_blocks, used_blocks, shared_blocks, logical_blocks, tokens;
    double internal_fragmentation, sharing_saving;
} pkv_bm_stats_t;

PKV_API pkv_status pkv_bm_create(int num_blocks, int block_size, pkv_block_manager **out);
PKV_API void pkv_bm_destroy(pkv_block_manager *bm);
PKV_API pkv_status pkv_bm_allocate(pkv_block_manager *bm, const uint64_t *hashes, int n,
                                   int32_t *out_ids);
PKV_API pkv_status pkv_bm_free(pkv_block_manager *bm, const int32_t *ids, int n);
PKV_API pkv_status pkv_bm_fork(pkv_block_manager *bm, const int32_t *ids, int n);
PKV_API pkv_status pkv_bm_cow(pkv_block_manager *bm, const int32_t *ids, int n,
                              int32_t *out_ids, int32_t *copy_pairs, int *num_copies);
PKV_API pkv_status pkv_bm_set_fill(pkv_block_manager *bm, const int32_t *ids,
                                   const int32_t *tokens, int n);
PKV_API pkv_status pkv_bm_stats(pkv_block_manager *bm, pkv_bm_stats_t *out);
PKV_API pkv_status pkv_bm_refcounts(pkv_block_manager *bm, int32_t *out, int n);

/*
 * pkv_copy_blocks -- the copies that copy-on-write asks for ([GLO] section
 * 4.1.1), batched: for every pair (pairs[i][0] = source, pairs[i][1] =
 * destination block), the block's bytes in every pool are copied.
 *
 *   pools        host array of num_pools (<= 8) device pointers, each a pool
 *                laid out [num_blocks][...] with block_bytes[p] bytes per
 *                block (K and V pools: num_kv_heads * 16 * head_dim * element
 *                size; INT8 scales: num_kv_heads * 4); 4-byte aligned, block
 *                sizes multiples of 4 (16-byte units where both allow)
 *   pairs        device int32 [num_pairs][2]
 * A pair naming a block outside [0, num_blocks) sets PKV_DEV_BAD_BLOCK and is
 * skipped; a pair with source == destination is a no-op.  Destinations must
 * be distinct and must not be sources of the same call.
 */
PKV_API pkv_status pkv_copy_blocks(void *const *pools, const int64_t *block_bytes,
                                   int num_pools, int num_blocks, const int32_t *pairs,
                                   int num_pairs, int32_t *dev_status, void *stream);

/*
 * Bytes of workspace a decode call with these sizes needs (any KV variant).
 * Pure host arithmetic: no CUDA call.  Returns 0 for invalid sizes.
 */
PKV_API size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int max_context_len);

/*
 * Tuning and test control: cap the number of decode workers (one worker =
 * one warp streaming a contiguous range of KV pages; each range ends in a
 * partial result that the split-context reduce merges).  0 restores the
 * automatic choice: every resident warp of the device (seven per SM for fp16
 * KV at head_dim 128, ten at 64), and no more than the larger of four per
 * work item and one per eight pages of the longest possible page stream.  A
 * cap also selects the persistent workers for batches that would otherwise
 * run one item per thread-block cluster.  Process-wide.
 */
PKV_API pkv_status pkv_set_decode_workers(int max_workers);

/* Static description of a status code. */
PKV_API const char *pkv_status_string(pkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */

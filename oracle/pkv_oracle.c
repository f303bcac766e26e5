/*
 * pkv_oracle.c -- plain CPU oracle for paged decode attention and for the
 * per-(block, kv-head) symmetric INT8 quantizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package smoke check and the timed CPU
 * baseline of the benchmark use it.  It shares no source, header, table or
 * helper with the CUDA library; the two only ever see the same seeded inputs.
 *
 * What it computes, and where that is defined:
 *
 *  - pkv_oracle_decode: single-query attention for every (sequence, query
 *    head), gathering K and V token by token through the block table, then a
 *    dense max-subtracted softmax and a weighted sum of V, all in fp64.
 *      * block-table address translation: physical block = table[t / B],
 *        slot = t % B ("PagedAttention & KV-Cache Memory Management",
 *        section 2.1 "Logical Token Blocks & Page Tables");
 *      * softmax attention with FP32-or-better accumulation, GQA head groups
 *        ("paged-attention-runtime" summary, "CORE CAPABILITIES" 2 and 4;
 *        PagedKV-Fusion README, "Architecture", component B "online softmax
 *        . GQA").  The online (streaming) softmax of the kernels is an exact
 *        reformulation of this dense softmax, so the oracle uses the dense
 *        form, which is the plain definition.
 *      * INT8 KV: value = code * scale with one fp32 scale per (block,
 *        kv-head) for K and one for V (PagedKV-Fusion README, "Overview",
 *        component B, and the "Memory footprint" table whose exact MiB
 *        figures fix that granularity).
 *
 *  - pkv_oracle_quantize: per (block, kv-head) tile of B x d fp16 values,
 *    amax = max |x| in fp32, scale = amax / 127 (fp32 division),
 *    code = round-half-to-even(x / scale) clamped to [-127, 127]
 *    (PagedKV-Fusion README, "Overview" component B and "Architecture":
 *    "per-block,head symmetric INT8").  The pages say "symmetric" only; the
 *    absmax/127 scale, the rounding mode and the NaN rules are the readings
 *    this project adopts (they are listed with the other readings in the
 *    design notes).  Computed in fp32 so that codes and scales can be
 *    compared bit for bit.
 *
 *  - FP8 KV ("PagedAttention & KV-Cache Memory Management", section 5.1:
 *    per-block scaled FP8 keys and values, scale_k / scale_v per block):
 *    pkv_oracle_e4m3_to_double decodes an OCP E4M3 byte (sign, 4 exponent
 *    bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,
 *    largest finite 448); pkv_oracle_e4m3_from_float rounds an fp32 number
 *    to the nearest finite E4M3 value (ties to the code with an even last
 *    bit), saturating at +-448; pkv_oracle_quantize_fp8
 *    quantizes a tile with scale = amax / 448 exactly as the INT8 quantizer
 *    does with 127 (a NaN quotient gives code 0).
 *
 *  - pkv_oracle_append: the write that precedes a decode step.  The new
 *    token of sequence s sits at position t = positions[s]; its K and V rows
 *    (one per kv head) go to slot t % B of physical block table[s][t / B]
 *    -- the inverse of the decode gather ("PagedAttention & KV-Cache Memory
 *    Management", section 2.1, and its prefill step that writes each token
 *    at phys_block_id * B + token_offset; section 3.3.2 "append the delta
 *    tokens").  Plain row copies of fp16 bit patterns, one sequence after
 *    another.  The INT8 cache re-quantizes the written (block, kv-head) tiles
 *    with pkv_oracle_quantize afterwards (done by the Python wrapper).
 *
 *  - pkv_oracle_evict_scores / pkv_oracle_evict_select: the
 *    least-reference-count + age eviction score of "PagedAttention &
 *    KV-Cache Memory Management", section 4.3.1,
 *      score = alpha * (max_refcnt - refcnt) + beta * (current_tick - last_used),
 *    evaluated in fp32 one rounding per operation, and the choice of the k
 *    blocks to evict ("PagedKV-Fusion" README: scoring of every physical
 *    block, then the eviction ids).  Blocks with refcnt <= 0 are free and are
 *    not candidates; max_refcnt is the largest refcnt present.  A larger
 *    score means more evictable; equal scores go to the smaller block id.
 *
 * Conventions shared with the library (by specification, not by code):
 *   pools    [num_blocks][num_kv_heads][block_size][head_dim]
 *   scales   [num_blocks][num_kv_heads]
 *   query    [num_seqs][num_heads][head_dim]        (fp16 bit patterns)
 *   tables   [num_seqs][max_blocks_per_seq]         (int32)
 *   out      [num_seqs][num_heads][head_dim]        (fp64 here)
 *   q head h reads kv head h / (num_heads / num_kv_heads).
 * Per-(seq, head) flags: bit 0 = a block id outside [0, num_blocks) was
 * needed, bit 1 = the context length is outside [0, min(max_context_len,
 * max_blocks_per_seq * block_size)].  A flagged (seq, head) outputs zeros;
 * context length 0 outputs zeros with no flag.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BAD_BLOCK 1u
#define ORACLE_BAD_CTX 2u

/* IEEE binary16 bit pattern -> exact double (every half is a double). */
double pkv_oracle_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(mant | 0x400), expo - 25); /* 1.mant * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Exact value of an E4M3 byte: (8 + m) * 2^(e - 10) for e > 0, m * 2^-9 for
   e == 0; NaN for exponent and mantissa all ones. */
double pkv_oracle_e4m3_to_double(uint8_t c)
{
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* Nearest finite E4M3 code of a non-NaN fp32 value; ties go to the code
   with an even last bit; magnitudes beyond 448 give +-448.  The grid: below
   2^-6 the step is 2^-9 (subnormals, code = multiple of the step); in the
   binade [2^E, 2^(E+1)) the step is 2^(E-3), code = (E + 7) << 3 | (q - 8)
   with q = a / 2^(E-3) in [8, 16).  q is rounded to nearest-even in double
   (a and the power-of-two scaling are exact). */
uint8_t pkv_oracle_e4m3_from_float(float y)
{
    const int sign = signbit(y) ? 1 : 0;
    const double a = fabs((double)y);
    int code;
    if (a > 448.0) {
        code = 0x7E;
    } else if (a < ldexp(1.0, -6)) {
        code = (int)nearbyint(ldexp(a, 9)); /* 0 .. 8; 8 is 2^-6, the first normal */
    } else {
        int k;
        (void)frexp(a, &k);                 /* a = f * 2^k, f in [0.5, 1) */
        int e = k - 1;                      /* a in [2^e, 2^(e+1)) */
        int q = (int)nearbyint(ldexp(a, 3 - e));
        if (q == 16) {                      /* rounded up into the next binade */
            q = 8;
            ++e;
        }
        code = ((e + 7) << 3) | (q - 8);
        if (code > 0x7E) code = 0x7E;       /* 464 and up saturate */
    }
    return (uint8_t)((sign << 7) | code);
}

/* One element of K or V for token slot `slot` of physical block `blk`. */
static double kv_element(int kv_kind, const void *pool, const float *scales,
                         int64_t blk, int kvh, int slot, int i,
                         int num_kv_heads, int block_size, int head_dim)
{
    const int64_t tile = blk * num_kv_heads + kvh;
    const int64_t idx = (tile * block_size + slot) * head_dim + i;
    if (kv_kind == 0) {
        return pkv_oracle_half_to_double(((const uint16_t *)pool)[idx]);
    }
    if (kv_kind == 2) {
        return pkv_oracle_e4m3_to_double(((const uint8_t *)pool)[idx]) * (double)scales[tile];
    }
    return (double)((const int8_t *)pool)[idx] * (double)scales[tile];
}

/*
 * kv_kind 0: kpool/vpool are fp16 bit patterns, kscale/vscale ignored.
 * kv_kind 1: kpool/vpool are int8 codes, kscale/vscale fp32 per tile.
 * flags: optional [num_seqs][num_heads] output (may be NULL).
 * Returns 0, or -1 on an argument the oracle cannot interpret.
 */
int pkv_oracle_decode(double *out, const uint16_t *query, int kv_kind,
                      const void *kpool, const void *vpool,
                      const float *kscale, const float *vscale,
                      const int32_t *block_tables, const int32_t *context_lens,
                      int num_seqs, int num_heads, int num_kv_heads,
                      int head_dim, int block_size, int max_blocks_per_seq,
                      int64_t num_blocks, int max_context_len,
                      double softmax_scale, int num_threads, uint32_t *flags)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_seq < 0 || kv_kind < 0 || kv_kind > 2) {
        return -1;
    }
    const int group = num_heads / num_kv_heads;
    const int64_t pairs = (int64_t)num_seqs * num_heads;
    int64_t ctx_cap = (int64_t)max_blocks_per_seq * block_size;
    if (max_context_len < ctx_cap) ctx_cap = max_context_len;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel
    {
        int cap = 0;
        double *z = NULL; /* scores of one (seq, head) */
#pragma omp for schedule(dynamic, 1)
        for (int64_t pair = 0; pair < pairs; ++pair) {
            const int s = (int)(pair / num_heads);
            const int h = (int)(pair % num_heads);
            const int kvh = h / group;
            double *o = out + pair * head_dim;
            const uint16_t *qv = query + pair * head_dim;
            const int ctx = context_lens[s];
            uint32_t flag = 0;
            for (int i = 0; i < head_dim; ++i) o[i] = 0.0;

            if (ctx < 0 || ctx > ctx_cap) flag |= ORACLE_BAD_CTX;
            /* every block the context needs must be a real block */
            for (int t = 0; !flag && t < ctx; t += block_size) {
                const int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                if (blk < 0 || blk >= num_blocks) flag |= ORACLE_BAD_BLOCK;
            }
            if (flags) flags[pair] = flag;
            if (flag || ctx == 0) continue;

            if (ctx > cap) {
                free(z);
                cap = ctx;
                z = (double *)malloc(sizeof(double) * (size_t)cap);
            }
            /* scores z_t = softmax_scale * <q, K_t> over the gathered keys */
            for (int t = 0; t < ctx; ++t) {
                const int64_t blk = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                const int slot = t % block_size;
                double dot = 0.0;
                for (int i = 0; i < head_dim; ++i) {
                    const double qi = pkv_oracle_half_to_double(qv[i]);
                    const double ki = kv_element(kv_kind, kpool, kscale, blk, kvh, slot, i,
                                                 num_kv_heads, block_size, head_dim);
                    dot += qi * ki;
                }
                z[t] = softmax_scale * dot;
            }
            /* softmax weights w_t = exp(z_t - max z) / sum exp(z - max z) */
            double zmax = z[0];
            for (int t = 1; t < ctx; ++t) if (z[t] > zmax) zmax = z[t];
            double denom = 0.0;
            for (int t = 0; t < ctx; ++t) {
                z[t] = exp(z[t] - zmax);
                denom += z[t];
            }
            /* out = sum_t w_t V_t */
            for (int t = 0; t < ctx; ++t) {
                const int64_t blk = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
                const int slot = t % block_size;
                const double w = z[t] / denom;
                for (int i = 0; i < head_dim; ++i) {
                    o[i] += w * kv_element(kv_kind, vpool, vscale, blk, kvh, slot, i,
                                           num_kv_heads, block_size, head_dim);
                }
            }
        }
        free(z);
    }
    return 0;
}

/* Quantize one tile of n fp16 values (bit patterns) into codes + scale. */
static void quantize_tile(int8_t *codes, float *scale_out, const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t e = 0; e < n; ++e) {
        const float a = fabsf((float)pkv_oracle_half_to_double(x[e]));
        if (a > amax) amax = a; /* NaN never compares greater: ignored */
    }
    const float scale = amax / 127.0f;
    for (int64_t e = 0; e < n; ++e) {
        const float v = (float)pkv_oracle_half_to_double(x[e]);
        const float y = v / scale; /* 0/0 and inf/inf give NaN -> code 0 */
        int c = 0;
        if (!isnan(y)) {
            float r = nearbyintf(y); /* default rounding: to nearest, ties to even */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            c = (int)r;
        }
        codes[e] = (int8_t)c;
    }
    *scale_out = scale;
}

/* FP8 version of quantize_tile: scale = amax / 448, code = E4M3 of x / scale. */
static void quantize_tile_fp8(uint8_t *codes, float *scale_out, const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t e = 0; e < n; ++e) {
        const float a = fabsf((float)pkv_oracle_half_to_double(x[e]));
        if (a > amax) amax = a; /* NaN never compares greater: ignored */
    }
    const float scale = amax / 448.0f;
    for (int64_t e = 0; e < n; ++e) {
        const float v = (float)pkv_oracle_half_to_double(x[e]);
        const float y = v / scale; /* 0/0 and inf/inf give NaN -> code 0 */
        codes[e] = isnan(y) ? 0 : pkv_oracle_e4m3_from_float(y);
    }
    *scale_out = scale;
}

int64_t pkv_oracle_quantize_fp8(uint8_t *code_pool, float *scales, const uint16_t *pool,
                                const int32_t *block_ids, int64_t num_ids, int64_t num_blocks,
                                int num_kv_heads, int block_size, int head_dim)
{
    if (num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0) return -1;
    const int64_t tile_elems = (int64_t)block_size * head_dim;
    const int64_t count = block_ids ? num_ids : num_blocks;
    int64_t bad = 0;
    for (int64_t j = 0; j < count; ++j) {
        const int64_t blk = block_ids ? block_ids[j] : j;
        if (blk < 0 || blk >= num_blocks) {
            ++bad;
            continue;
        }
        for (int kvh = 0; kvh < num_kv_heads; ++kvh) {
            const int64_t tile = blk * num_kv_heads + kvh;
            quantize_tile_fp8(code_pool + tile * tile_elems, scales + tile,
                              pool + tile * tile_elems, tile_elems);
        }
    }
    return bad;
}

/*
 * Quantize the tiles (block_ids[j], kv-head) of one fp16 pool.
 * block_ids == NULL means every block 0..num_blocks-1 in order.
 * Codes and scales are written at the same (block, kv-head) positions of
 * code_pool [num_blocks][num_kv_heads][block_size][head_dim] and
 * scales [num_blocks][num_kv_heads].  Returns the number of ids outside
 * [0, num_blocks) (those are skipped), or -1 on bad arguments.
 */
int64_t pkv_oracle_quantize(int8_t *code_pool, float *scales, const uint16_t *pool,
                            const int32_t *block_ids, int64_t num_ids,
                            int64_t num_blocks, int num_kv_heads, int block_size,
                            int head_dim)
{
    if (num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0) return -1;
    const int64_t tile_elems = (int64_t)block_size * head_dim;
    const int64_t count = block_ids ? num_ids : num_blocks;
    int64_t bad = 0;
    for (int64_t j = 0; j < count; ++j) {
        const int64_t blk = block_ids ? block_ids[j] : j;
        if (blk < 0 || blk >= num_blocks) {
            ++bad;
            continue;
        }
        for (int kvh = 0; kvh < num_kv_heads; ++kvh) {
            const int64_t tile = blk * num_kv_heads + kvh;
            quantize_tile(code_pool + tile * tile_elems, scales + tile,
                          pool + tile * tile_elems, tile_elems);
        }
    }
    return bad;
}

/*
 * Append one token per sequence into fp16 pools (bit patterns).
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim]
 *   positions     [num_seqs]: token index of the new token; < 0 = no token
 *   flags         optional [num_seqs] output: ORACLE_BAD_CTX when the
 *                 position is beyond max_blocks_per_seq * block_size,
 *                 ORACLE_BAD_BLOCK when table[s][t / B] is not in
 *                 [0, num_blocks); a flagged sequence writes nothing.
 *   written_blocks optional [num_seqs] output: the physical block written,
 *                 or -1.
 * Returns the number of flagged sequences, or -1 on bad arguments.
 */
int64_t pkv_oracle_append(uint16_t *kpool, uint16_t *vpool, const uint16_t *k_new,
                          const uint16_t *v_new, const int32_t *block_tables,
                          const int32_t *positions, int num_seqs, int num_kv_heads,
                          int head_dim, int block_size, int max_blocks_per_seq,
                          int64_t num_blocks, uint32_t *flags, int32_t *written_blocks)
{
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_seq < 0 || num_blocks < 0) {
        return -1;
    }
    int64_t bad = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int64_t t = positions[s];
        uint32_t flag = 0;
        int64_t blk = -1;
        if (t >= (int64_t)max_blocks_per_seq * block_size) {
            flag = ORACLE_BAD_CTX;
        } else if (t >= 0) {
            blk = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
            if (blk < 0 || blk >= num_blocks) flag = ORACLE_BAD_BLOCK;
        }
        if (flags) flags[s] = flag;
        if (flag) {
            ++bad;
            blk = -1;
        }
        if (written_blocks) written_blocks[s] = (int32_t)blk;
        if (blk < 0) continue;
        const int slot = (int)(t % block_size);
        for (int kvh = 0; kvh < num_kv_heads; ++kvh) {
            const int64_t dst = (((blk * num_kv_heads) + kvh) * block_size + slot) * head_dim;
            const int64_t src = ((int64_t)s * num_kv_heads + kvh) * head_dim;
            for (int i = 0; i < head_dim; ++i) {
                kpool[dst + i] = k_new[src + i];
                vpool[dst + i] = v_new[src + i];
            }
        }
    }
    return bad;
}

/*
 * Eviction scores of num_blocks physical blocks, fp32, one rounding per
 * operation (the file is built without FMA contraction):
 *   d_ref = (float)(max_refcnt - refcnt[b])          exact int64 difference
 *   d_age = (float)(current_tick - last_used[b])     exact int64 difference
 *   score = alpha * d_ref + beta * d_age
 * max_refcnt = the largest refcnt[b] (0 if none is positive).  Free blocks
 * (refcnt <= 0) get -inf; a NaN score (inf - inf) is stored as -inf too.
 * Returns the number of candidate (refcnt > 0) blocks.
 */
int64_t pkv_oracle_evict_scores(float *scores, const int32_t *refcnt, const int64_t *last_used,
                                int64_t num_blocks, int64_t current_tick, float alpha,
                                float beta)
{
    int32_t max_ref = 0;
    int64_t candidates = 0;
    for (int64_t b = 0; b < num_blocks; ++b) {
        if (refcnt[b] > max_ref) max_ref = refcnt[b];
        if (refcnt[b] > 0) ++candidates;
    }
    for (int64_t b = 0; b < num_blocks; ++b) {
        if (refcnt[b] <= 0) {
            scores[b] = -INFINITY;
            continue;
        }
        const float d_ref = (float)((int64_t)max_ref - refcnt[b]);
        const float d_age = (float)(current_tick - last_used[b]);
        const float a = alpha * d_ref;
        const float c = beta * d_age;
        float sc = a + c;
        if (isnan(sc)) sc = -INFINITY;
        scores[b] = sc;
    }
    return candidates;
}

typedef struct {
    float score;
    int32_t id;
} evict_entry;

/* Descending score, then ascending block id. */
static int evict_order(const void *pa, const void *pb)
{
    const evict_entry *a = (const evict_entry *)pa, *b = (const evict_entry *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

static int id_order(const void *pa, const void *pb)
{
    const int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * The k blocks to evict: sort the candidates (refcnt > 0) by score,
 * largest first, equal scores by smaller id, keep the first min(k, count),
 * and return them in ascending block-id order in evict_ids[0..n).
 * Returns n, or -1 on bad arguments / allocation failure.
 */
int64_t pkv_oracle_evict_select(int32_t *evict_ids, const float *scores, const int32_t *refcnt,
                                int64_t num_blocks, int64_t k)
{
    if (num_blocks < 0 || k < 0) return -1;
    evict_entry *c = (evict_entry *)malloc(sizeof(evict_entry) * (size_t)(num_blocks + 1));
    if (!c) return -1;
    int64_t n = 0;
    for (int64_t b = 0; b < num_blocks; ++b) {
        if (refcnt[b] > 0) {
            c[n].score = scores[b];
            c[n].id = (int32_t)b;
            ++n;
        }
    }
    qsort(c, (size_t)n, sizeof(evict_entry), evict_order);
    if (k < n) n = k;
    for (int64_t j = 0; j < n; ++j) evict_ids[j] = c[j].id;
    free(c);
    qsort(evict_ids, (size_t)n, sizeof(int32_t), id_order);
    return n;
}

/* Threads the OpenMP runtime will use for a parallel region (1 without OpenMP). */
int pkv_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * The C ABI from plain C99: include/pkv.h compiled by a C compiler and
 * libpkv.so linked by the system linker, calling only what needs no GPU:
 * status strings, workspace arithmetic, the host-side argument checks of the
 * decode, quantize and append entry points (rejected before any CUDA call),
 * calls with nothing to do, and the host block manager.  Prints one "ok"
 * line per check and exits 0, or prints the failed check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pkv.h"

static int failures = 0;

static void check(int cond, const char *what)
{
    printf("%s %s\n", cond ? "ok" : "FAILED", what);
    if (!cond) ++failures;
}

/* aligned, never dereferenced: every call below returns before using it */
#define FAKE ((void *)(uintptr_t)0x10000)

int main(void)
{
    /* status strings: one for every code */
    const pkv_status codes[] = {PKV_OK,           PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED,
                                PKV_ERR_MISALIGNED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA,
                                PKV_ERR_EXHAUSTED};
    for (size_t i = 0; i < sizeof codes / sizeof codes[0]; ++i) {
        const char *s = pkv_status_string(codes[i]);
        check(s != NULL && strlen(s) > 0, "status string");
    }

    /* workspace: two records of (head_dim + 4) floats per worker and head of
       a record, at most 4096 workers and never more than the pages */
    check(pkv_decode_workspace_size(64, 32, 8, 128, 2048) ==
              (size_t)4096 * 2 * 4 * (128 + 4) * 4,
          "workspace of 64 x 2048, 32 / 8 heads, d 128");
    check(pkv_decode_workspace_size(2, 8, 2, 64, 37) == (size_t)(2 * 2 * 3) * 2 * 4 * (64 + 4) * 4,
          "workspace of 2 x 37, 8 / 2 heads, d 64");
    check(pkv_decode_workspace_size(4, 8, 3, 128, 16) == 0, "workspace: heads not divisible");
    check(pkv_decode_workspace_size(4, 8, 2, 96, 16) == 0, "workspace: unsupported head_dim");

    /* decode argument checks, before any CUDA call */
    const size_t ws = (size_t)1 << 30;
    check(pkv_paged_decode_fp16(NULL, FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 64, 2, 8, 2, 64, 16,
                                0.125f, FAKE, ws, NULL, NULL) == PKV_ERR_INVALID_ARG,
          "fp16 decode: null output");
    check(pkv_paged_decode_int8(FAKE, FAKE, FAKE, FAKE, NULL, FAKE, 16, FAKE, 4, FAKE, 64, 2, 8,
                                2, 64, 16, 0.125f, FAKE, ws, NULL, NULL) == PKV_ERR_INVALID_ARG,
          "INT8 decode: null K scales");
    check(pkv_paged_decode_int8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 64, 2, 8,
                                2, 96, 16, 0.125f, FAKE, ws, NULL, NULL) == PKV_ERR_UNSUPPORTED,
          "INT8 decode: head_dim 96");
    check(pkv_paged_decode_int8(FAKE, FAKE, (const int8_t *)FAKE + 4, FAKE, FAKE, FAKE, 16, FAKE,
                                4, FAKE, 64, 2, 8, 2, 64, 16, 0.125f, FAKE, ws, NULL,
                                NULL) == PKV_ERR_MISALIGNED,
          "INT8 decode: misaligned codes");
    check(pkv_paged_decode_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 64, 2, 8, 2,
                               64, 16, 0.125f, FAKE, 100, NULL, NULL) == PKV_ERR_WORKSPACE,
          "FP8 decode: workspace too small");
    check(pkv_paged_decode_int8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, FAKE, 4, FAKE, 64, 0, 8,
                                2, 64, 16, 0.125f, FAKE, ws, NULL, NULL) == PKV_OK,
          "INT8 decode: no sequences, nothing launched");

    /* quantize and append argument checks */
    check(pkv_quantize_blocks(FAKE, FAKE, NULL, FAKE, FAKE, FAKE, NULL, 0, 16, 2, 64, 16, NULL,
                              NULL) == PKV_ERR_INVALID_ARG,
          "quantize: null K codes");
    check(pkv_quantize_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 16, 2, 64, 16, NULL,
                              NULL) == PKV_OK,
          "quantize: empty id list, nothing launched");
    check(pkv_quantize_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 0, 16, 2, 64, 32, NULL,
                              NULL) == PKV_ERR_UNSUPPORTED,
          "quantize: block size 32");
    check(pkv_append_fp16(FAKE, FAKE, 16, FAKE, FAKE, FAKE, 4, FAKE, 0, 2, 64, 16, NULL, NULL) ==
              PKV_OK,
          "append: no sequences, nothing launched");

    /* the host block manager: allocate with prefix sharing, stats, free */
    pkv_block_manager *bm = NULL;
    check(pkv_bm_create(8, 16, &bm) == PKV_OK && bm != NULL, "block manager: create");
    const uint64_t hashes[3] = {11, 0, 11}; /* 0: no prefix hash */
    int32_t ids[3] = {-1, -1, -1};
    check(pkv_bm_allocate(bm, hashes, 3, ids) == PKV_OK, "block manager: allocate");
    check(ids[0] == ids[2] && ids[0] != ids[1], "block manager: equal prefix hash shares a block");
    pkv_bm_stats_t st;
    check(pkv_bm_stats(bm, &st) == PKV_OK && st.used_blocks == 2 && st.shared_blocks == 1 &&
              st.logical_blocks == 3 && st.free_blocks == 6,
          "block manager: stats after allocation");
    check(pkv_bm_free(bm, ids, 3) == PKV_OK, "block manager: free");
    check(pkv_bm_stats(bm, &st) == PKV_OK && st.free_blocks == 8 && st.used_blocks == 0,
          "block manager: all free again");
    check(pkv_bm_free(bm, ids, 1) == PKV_ERR_INVALID_ARG, "block manager: freeing a free block");
    pkv_bm_destroy(bm);
    pkv_block_manager *none = NULL;
    check(pkv_bm_create(-1, 16, &none) == PKV_ERR_INVALID_ARG && none == NULL,
          "block manager: negative block count");

    printf("%s\n", failures ? "C ABI checks failed" : "C ABI checks passed");
    return failures ? 1 : 0;
}

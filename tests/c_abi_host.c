/* A C99 client of libpagedkv.so that uses only host entry points (no GPU):
 * the block pool with fork and copy-on-write, block-table export, a
 * sliding-window pool with room for prefill chunks and its logically ordered
 * tables, the SplitFuse composer, workspace sizing and status strings.  It checks each
 * result against values worked out by hand from the rules in pagedkv.h and
 * prints "ok" when all hold.  Built and run by tests/test_c_abi.py. */
#include <stdio.h>
#include <string.h>

#include "pagedkv.h"

static int failures = 0;

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            printf("FAILED line %d: %s\n", __LINE__, #cond);          \
            ++failures;                                               \
        }                                                             \
    } while (0)

int main(void) {
    pkv_pool* pool = NULL;
    int64_t slots[6];
    int64_t slot = -1;
    int32_t src = 0, dst = 0, rc = 0, n = 0, i;
    int32_t tables[2 * 4], ctx[2];
    int64_t ids[2] = {1, 2};
    int32_t prompts[2] = {4, 6}, chunks[2] = {0, 0}, dec = 0, used = 0;
    pkv_cache_desc desc = {PKV_BF16, 100, 16, 8, 32, 128};

    /* 8 blocks of 4 tokens, no watermark, blocks handed out 0, 1, 2, ... */
    CHECK(pkv_pool_create(8, 4, 0, NULL, &pool) == PKV_OK && pool != NULL);
    CHECK(pkv_seq_add(pool, 1, 6, slots) == PKV_OK);
    for (i = 0; i < 6; ++i) CHECK(slots[i] == i);           /* blocks 0 and 1 */
    CHECK(pkv_pool_num_free(pool, &n) == PKV_OK && n == 6);

    /* the fork shares both blocks */
    CHECK(pkv_seq_fork(pool, 1, 2) == PKV_OK);
    CHECK(pkv_block_ref_count(pool, 0, &rc) == PKV_OK && rc == 2);
    CHECK(pkv_block_ref_count(pool, 1, &rc) == PKV_OK && rc == 2);

    /* growing the child: its last block (1) is shared, so block 2 replaces it
     * and the caller copies 1 -> 2 before the token goes to row 2 of block 2 */
    CHECK(pkv_seq_append_slot(pool, 2, &slot, &src, &dst) == PKV_OK);
    CHECK(src == 1 && dst == 2 && slot == 2 * 4 + 2);
    CHECK(pkv_block_ref_count(pool, 1, &rc) == PKV_OK && rc == 1);

    /* growing the parent: block 1 is its own now, no copy */
    CHECK(pkv_seq_append_slot(pool, 1, &slot, &src, &dst) == PKV_OK);
    CHECK(src == -1 && dst == -1 && slot == 1 * 4 + 2);

    CHECK(pkv_block_tables(pool, ids, 2, 4, tables, ctx) == PKV_OK);
    CHECK(tables[0] == 0 && tables[1] == 1 && tables[2] == -1 && tables[3] == -1);
    CHECK(tables[4] == 0 && tables[5] == 2 && tables[6] == -1 && tables[7] == -1);
    CHECK(ctx[0] == 7 && ctx[1] == 7);
    CHECK(pkv_block_tables(pool, ids, 2, 1, tables, ctx) == PKV_ERR_INVALID);

    /* freeing the child leaves block 0 to the parent and returns block 2 */
    CHECK(pkv_seq_free(pool, 2) == PKV_OK);
    CHECK(pkv_block_ref_count(pool, 0, &rc) == PKV_OK && rc == 1);
    CHECK(pkv_pool_num_free(pool, &n) == PKV_OK && n == 6);
    CHECK(pkv_seq_len(pool, 1, &n) == PKV_OK && n == 7);
    CHECK(pkv_seq_len(pool, 2, &n) != PKV_OK);
    CHECK(pkv_pool_destroy(pool) == PKV_OK);

    /* budget 8: the 3 decodes first, then 4 + 1 prompt tokens */
    CHECK(pkv_splitfuse_compose(8, 3, 2, prompts, chunks, &dec, &used) == PKV_OK);
    CHECK(dec == 3 && chunks[0] == 4 && chunks[1] == 1 && used == 8);

    /* the decode workspace depends only on the shapes */
    CHECK(pkv_decode_workspace_bytes(&desc, 64, 4096) > 0);
    CHECK(pkv_decode_workspace_bytes(&desc, 64, 4096) ==
          pkv_decode_workspace_bytes(&desc, 64, 4096));
    CHECK(PKV_INT8_TILE_BYTES(128) == 2112 && PKV_INT8_TILE_BYTES(64) == 1088);
    /* the 8-bit pool: per (block, kv head) a K tile and a V tile */
    CHECK(PKV_INT8_POOL_BYTES(3, 2, 128) == (size_t)3 * 2 * 2 * 2112);

    CHECK(pkv_status_string(PKV_OK) != NULL);
    CHECK(pkv_status_string(PKV_ERR_NO_BLOCKS) != NULL &&
          strlen(pkv_status_string(PKV_ERR_NO_BLOCKS)) > 0);
    CHECK(pkv_status_string(12345) != NULL);

    /* a sliding-window pool with room for chunks of up to 6 queries: window 8
     * (2 blocks of 4) + ceil(5 / 4) = 4 ring blocks, handed out 0, 1, 2, 3 */
    {
        pkv_pool* wp = NULL;
        int64_t wid = 7, wslots[6], wslot = -1;
        int32_t q6 = 6, q1 = 1, q10 = 10, wt[5], wctx = 0;
        CHECK(pkv_pool_create_window(32, 4, 0, NULL, 8, 6, &wp) == PKV_OK && wp != NULL);
        CHECK(pkv_seq_add(wp, wid, 6, wslots) == PKV_OK && wslots[5] == 1 * 4 + 1);
        for (i = 0; i < 15; ++i)
            CHECK(pkv_seq_append_slot(wp, wid, &wslot, &src, &dst) == PKV_OK && src == -1);
        /* 21 tokens: logical blocks 4 and 5 reuse ring entries 0 and 1 */
        CHECK(wslot == 1 * 4 + 0);
        /* the last 6 tokens as queries: first key 21 - 6 - 8 + 1 = 8, block 2;
         * logical blocks 2..5 are ring entries 2, 3, 0, 1; context 21 - 8 */
        CHECK(pkv_window_tables(wp, &wid, &q6, 1, 5, wt, &wctx) == PKV_OK);
        CHECK(wt[0] == 2 && wt[1] == 3 && wt[2] == 0 && wt[3] == 1 && wt[4] == -1 && wctx == 13);
        /* one decode query: first key 13, block 3; context 21 - 12 */
        CHECK(pkv_window_tables(wp, &wid, &q1, 1, 5, wt, &wctx) == PKV_OK);
        CHECK(wt[0] == 3 && wt[1] == 0 && wt[2] == 1 && wt[3] == -1 && wctx == 9);
        /* 10 + 8 - 1 keys do not fit the ring's 16 tokens */
        CHECK(pkv_window_tables(wp, &wid, &q10, 1, 5, wt, &wctx) == PKV_ERR_INVALID);
        CHECK(pkv_block_tables(wp, &wid, 1, 5, wt, &wctx) == PKV_ERR_UNSUPPORTED);
        CHECK(pkv_pool_destroy(wp) == PKV_OK);
    }

    if (failures) return 1;
    printf("ok\n");
    return 0;
}

/* A plain C program against include/pkv.h and libpkv.so: the host-only calls
 * (status strings, workspace sizes, argument checks, the cascade grouping and
 * the sparse policy) used without any CUDA header or device.  Prints one line
 * per check and exits non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "pkv.h"

static int fails = 0;
#define CHECK(cond, what)                                         \
    do {                                                          \
        if (cond) {                                               \
            printf("ok   %s\n", what);                            \
        } else {                                                  \
            printf("FAIL %s\n", what);                            \
            fails++;                                              \
        }                                                         \
    } while (0)

int main(void) {
    CHECK(strcmp(pkv_status_string(PKV_OK), "ok") == 0, "status string");
    CHECK(pkv_split_workspace_bytes(8, 32, 128, 16) > 0, "split workspace size");
    CHECK(pkv_balanced_workspace_bytes(8, 8, 128) > 0, "balanced workspace size");
    CHECK(pkv_cascade_workspace_bytes(4, 32, 8, 128, 1, 4) > 0, "cascade workspace size");
    CHECK(pkv_sparse_workspace_bytes(4, 8, 128, 8) > 0, "sparse workspace size");

    /* a NULL cache is refused before anything reaches the device */
    pkv_status st = pkv_paged_attention(NULL, PKV_F32, NULL, PKV_BF16, 32, 0.088f, NULL, NULL, NULL, NULL);
    CHECK(st == PKV_ERR_INVALID_ARG && strstr(pkv_last_error(), "NULL") != NULL, "NULL cache refused");

    /* cascade grouping on host arrays: sequences 0..2 share 4 leading blocks */
    const int32_t tables[4 * 6] = {7, 8, 9, 10, 11, -1,
                                   7, 8, 9, 10, 12, 13,
                                   7, 8, 9, 10, 14, -1,
                                   1, 2, 3, -1, -1, -1};
    const int32_t ctx[4] = {80, 90, 70, 40};
    int32_t members[2 * 4], blocks[2], n = -1;
    st = pkv_cascade_plan(tables, ctx, 4, 6, 2, 2, 4, 2, members, blocks, &n);
    CHECK(st == PKV_OK && n == 1 && blocks[0] == 4, "cascade plan finds the shared prefix");
    int seen = 0;
    for (int j = 0; j < 4; ++j) seen |= members[j] >= 0 ? 1 << members[j] : 0;
    CHECK(seen == 0x7 && members[3] == -1, "cascade plan members 0, 1, 2");

    /* sparse policy: 3 of 10 pages listed -> 70 % skipped */
    const int32_t counts[2] = {1, 2}, lens[2] = {64, 96};
    CHECK(pkv_sparse_worthwhile(counts, lens, 2, 0.6f) == 1, "sparse worthwhile at 0.6");
    CHECK(pkv_sparse_worthwhile(counts, lens, 2, 0.8f) == 0, "sparse not worthwhile at 0.8");
    return fails ? 1 : 0;
}

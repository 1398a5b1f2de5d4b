/* Plain-C client of the C ABI: includes include/fmha.h as C (no C++), links
 * against the library and exercises the calls that need no GPU.  Exit status
 * 0 when every check holds; the failing check's line otherwise. */
#include <stdio.h>
#include <string.h>

#include "fmha.h"

#define CHECK(cond)                                              \
    do {                                                         \
        if (!(cond)) {                                           \
            fprintf(stderr, "check failed at line %d\n", __LINE__); \
            return __LINE__;                                     \
        }                                                        \
    } while (0)

int main(void) {
    int first = -1, chunk = 0, kernel = 0;
    CHECK(fmha_version() >= 100);
    CHECK(fmha_build_flags() == 0 || fmha_build_flags() == FMHA_BUILD_CHECKED);
    /* split layout: 4096-key window over 8192 keys in 512-key chunks */
    CHECK(fmha_split_layout(1, 8192, 4096, 512, &first) == 8 && first == 4096);
    /* planner: MQA decode at hd 512 runs on the hd-512 tensor-core kernel (3) */
    CHECK(fmha_fwd_plan(16, 128, 1, 1, 512, 512, 0, 0, &chunk, &kernel) >= 1 && kernel == 3 && chunk >= 1);
    /* argument errors come back as codes with a message, before any CUDA call */
    CHECK(fmha_fwd(NULL, NULL, NULL, NULL, NULL, 1, 2, 1, 1, 8, 64, 0.125f, 0, 0, NULL) == FMHA_ERR_NULL);
    CHECK(strlen(fmha_get_last_error()) > 0);
    CHECK(fmha_fwd((void*)16, (void*)16, (void*)16, (void*)16, (float*)16, 1, 2, 1, 1, 8, 80, 0.125f, 0, 0, NULL) ==
          FMHA_ERR_HEADDIM);
    CHECK(fmha_fwd_host(NULL, NULL, NULL, NULL, NULL, 1, 2, 1, 1, 8, 64, 0.125f, 0, 0, NULL) == FMHA_ERR_NULL);
    CHECK(fmha_splitkv_workspace_bytes(2, 8, 1, 128, 4) == (size_t)4 * 16 * (128 * 4 + 4));
    CHECK(fmha_workspace_bytes(2, 8, 1, 128, 4) == fmha_splitkv_workspace_bytes(2, 8, 1, 128, 4));
    CHECK(fmha_workspace_bytes(-1, 8, 1, 128, 4) == 0);
    printf("c abi ok\n");
    return 0;
}

/*
 * A plain C99 client of libfa: compiles against include/fa.h alone, links
 * libfa.so, and makes the calls that need no GPU (size queries, status
 * strings, argument checks).  Prints "ok" and exits 0 when every answer is
 * the documented one.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa.h"

static int failures = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

int main(void) {
    /* any 256-byte-aligned, non-null address: rejected calls never touch it */
    char* raw = malloc(512);
    if (raw == NULL) return 2;
    void* p = (void*)(((uintptr_t)raw + 255u) & ~(uintptr_t)255u);

    expect(strcmp(fa_status_string(FA_OK), "FA_OK") == 0, "status string of FA_OK");
    expect(strcmp(fa_status_string(FA_ERR_INVALID_ARG), "FA_ERR_INVALID_ARG") == 0,
           "status string of FA_ERR_INVALID_ARG");

    /* workspace: 4*B*H*N for D, the fp16 copies and 512 bytes of scales, each
       part rounded up to 256 bytes */
    expect(fa_bwd_workspace_size(2, 3, 1, 5, 64) == 11008, "workspace size, small case");
    expect(fa_bwd_workspace_size(1, 1, 1, 1, 96) == 0, "workspace size, unsupported d");
    expect(fa_bwd_workspace_size(1, 6, 4, 1, 64) == 0, "workspace size, H % Hkv != 0");

    /* argument checks: returned before any device work */
    expect(fa_fwd(p, p, p, p, (float*)p, 0, 1, 1, 128, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with B = 0");
    expect(fa_fwd(p, p, p, p, (float*)p, 1, 6, 4, 128, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with H % Hkv != 0");
    expect(fa_fwd(p, p, p, p, (float*)p, 1, 1, 1, 128, 64, 0, -1.0f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with a negative scale");
    expect(fa_fwd(p, p, p, p, (float*)p, 1, 1, 1, 128, 96, 0, 0.125f, NULL) ==
               FA_ERR_UNSUPPORTED, "fa_fwd with d = 96");
    expect(fa_fwd((char*)p + 8, p, p, p, (float*)p, 1, 1, 1, 128, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with q not 16-byte aligned");
    expect(fa_bwd(p, p, p, p, p, (float*)p, p, p, p, p, NULL, 1, 1, 1, 0, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_bwd with N = 0");
    expect(fa_fwd_fp8_workspace_size(1, 4, 2, 256, 64) == 0, "fp8 workspace, d = 64");
    expect(fa_fwd_splitkv_num_splits(1, 8, 2, 10, 5, 128, 1, 0) == 0,
           "split-KV plan, causal with Nq > Nk");

    free(raw);
    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}

/* A plain C99 consumer of mbw.h: compiles the header as C with strict
 * warnings, links libmbw.so, and exercises the calls whose argument checks
 * run before any CUDA work (no GPU needed). Exit status 0 when every call
 * returns the documented status. */
#include <stdio.h>
#include <string.h>

#include "mbw.h"

static int failures = 0;

static void expect(const char *what, mbw_status got, mbw_status want) {
    if (got != want) {
        fprintf(stderr, "%s: got %d (%s), want %d\n", what, got, mbw_status_string(got), want);
        ++failures;
    } else if (want != MBW_OK && mbw_last_error()[0] == '\0') {
        fprintf(stderr, "%s: no error detail\n", what);
        ++failures;
    }
}

int main(void) {
    static const char *names[] = {"MBW_OK", "MBW_ERR_INVALID_ARG", "MBW_ERR_MISALIGNED", "MBW_ERR_BAD_SHAPE",
                                  "MBW_ERR_WORKSPACE_TOO_SMALL", "MBW_ERR_UNSUPPORTED", "MBW_ERR_CUDA",
                                  "MBW_ERR_DEVICE_TIMEOUT"};
    /* fake, 16-byte aligned addresses: the argument checks never dereference them */
    void *a = (void *)(uintptr_t)0x10000, *b = (void *)(uintptr_t)0x20000, *c = (void *)(uintptr_t)0x30000;
    mbw_status s;
    for (s = MBW_OK; s <= MBW_ERR_DEVICE_TIMEOUT; ++s) {
        if (strcmp(mbw_status_string(s), names[s]) != 0) {
            fprintf(stderr, "status %d is named %s\n", s, mbw_status_string(s));
            ++failures;
        }
    }
    expect("gemv_bf16 negative N", gemv_bf16(a, b, c, -1, 64, NULL, 0, NULL), MBW_ERR_INVALID_ARG);
    expect("gemv_bf16 K % 8", gemv_bf16(a, b, c, 8, 60, NULL, 0, NULL), MBW_ERR_BAD_SHAPE);
    expect("gemv_bf16 N == 0", gemv_bf16(NULL, NULL, NULL, 0, 64, NULL, 0, NULL), MBW_OK);
    expect("gemv_bf16 N above MBW_MAX_DIM", gemv_bf16(a, b, c, MBW_MAX_DIM + 1, 64, NULL, 0, NULL),
           MBW_ERR_BAD_SHAPE);
    expect("gemv_int4_g64 K % 64", gemv_int4_g64(a, b, c, c, 8, 96, NULL, 0, NULL), MBW_ERR_BAD_SHAPE);
    expect("gemv_int4_awq_g128 misaligned codes",
           gemv_int4_awq_g128((const uint8_t *)a + 16, b, c, c, a, 1, 8, 256, NULL, 0, NULL), MBW_ERR_MISALIGNED);
    expect("gemm_skinny_bf16 M == 0", gemm_skinny_bf16(a, b, c, 0, 8, 16, NULL, 0, NULL), MBW_OK);
    expect("gemv_int8_pc K % 128", gemv_int8_pc(a, b, c, a, 1, 8, 192, NULL, 0, NULL), MBW_ERR_BAD_SHAPE);
    expect("mbw_repack_int4 NULL", mbw_repack_int4(NULL, b, 8, 64, NULL), MBW_ERR_INVALID_ARG);
    expect("mbw_set_output_fp32(2)", mbw_set_output_fp32(2), MBW_ERR_INVALID_ARG);
    expect("mbw_plan_select unknown op", mbw_plan_select(9, 1, 8, 64, 0), MBW_ERR_INVALID_ARG);
    expect("mbw_selftest_wait_expiry(0)", mbw_selftest_wait_expiry(0, NULL), MBW_ERR_INVALID_ARG);
    expect("mbw_selftest_wait_expiry(limit + 1)", mbw_selftest_wait_expiry(MBW_WAIT_LIMIT + 1, NULL),
           MBW_ERR_INVALID_ARG);
    if (mbw_launch_count() != 0) {
        fprintf(stderr, "launches counted without any launch\n");
        ++failures;
    }
    printf("%s\n", failures ? "FAIL" : "ok");
    return failures ? 1 : 0;
}

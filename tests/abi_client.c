/* A plain C99 client of the C ABI: it includes only include/q4gemv.h, links
 * libq4gemv.so and makes the calls that need no GPU (packed sizes, status text,
 * argument checks that fail before any CUDA call, empty problems).  Built and
 * run by tests/test_abi.py; prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "q4gemv.h"

static int failures = 0;

static void expect(int cond, const char *what)
{
    if (!cond) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

int main(void)
{
    /* an aligned address that is never dereferenced: every call below fails its
     * host-side checks (or is empty) before anything touches it */
    void *const A = (void *)(uintptr_t)0x100000;
    float *const F = (float *)A;
    q4gemv_pack_info_t info;

    /* the 0.5B LM head, 151936 x 896, group 32 */
    expect(q4gemv_pack_info(151936, 896, 32, &info) == Q4_OK, "pack_info status");
    expect(info.codes_bytes == 68067328, "codes bytes of 151936 x 896");
    expect(info.scales_bytes == 8508416, "scales bytes of 151936 x 896, g = 32");
    expect(info.zeros_bytes == 2127104, "zero-point bytes of 151936 x 896, g = 32");
    expect(info.blocks_per_row == 28 && info.zeros_row_bytes == 14, "groups and zero bytes per row");
    expect(info.base_alignment == 16, "base alignment");
    /* an odd group count pads the zero-point row: K = 896, g = 128 -> 7 groups, 4 bytes */
    expect(q4gemv_pack_info(4, 896, 128, &info) == Q4_OK && info.zeros_row_bytes == 4, "padded zero row");
    expect(q4gemv_pack_info(4, 96, 64, &info) == Q4_ERR_INVALID_ARG, "K % g != 0 rejected");
    expect(q4gemv_pack_info(4, 64, 32, NULL) == Q4_ERR_INVALID_ARG, "NULL out rejected");

    expect(strcmp(q4gemv_status_string(99), "unknown status") == 0, "unknown status text");
    expect(strlen(q4gemv_status_string(Q4_ERR_MISALIGNED)) > 0, "status text");

    /* argument checks, no launch */
    expect(q4gemv_run(A, A, NULL, F, F, 17, 64, 64, 32, NULL) == Q4_ERR_UNSUPPORTED, "M > 16");
    expect(q4gemv_run(A, A, NULL, F, F, 1, 64, 64, 48, NULL) == Q4_ERR_INVALID_ARG, "group 48");
    expect(q4gemv_run(NULL, A, NULL, F, F, 1, 64, 64, 32, NULL) == Q4_ERR_INVALID_ARG, "null codes");
    expect(q4gemv_run((char *)A + 8, A, NULL, F, F, 1, 64, 64, 32, NULL) == Q4_ERR_MISALIGNED, "codes 8 B off");
    expect(q4gemv_fused_run(A, A, NULL, F, NULL, 0.0f, F, 1, 63, 64, 32, Q4_EPILOGUE_SWIGLU, NULL) ==
               Q4_ERR_INVALID_ARG, "odd N with SwiGLU");
    expect(q4_0_gemv_run(A, F, F, 1, 64, 48, NULL) == Q4_ERR_INVALID_ARG, "Q4_0 K % 32 != 0");
    expect(q8_0_gemv_run(A, F, F, 1, 64, 48, NULL) == Q4_ERR_INVALID_ARG, "Q8_0 K % 32 != 0");
    expect(q8_0_gemv_run(A, F, F, 17, 64, 64, NULL) == Q4_ERR_UNSUPPORTED, "Q8_0 M > 16");
    expect(q4gemm_run(A, A, NULL, A, F, 1, 64, 100, 32, NULL) == Q4_ERR_INVALID_ARG, "gemm K % g != 0");
    expect(f32gemv_run(F, F, F, 17, 64, 64, NULL) == Q4_ERR_UNSUPPORTED, "f32 M > 16");

    {
        q4gemv_segment_t segs[2] = {{A, A, NULL, F, F, 64}, {A, A, NULL, (const float *)((char *)A + 4), F, 64}};
        expect(q4gemv_grouped_run(segs, 2, 896, 32, NULL) == Q4_ERR_MISALIGNED, "grouped: x 4 B off");
        expect(q4gemv_grouped_run(NULL, 0, 896, 32, NULL) == Q4_OK, "grouped: empty list");
        expect(q4gemv_grouped_run(NULL, 1, 896, 32, NULL) == Q4_ERR_INVALID_ARG, "grouped: null list");
        segs[1].N = 0;   /* an empty entry is skipped, but the first still fails on K % g */
        expect(q4gemv_grouped_run(segs, 2, 100, 32, NULL) == Q4_ERR_INVALID_ARG, "grouped: K % g != 0");
    }

    {   /* per-call options: checked before the arguments; outputs may not overlap inputs */
        q4_run_options_t bad = {0x80u, 0u, 0u}, reserved = {0u, 1u, 0u};
        q4_run_options_t good = {Q4_RUN_OVERLAPPED | Q4_RUN_EXACT_X | Q4_RUN_WAIT_TIMEOUT, 0u, 1000u};
        q4_run_options_t exact = {Q4_RUN_EXACT_X, 0u, 0u};
        char *const B = (char *)(uintptr_t)0x10000000;
        expect(q4gemv_run_ex(A, A, NULL, F, F, 1, 64, 64, 32, &bad, NULL) == Q4_ERR_INVALID_ARG, "unknown flag");
        expect(q4gemv_run_ex(A, A, NULL, F, F, 1, 64, 64, 32, &reserved, NULL) == Q4_ERR_INVALID_ARG,
               "reserved field");
        expect(q4gemv_run_ex(A, A, NULL, F, F, 17, 64, 64, 32, &good, NULL) == Q4_ERR_UNSUPPORTED, "ex: M > 16");
        expect(q4gemm_run_ex(A, A, NULL, A, F, 128, 64, 64, 32, &exact, NULL) == Q4_ERR_INVALID_ARG,
               "gemm: exact-x flag");
        expect(q4gemv_run_ex(B, B + 0x100000, NULL, (const float *)(B + 0x200000), (float *)(B + 0x200000), 1, 64,
                             64, 32, NULL, NULL) == Q4_ERR_INVALID_ARG, "y on x");
    }

    /* empty problems: Q4_OK, pointers unused */
    expect(q4gemv_run(NULL, NULL, NULL, NULL, NULL, 0, 64, 64, 32, NULL) == Q4_OK, "M = 0");
    expect(q4gemv_run(NULL, NULL, NULL, NULL, NULL, 3, 0, 64, 32, NULL) == Q4_OK, "N = 0");
    expect(q4gemm_run(NULL, NULL, NULL, NULL, NULL, 0, 64, 64, 32, NULL) == Q4_OK, "gemm M = 0");

    /* host-only state */
    expect(q4gemv_set_overlapped_launch(1) == 0 && q4gemv_set_overlapped_launch(0) == 1, "overlap toggle");
    expect(q4gemv_bounds_violations(NULL) == -1, "no bounds checks in the product build");

    if (failures == 0)
        printf("ok\n");
    return failures == 0 ? 0 : 1;
}

/*
 * Plain C99 client of include/qk.h, built and run by tests/test_abi.py: the
 * header must compile as strict C and the library must link and answer from
 * C.  Every compute call below carries an invalid argument, so each returns
 * its status from host validation and nothing reaches a GPU.
 * Prints one line per check and exits non-zero on the first mismatch.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "qk.h"

static int failures = 0;

static void expect(const char *what, long long got, long long want)
{
    printf("%s %lld %lld\n", what, got, want);
    if (got != want) ++failures;
}

int main(void)
{
    /* never dereferenced: every call fails validation first */
    void *fake = (void *)(uintptr_t)0x10000;
    float *fx = (float *)fake;
    float *bad_x = (float *)((uintptr_t)0x10002);   /* not 4-byte aligned */
    int32_t *ids = (int32_t *)fake;

    expect("row_bytes_q8_0", qk_row_bytes_q8_0(576), 18 * 34);
    expect("row_bytes_q4_k", qk_row_bytes_q4_k(896), 4 * 144);
    expect("row_bytes_q6_k", qk_row_bytes_q6_k(4096), 16 * 210);
    expect("status_string", strcmp(qk_status_string(QK_OK), "ok"), 0);
    expect("status_string_unknown", strcmp(qk_status_string(99), "unknown status"), 0);
    expect("version", qk_version() > 0, 1);

    expect("gemv_null_w", qmatvec_q4_k(NULL, 0, 8, 256, fx, 1, fx, 0, NULL), QK_ERR_NULL);
    expect("gemv_rows0", qmatvec_q8_0(fake, 0, 0, 256, fx, 1, fx, 0, NULL), QK_ERR_BAD_DIM);
    expect("gemv_batch9", qmatvec_q6_k(fake, 0, 8, 256, fx, 9, fx, 0, NULL), QK_ERR_BATCH);
    expect("gemv_align_x", qmatvec_q4_k(fake, 0, 8, 256, bad_x, 1, fx, 0, NULL), QK_ERR_ALIGN);
    expect("swiglu_neg_up", qmatvec_swiglu_q4_k(fake, 0, -1, 8, 256, fx, 1, fx, 0, NULL), QK_ERR_BAD_DIM);
    expect("experts_null_ids", qmatvec_experts_q8_0(fake, 4, 8, 256, fx, 1, NULL, 2, fx, 0, NULL), QK_ERR_NULL);
    expect("experts_xk0", qmatvec_experts_q4_k(fake, 4, 8, 256, fx, 0, ids, 2, fx, 0, NULL), QK_ERR_BAD_DIM);
    expect("gemm_no_workspace", qgemm_q4_k(fake, 0, 128, 256, fx, 4, fx, 0, NULL, 0, NULL), QK_ERR_WORKSPACE);
    expect("gemm_m0", qgemm_q8_0(fake, 0, 128, 256, fx, 0, fx, 0, fake, 1 << 20, NULL), QK_ERR_BAD_DIM);
    expect("gemm_swiglu_align", qgemm_swiglu_q8_0(fake, 0, 128, 128, 256, bad_x, 4, fx, 0, fake, 1 << 20, NULL),
           QK_ERR_ALIGN);
    expect("noalloc_null", qgemm_q4_k_noalloc(fake, 0, 128, 256, NULL, 4, fx, 0, NULL), QK_ERR_NULL);
    expect("workspace_bytes", qgemm_q4_k_workspace_bytes(512, 14336, 4096) >= (size_t)512 * 4096 * 2, 1);

    /* strict-blocks mode: K = 300 is not a whole number of Q4_K blocks */
    {
        const int old = qk_set_strict_blocks(1);
        expect("strict_on", qmatvec_q4_k(fake, 0, 8, 300, bad_x, 1, fx, 0, NULL), QK_ERR_BAD_DIM);
        expect("strict_whole", qmatvec_q4_k(fake, 0, 8, 512, bad_x, 1, fx, 0, NULL), QK_ERR_ALIGN);
        expect("strict_prev", qk_set_strict_blocks(0), 1);
        expect("strict_off", qmatvec_q4_k(fake, 0, 8, 300, bad_x, 1, fx, 0, NULL), QK_ERR_ALIGN);
        qk_set_strict_blocks(old);
    }
    {
        const uint64_t old = qk_set_wait_limit_ns(12345);
        expect("wait_limit", (long long)qk_set_wait_limit_ns(old), 12345);
    }
    printf("failures %d\n", failures);
    return failures ? 1 : 0;
}

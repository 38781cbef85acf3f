/* A plain C11 caller of libks, built and run by tests/test_c_abi.py on a machine without a GPU:
 * the header compiles as C, the library links, and the calls that fail argument checks return
 * their documented status before touching the device. No valid call is made (it would launch a
 * kernel). Exit status 0 means every check held. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ks.h"

static int failures = 0;

static void expect(int got, int want, const char *what) {
    if (got != want) {
        fprintf(stderr, "FAIL %s: got %d (%s), want %d\n", what, got,
                ks_status_string((ks_status_t)got), want);
        ++failures;
    }
}

int main(void) {
    void *a = (void *)(uintptr_t)0x10000, *b = (void *)(uintptr_t)0x40010000,
         *w = (void *)(uintptr_t)0x80010000;
    expect(ks_version() >= 100, 1, "version");
    expect(strcmp(ks_status_string(KS_ERR_OVERLAP), "KS_ERR_OVERLAP") == 0, 1, "status name");

    expect(ks_rms_norm(a, b, w, 4, 0, 1e-6f, KS_DTYPE_BF16, NULL), KS_ERR_INVALID_ARGUMENT,
           "rms_norm hidden 0");
    expect(ks_rms_norm(a, b, w, -1, 64, 1e-6f, KS_DTYPE_BF16, NULL), KS_ERR_INVALID_ARGUMENT,
           "rms_norm rows < 0");
    expect(ks_rms_norm(a, b, w, 4, 64, 0.0f, KS_DTYPE_BF16, NULL), KS_ERR_INVALID_ARGUMENT,
           "rms_norm eps 0");
    expect(ks_rms_norm(a, b, w, 4, 64, 1e-6f, (ks_dtype_t)9, NULL), KS_ERR_UNSUPPORTED_DTYPE,
           "rms_norm dtype");
    expect(ks_rms_norm(NULL, NULL, NULL, 0, 64, 1e-6f, KS_DTYPE_BF16, NULL), KS_SUCCESS,
           "rms_norm empty");
    expect(ks_fused_add_rms_norm(a, a, w, 4, 64, 1e-6f, KS_DTYPE_BF16, NULL), KS_ERR_OVERLAP,
           "fused overlap");
    expect(ks_silu_and_mul(a, a, 4, 64, KS_DTYPE_F16, NULL), KS_ERR_OVERLAP, "silu overlap");
    expect(ks_softmax(a, b, 4, 0, KS_DTYPE_F32, NULL), KS_ERR_INVALID_ARGUMENT, "softmax width 0");
    expect(ks_layer_norm(a, b, NULL, NULL, 4, 64, -1.0f, KS_DTYPE_BF16, NULL),
           KS_ERR_INVALID_ARGUMENT, "layer_norm eps");
    expect(ks_rms_norm_host(a, b, w, 4, 64, 1e-6f, KS_DTYPE_BF16, b, 0, NULL),
           KS_ERR_INVALID_ARGUMENT, "host empty workspace");
    expect(ks_fused_add_rms_norm_host_noalloc(a, b, w, 1, (int64_t)1 << 22, 1e-6f, KS_DTYPE_BF16,
                                              NULL),
           KS_ERR_INVALID_ARGUMENT, "noalloc row too wide");

    ks_plan_t p;
    expect(ks_plan_launch(1, 32768, 8192, KS_DTYPE_BF16, 1, 152, 2, &p), KS_SUCCESS, "plan");
    expect(p.kernel, KS_KERNEL_CTA_ROW, "plan kernel");
    expect(p.vec_per_thread, 2, "plan vectors per thread");
    expect(p.block, 512, "plan block");
    expect(p.flags, KS_PLAN_NO_PREFETCH, "plan flags");
    expect(ks_set_launch_options(KS_LAUNCH_PDL), KS_SUCCESS, "options on");
    expect(ks_get_launch_options(), KS_LAUNCH_PDL, "options read");
    expect(ks_set_launch_options(0), KS_SUCCESS, "options off");
    expect((int)ks_host_chunk_rows(0, 8192, KS_DTYPE_BF16, 3 * 16384 * 10), 10, "chunk rows");

    if (failures == 0) printf("c abi ok\n");
    return failures == 0 ? 0 : 1;
}

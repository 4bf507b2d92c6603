/* Drives the host-side argument validation of libgdn.so (include/gdn.h,
 * include/gdn_proj.h) with bad arguments, none of which may reach a device, so
 * that a build of the library with AddressSanitizer and
 * UndefinedBehaviorSanitizer checks the validation code on a machine without a
 * GPU.  Device pointers are fake, 16-byte aligned addresses that the
 * validation never dereferences.  Exit status 0 and "ok" when every call
 * returns the status the header documents. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn.h"
#include "gdn_proj.h"

static int fails = 0;
#define EXPECT(call, want)                                                              \
    do {                                                                                \
        const int got_ = (int)(call);                                                   \
        if (got_ != (int)(want)) {                                                      \
            printf("line %d: %s -> %d, expected %d\n", __LINE__, #call, got_, (int)(want)); \
            ++fails;                                                                    \
        }                                                                               \
    } while (0)

static void* P(uintptr_t k) { return (void*)(uintptr_t)(0x10000000u + k * 0x1000000u); }

int main(void) {
    gdn_dims d = {16, 32, 1e-6f, GDN_BF16, GDN_F32, 0};
    gdn_weights w = {(const float*)P(1), (const float*)P(2), (const float*)P(3), (const float*)P(4)};
    gdn_dims bad = d;

    for (int s = 0; s <= 6; ++s) EXPECT(strlen(gdn_status_string((gdn_status)s)) > 0, 1);
    EXPECT(strcmp(gdn_status_string((gdn_status)99), "unknown status"), 0);
    EXPECT(gdn_version() >= 100, 1);

    /* dims */
    EXPECT(gdn_decode_step(NULL, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_INVALID_ARG);
    bad.H_v = 40;
    EXPECT(gdn_decode_step(&bad, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_INVALID_ARG);
    bad = d; bad.H_k = 1; bad.H_v = 17;
    EXPECT(gdn_decode_step(&bad, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_UNSUPPORTED);
    bad = d; bad.eps = 0.0f;
    EXPECT(gdn_decode_step(&bad, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_INVALID_ARG);
    bad = d; bad.flags = 0x80;
    EXPECT(gdn_decode_step(&bad, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_INVALID_ARG);
    bad = d; bad.act_dtype = GDN_F32; bad.flags = GDN_FLAG_STATE_BF16;
    EXPECT(gdn_decode_step(&bad, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_UNSUPPORTED);

    /* decode */
    EXPECT(gdn_decode_step(&d, &w, -1, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_decode_step(&d, &w, 0, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_OK);
    EXPECT(gdn_decode_step(&d, NULL, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_decode_step(&d, &w, 4, (char*)P(5) + 8, P(6), P(7), P(8), P(9), P(10), P(11), NULL, NULL, NULL),
           GDN_E_ALIGNMENT);
    EXPECT(gdn_decode_step(&d, &w, 4, P(5), P(6), P(7), P(8), P(9), P(10), P(5), NULL, NULL, NULL), GDN_E_INVALID_ARG);

    /* verify / commit */
    EXPECT(gdn_verify_k(&d, &w, 2, 0, P(5), P(6), P(7), P(8), P(9), P(10), P(11), P(12), P(13), NULL, NULL, NULL),
           GDN_E_INVALID_ARG);
    EXPECT(gdn_verify_k(&d, &w, 2, GDN_MAX_VERIFY_K + 1, P(5), P(6), P(7), P(8), P(9), P(10), P(11), P(12), P(13), NULL,
                        NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_verify_k(&d, &w, 2, 3, P(5), P(6), P(7), P(8), P(9), P(10), P(11), P(10), P(13), NULL, NULL, NULL),
           GDN_E_INVALID_ARG);
    EXPECT(gdn_commit(&d, 2, 0, (const int32_t*)P(5), P(6), P(7), P(8), P(9), NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_commit(&d, 2, 3, NULL, P(6), P(7), P(8), P(9), NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_commit_ring(&d, 2, 3, 3, (const int32_t*)P(5), P(6), P(7), (int32_t*)P(8), NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_verify_k_ring(&d, &w, 2, 3, 2, P(5), P(6), P(7), P(8), P(9), P(10), (const int32_t*)P(11), P(12), P(13),
                             NULL, NULL, NULL), GDN_E_INVALID_ARG);

    /* guard */
    EXPECT(gdn_state_faults(&d, -1, (const int32_t*)P(5), 2, (int32_t*)P(6), NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_state_faults(&d, 4, (const int32_t*)P(5), -1, (int32_t*)P(6), NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_state_reset(&d, 4, 2, P(5), NULL, NULL, (int32_t*)P(6), NULL), GDN_E_INVALID_ARG);

    /* prefill */
    const int32_t cu_bad[3] = {1, 5, 9};
    const int32_t cu_dec[3] = {0, 9, 5};
    const int32_t cu_ok[3] = {0, 70, 100};
    EXPECT(gdn_prefill_chunked(&d, &w, 2, cu_bad, (const int32_t*)P(5), P(6), P(7), P(8), P(9), P(10), P(11), 1, P(12),
                               NULL, P(13), 1u << 30, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_prefill_chunked(&d, &w, 2, cu_dec, (const int32_t*)P(5), P(6), P(7), P(8), P(9), P(10), P(11), 1, P(12),
                               NULL, P(13), 1u << 30, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_prefill_chunked(&d, &w, 2, cu_ok, (const int32_t*)P(5), P(6), P(7), P(8), P(9), P(10), P(11), 1, P(12),
                               NULL, NULL, 0, NULL, NULL), GDN_E_WORKSPACE);
    EXPECT(gdn_prefill_chunked(&d, &w, -1, cu_ok, (const int32_t*)P(5), P(6), P(7), P(8), P(9), P(10), P(11), 1, P(12),
                               NULL, P(13), 1u << 30, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_prefill_workspace_bytes(&d, 1, 0) > 0, 1);
    EXPECT(gdn_prefill_workspace_bytes(&d, 1, 8192) >= gdn_prefill_workspace_bytes(&d, 1, 4096), 1);
    EXPECT(gdn_prefill_workspace_bytes(NULL, 1, 64), 0);
    bad = d; bad.act_dtype = GDN_F32;
    EXPECT(gdn_prefill_workspace_bytes(&bad, 1, 64), 0);
    const int32_t cu_big[2] = {0, 1 << 20};
    EXPECT(gdn_prefill_chunked_static(&d, &w, 1, cu_big, (const int32_t*)P(5), P(6), P(7), P(8), P(9), P(10), P(11), 1,
                                      P(12), NULL, NULL, NULL), GDN_E_WORKSPACE);

    /* projections */
    gdn_in_proj_weights pw = {P(1), P(2), P(3), P(4)};
    EXPECT(gdn_in_proj(&d, 4, 2048, P(5), &pw, P(6), P(7), P(8), P(9), NULL, 0, NULL, NULL), GDN_E_UNSUPPORTED);   /* fp32 out */
    d.out_dtype = GDN_BF16;   /* the projections run bf16 in and out */
    EXPECT(gdn_in_proj(&d, -1, 2048, P(5), &pw, P(6), P(7), P(8), P(9), NULL, 0, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_in_proj(&d, 4, 2044, P(5), &pw, P(6), P(7), P(8), P(9), NULL, 0, NULL, NULL), GDN_E_INVALID_ARG);
    EXPECT(gdn_in_proj(&d, 4, 2048, P(5), &pw, P(6), P(7), P(8), P(9), NULL, 0, (int32_t*)((char*)P(10) + 2), NULL),
           GDN_E_ALIGNMENT);
    EXPECT(gdn_in_proj(&d, 0, 2048, P(5), &pw, P(6), P(7), P(8), P(9), NULL, 0, NULL, NULL), GDN_OK);
    EXPECT(gdn_out_proj(&d, 4, 2048, NULL, P(6), P(7), NULL, 0, NULL, NULL), GDN_E_INVALID_ARG);

    printf(fails ? "%d failures\n" : "ok\n", fails);
    return fails ? 1 : 0;
}

/*
 * The library's host-side argument checks under AddressSanitizer and
 * UndefinedBehaviorSanitizer (built and run by tests/test_sanitizers.py
 * against a sanitized build of the library's host code).  Every call here is
 * rejected before any CUDA call or launch: fake device addresses are never
 * dereferenced.  Exit status 0: every call returned the expected status.
 */
#include <stdio.h>
#include <stdint.h>
#include <string.h>

#include "rvqmoe.h"

static int failures = 0;
#define EXPECT(call, want)                                                              \
    do {                                                                                \
        const int _got = (int)(call);                                                   \
        if (_got != (int)(want)) {                                                      \
            fprintf(stderr, "line %d: %s returned %d, expected %d (%s)\n", __LINE__,      \
                    #call, _got, (int)(want), rvq_last_error());                         \
            ++failures;                                                                 \
        }                                                                               \
    } while (0)

static uint64_t state = 400;
static int pick(const int *v, int nv)
{
    state = state * 6364136223846793005ULL + 1442695040888963407ULL;
    return v[(state >> 33) % (uint64_t)nv];
}

int main(void)
{
    void *A16 = (void *)(uintptr_t)0x10000, *A256 = (void *)(uintptr_t)0x20000;
    char *A16c = (char *)A16;
    rvq_stream_t s = NULL;
    for (int c = 0; c < 12; ++c) (void)strlen(rvq_status_string((rvq_status)c));
    EXPECT(rvq_code_bytes(32, 512), 3 * 32 * 512 / 8);
    EXPECT(rvq_code_bytes(33, 512), 0);
    EXPECT(rvq_code_bytes(-32, 512), 0);
    EXPECT(rvq_pack(A16, 33, 512, A16, 1 << 20, s), RVQ_EINVAL);
    EXPECT(rvq_pack(A16, 32, 512, (uint8_t *)(A16c + 4), 1 << 20, s), RVQ_EALIGN);
    EXPECT(rvq_pack(A16, 32, 512, A16, 100, s), RVQ_ENOMEM);
    EXPECT(rvq_unpack(A16, 32, 512, A16, 100, s), RVQ_ENOMEM);
    EXPECT(rvq_lut_build(A16, A16, RVQ_F32, 1, 12, A16, s), RVQ_EINVAL);
    EXPECT(rvq_gemv(A16, A16, 256, 512, A16c + 8, RVQ_F32, 1, A16, A256, 1 << 20, s), RVQ_EALIGN);
    EXPECT(rvq_gemv(A16, A16, 256, 512, A16, RVQ_F32, 1, A16, A256, 16, s), RVQ_ENOMEM);
    EXPECT(rvq_gemv(A16, A16, 256, 512, A16, RVQ_F32, 0, A16, A256, 1 << 20, s), RVQ_EINVAL);
    EXPECT(rvq_gemv(NULL, A16, 256, 512, A16, RVQ_F32, 1, A16, A256, 1 << 20, s), RVQ_EINVAL);
    /* the no-allocation GEMV: shape, alignment and size checks before anything */
    EXPECT(rvq_gemv_noalloc(A16, A16, 250, 512, A16, RVQ_F32, 1, A16, s), RVQ_EINVAL);
    EXPECT(rvq_gemv_noalloc(A16, A16, 256, 512, A16c + 4, RVQ_F32, 1, A16, s), RVQ_EALIGN);
    EXPECT(rvq_gemv_noalloc(A16, A16, 7168, 2048, A16, RVQ_F32, 1024, A16, s), RVQ_ENOMEM);
    EXPECT(moe_router_logits(A16, NULL, A16, RVQ_BF16, 1, 300, 512, A16, s), RVQ_EINVAL);
    EXPECT(moe_route(A16, 4, 8, 9, A16, A16, A16, A16, A256, 256, s), RVQ_EINVAL);
    EXPECT(moe_route(A16, 4, 64, 8, A16, A16, A16, A16, A256, 8, s), RVQ_ENOMEM);
    EXPECT(moe_combine(A16, A16, 2, 2, 6, A16, RVQ_F32, A16, s), RVQ_EINVAL);
    EXPECT(rvq_encode(A16, 1, 2040, 2, A16, A16, A256, 1 << 20, s), RVQ_EINVAL);
    rvq_moe_bank bank;
    const uint64_t rb = moe_bank_record_bytes(2048, 1024);
    EXPECT(moe_bank_init(&bank, A256, rb * 64, 64, 2048, 1024, 3), RVQ_OK);
    EXPECT(moe_bank_init(&bank, (uint8_t *)A256 + 16, rb * 64, 64, 2048, 1024, 0), RVQ_EALIGN);
    EXPECT(moe_bank_init(&bank, A256, rb * 64, 64, 2000, 1024, 0), RVQ_EINVAL);
    EXPECT(moe_bank_init(&bank, A256, rb * 64, 64, 2048, 1024, 3), RVQ_OK);
    if (moe_workspace_bytes(&bank, 1, 8) <= 256) ++failures;
    /* the host-buffer layer call: null host buffers, a short workspace */
    EXPECT(moe_layer_forward_host(&bank, A16, NULL, NULL, RVQ_BF16, 1, 8, A16, A16, A16, A16, A16,
                                  A16, A16, (float *)A16, A256, 1 << 30, 0, s),
           RVQ_EINVAL);
    float host_out[4];
    uint16_t host_x[4];
    EXPECT(moe_layer_forward_host(&bank, A16, NULL, host_x, RVQ_BF16, 1, 8, A16, A16, A16, A16,
                                  A16, A16, A16, host_out, A256, 16, 0, s),
           RVQ_ENOMEM);
    /* 400 random shapes: invalid ones never pass the checks */
    const int R[] = {0, 1, 31, 32, 64, 96, 2048, -32, 1 << 20};
    const int C[] = {0, 8, 256, 511, 512, 1024, 7168, -512};
    for (int i = 0; i < 400; ++i) {
        const int rows = pick(R, 9), cols = pick(C, 8);
        const int valid = rows > 0 && cols > 0 && rows % 32 == 0 && cols % 512 == 0;
        const int rc = rvq_pack(A16, rows, cols, (uint8_t *)(A16c + 4 * (i & 1)), 0, s);
        if (!valid && rc != RVQ_EINVAL) ++failures;
        if (valid && rc != RVQ_EALIGN && rc != RVQ_ENOMEM) ++failures;
    }
    if (failures) fprintf(stderr, "host checks: %d failures\n", failures);
    printf("host checks done\n");
    return failures ? 1 : 0;
}

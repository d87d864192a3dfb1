/* Plain C99 caller of the library's C ABI: the header must compile as C, and the entry points
 * must link and answer their host-side checks without a GPU.  Built and run by
 * tests/test_c_abi.py; prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "moe.h"

static int fails = 0;
#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            ++fails;                                                  \
        }                                                             \
    } while (0)

int main(void) {
    void* fake = (void*)0x1000;
    moe_q4 q = {(const uint8_t*)0x1000, (const uint16_t*)0x2000};
    moe_experts bad_fmt = {8, 256, 128, q, q, q, 7};
    moe_experts ok = {8, 256, 128, q, q, q, MOE_WFMT_MXFP4};
    moe_shared sh = {64, q, q, q, NULL, MOE_WFMT_INT4};

    CHECK(strcmp(moe_status_string(MOE_OK), "ok") == 0);
    CHECK(strstr(moe_version(), "sm_103a") != NULL);
    CHECK(moe_workspace_size(16, 128, 8, 2048, 768, 0) > moe_workspace_size(1, 128, 8, 2048, 768, 0));
    CHECK(moe_dispatch_workspace_size(16384, 8, 256) > 0);
    /* rejected on the host before any device work */
    CHECK(moe_router_topk(fake, 0, 8, 4, 8, 9, (int32_t*)fake, (float*)fake, NULL) == MOE_ERR_INVALID_ARG);
    CHECK(moe_layer_forward((const uint16_t*)fake, NULL, (const uint16_t*)fake, &bad_fmt, NULL, 4, 2,
                            (float*)fake, NULL, NULL, MOE_ARM_AUTO, (void*)0x10000, (size_t)1 << 30,
                            NULL) == MOE_ERR_INVALID_ARG);
    CHECK(moe_layer_forward((const uint16_t*)fake, NULL, (const uint16_t*)fake, &ok, &sh, 0, 2, (float*)fake,
                            NULL, NULL, MOE_ARM_AUTO, (void*)0x10000, (size_t)1 << 30, NULL) == MOE_OK);
    CHECK(moe_mxfp4_scales(NULL, 16, (uint16_t*)fake, fake, 4096, NULL) == MOE_ERR_INVALID_ARG);
    CHECK(moe_rmsnorm((const float*)fake, (const uint16_t*)fake, 4, 100, 1e-6f, (uint16_t*)fake, NULL) ==
          MOE_ERR_INVALID_ARG);
    if (fails) return 1;
    printf("ok\n");
    return 0;
}

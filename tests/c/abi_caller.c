/* A C-only caller of libsoftmax: checks that include/softmax.h compiles as
 * C, that the library links, and the host-side behaviour that needs no GPU
 * (argument validation, status strings, the scheduler on a described GB300). */
#include <stdio.h>
#include <string.h>

#include "softmax.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #c); return 1; } } while (0)

int main(void)
{
    float buf[64];
    CHECK(softmax_abi_version() == SOFTMAX_ABI_VERSION);
    CHECK(strcmp(softmax_status_string(SOFTMAX_OK), "ok") == 0);
    CHECK(softmax_status_string(12345) != NULL);
    /* Validation happens before any device call. */
    CHECK(softmax_rows(buf, buf + 32, -1, 4, 4, 4, SOFTMAX_F32, NULL) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_rows(buf, buf + 32, 2, 4, 3, 4, SOFTMAX_F32, NULL) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_rows(NULL, buf, 2, 4, 4, 4, SOFTMAX_F32, NULL) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_rows(buf, buf + 32, 2, 4, 4, 4, 7, NULL) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_rows(buf, buf + 2, 2, 4, 4, 4, SOFTMAX_F32, NULL) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_rows(NULL, NULL, 0, 4, 4, 4, SOFTMAX_F32, NULL) == SOFTMAX_OK);
    CHECK(softmax_rows_path(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, NULL, 9) == SOFTMAX_ERR_INVALID_ARG);
    /* softmax_rows_ex: options are checked before any device call too. */
    softmax_options_t opt = {0.125f, 1, 0, 0};
    CHECK(softmax_rows_ex(NULL, NULL, 0, 4, 4, 4, SOFTMAX_F32, &opt, SOFTMAX_PATH_AUTO, NULL) == SOFTMAX_OK);
    opt.scale = 0.0f;
    CHECK(softmax_rows_ex(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, &opt, SOFTMAX_PATH_AUTO, NULL) == SOFTMAX_ERR_INVALID_ARG);
    opt.scale = -1.0f;
    CHECK(softmax_rows_ex(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, &opt, SOFTMAX_PATH_AUTO, NULL) == SOFTMAX_ERR_INVALID_ARG);
    opt.scale = 3.0e38f;
    CHECK(softmax_rows_ex(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, &opt, SOFTMAX_PATH_AUTO, NULL) == SOFTMAX_ERR_INVALID_ARG);
    opt.scale = 1.0f;
    opt.causal = 2;
    CHECK(softmax_rows_ex(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, &opt, SOFTMAX_PATH_AUTO, NULL) == SOFTMAX_ERR_INVALID_ARG);
    opt.causal = 1;
    opt.causal_offset = (int64_t)1 << 62;
    CHECK(softmax_rows_ex(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, &opt, SOFTMAX_PATH_AUTO, NULL) == SOFTMAX_ERR_INVALID_ARG);
    opt.causal_offset = 0;
    CHECK(softmax_rows_ex(buf, buf + 32, 1, 4, 4, 4, SOFTMAX_F32, &opt, 7, NULL) == SOFTMAX_ERR_INVALID_ARG);

    softmax_device_desc_t gb300 = {152, 2048, 233472, 232448, 65536, 10, 3, 16};
    softmax_plan_t plan;
    char text[256];
    CHECK(softmax_plan(&gb300, (void*)0x10000, (void*)0x20000000, 4096, 4096, 4096, 4096,
                       SOFTMAX_F32, SOFTMAX_PATH_AUTO, &plan) == SOFTMAX_OK);
    CHECK(plan.path == SOFTMAX_PATH_CTA && plan.bulk_copy == 1 && plan.cluster == 1 && plan.stages == 2);
    CHECK(softmax_plan_format(&plan, text, sizeof text) > 0 && strstr(text, "path=cta"));
    CHECK(softmax_plan(&gb300, (void*)0x10000, (void*)0x20000000, 256, 262144, 262144, 262144,
                       SOFTMAX_F32, SOFTMAX_PATH_AUTO, &plan) == SOFTMAX_OK);
    CHECK(plan.path == SOFTMAX_PATH_TWOPASS && plan.cluster == 4 && plan.stages == 3);
    /* softmax_plan_check: the scheduler's plan passes; one that no longer
     * covers the row is refused. */
    CHECK(softmax_plan_check(&gb300, (void*)0x10000, (void*)0x20000000, 256, 262144, 262144,
                             262144, SOFTMAX_F32, &plan) == SOFTMAX_OK);
    plan.slice_cols /= 2;
    CHECK(softmax_plan_check(&gb300, (void*)0x10000, (void*)0x20000000, 256, 262144, 262144,
                             262144, SOFTMAX_F32, &plan) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_plan_check(&gb300, (void*)0x10000, (void*)0x20000000, 256, 262144, 262144,
                             262144, SOFTMAX_F32, NULL) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_plan(&gb300, (void*)0x10000, (void*)0x20000000, 1 << 20, 16, 16, 16,
                       SOFTMAX_F32, SOFTMAX_PATH_AUTO, &plan) == SOFTMAX_OK);
    CHECK(plan.path == SOFTMAX_PATH_WARP && plan.lanes_per_row == 4);
    /* softmax_plan_describe: the same decision on the current device (none
     * here: UNSUPPORTED, never a made-up plan); its arguments are checked
     * first. */
    CHECK(softmax_plan_describe(4096, 4096, 7, text, sizeof text) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_plan_describe(-1, 4096, SOFTMAX_F32, text, sizeof text) == SOFTMAX_ERR_INVALID_ARG);
    CHECK(softmax_plan_describe(4096, 4096, SOFTMAX_F32, NULL, 16) == SOFTMAX_ERR_INVALID_ARG);
    {
        const int st = softmax_plan_describe(4096, 4096, SOFTMAX_F32, text, sizeof text);
        CHECK(st == SOFTMAX_OK ? strstr(text, "path=cta") != NULL : st == SOFTMAX_ERR_UNSUPPORTED);
    }
    gb300.cc_minor = 0;
    CHECK(softmax_plan(&gb300, (void*)0x10000, (void*)0x20000000, 4, 4, 4, 4, SOFTMAX_F32,
                       SOFTMAX_PATH_AUTO, &plan) == SOFTMAX_ERR_UNSUPPORTED);
    printf("ok\n");
    return 0;
}

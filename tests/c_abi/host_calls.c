/* Plain C99 client of include/kdaproj.h: links against libkdaproj.so and makes
 * the calls that need no GPU (argument checks, configuration helpers). Exits 0
 * when every result is the documented one, else prints the failed check. */
#include <stdio.h>
#include <string.h>

#include "kdaproj.h"

static int failures = 0;

static void check(int cond, const char *what) {
    if (!cond) {
        fprintf(stderr, "FAILED: %s (last error: %s)\n", what, kp_last_error());
        ++failures;
    }
}

int main(void) {
    char buf[64];
    void *p = buf + (16 - ((size_t)buf & 15));   /* 16-byte aligned host address, never used */
    kp_cfg cfg;
    kda_plan *plan = NULL;
    size_t bytes = 1;

    check(kp_version() == KDAPROJ_VERSION, "kp_version");
    check(skinny_gemm(p, p, p, 1, 8, 12, NULL, NULL) == KP_ESHAPE, "K not a multiple of 8");
    check(strstr(kp_last_error(), "multiple of 8") != NULL, "error text");
    check(skinny_gemm(p, p, p, 0, 8, 16, NULL, NULL) == KP_OK, "M = 0 is a no-op");
    check(skinny_gemm_ex(p, p, NULL, p, 1, 8, 16, 7, NULL, NULL) == KP_EINVAL, "element type");
    check(kda_proj_plan(7168, 4096, 100, 1024, 16, &plan) == KP_ESHAPE, "N_fab < 128");
    check(kda_proj_run(NULL, p, p, p, p, p, p, 1, NULL, NULL, NULL) == KP_ENOPLAN, "no plan");
    check(kda_proj_destroy(NULL) == KP_OK, "destroy NULL");

    memset(&cfg, 0, sizeof cfg);
    check(kp_select_config(1, 4096, 7168, 152, &cfg) == KP_OK, "kp_select_config");
    check(cfg.kind == KP_KIND_CC || cfg.kind == KP_KIND_TC05 || cfg.kind == KP_KIND_SMALLK,
          "selected kind");
    check(kp_scratch_bytes(1, 4096, 7168, &cfg, 152, &bytes) == KP_OK, "scratch of the selection");
    cfg.kind = KP_KIND_TC05;
    cfg.split_k = 3;   /* clusters are 1, 2, 4, 8 or 16 CTAs */
    check(kp_scratch_bytes(1, 4096, 7168, &cfg, 152, &bytes) == KP_ECONFIG, "bad cluster size");
    check(kp_table_clear() == KP_OK && kp_table_size() == 0, "table clear");

    if (failures == 0) printf("c abi ok\n");
    return failures == 0 ? 0 : 1;
}

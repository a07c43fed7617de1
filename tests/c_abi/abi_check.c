/* Host-side use of the C ABI from plain C99: the header compiles as C, the
 * library links and answers without any CUDA work (handle creation, groups,
 * argument validation, status strings).  Exit status 0 on success; a
 * message on stderr names the first failed check. */
#include <stdio.h>
#include <string.h>

#include "soma_opt.h"

#define CHECK(cond)                                              \
    do {                                                         \
        if (!(cond)) {                                           \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                            \
        }                                                        \
    } while (0)

int main(void) {
    CHECK(soma_abi_version() == SOMA_ABI_VERSION);
    CHECK(strcmp(soma_status_string(SOMA_OK), "ok") == 0);
    CHECK(sizeof(soma_tensor_t) == 56);
    CHECK(sizeof(soma_device_group_t) == 64);

    soma_opt_t opt = NULL;
    CHECK(soma_opt_create(&opt, 0) == SOMA_OK && opt != NULL);
    int32_t g = -1;
    CHECK(soma_opt_add_group(opt, 1e-3, 0.9, 0.999, 1e-8, 0.01, &g) == SOMA_OK && g == 0);
    CHECK(soma_opt_add_group(opt, -1.0, 0.9, 0.999, 1e-8, 0.0, &g) == SOMA_ERR_INVALID_ARG);
    CHECK(strstr(soma_opt_last_error(opt), "lr") != NULL);

    /* an entry naming an unknown group: rejected before any CUDA call */
    soma_tensor_t t;
    memset(&t, 0, sizeof t);
    t.param = (float *)0x10000;
    t.grad = (const void *)0x20000;
    t.exp_avg = (float *)0x30000;
    t.exp_avg_sq = (float *)0x40000;
    t.numel = 8;
    t.group = 3;
    t.grad_dtype = SOMA_DTYPE_F32;
    t.trainable = 1;
    t.owned = 1;
    CHECK(soma_opt_step(opt, &t, 1, 4.0, 1.0, NULL) == SOMA_ERR_BAD_GROUP);
    CHECK(soma_opt_step(opt, &t, 1, 0.0, 1.0, NULL) == SOMA_ERR_INVALID_ARG);
    int64_t step = -1;
    CHECK(soma_opt_get_group_step(opt, 0, &step) == SOMA_OK && step == 0);
    CHECK(soma_opt_set_group_step(opt, 0, 41) == SOMA_OK);
    CHECK(soma_opt_get_group_step(opt, 0, &step) == SOMA_OK && step == 41);

    int64_t builds = -1, reuses = -1;
    int32_t entries = -1;
    CHECK(soma_opt_get_cache_stats(opt, &builds, &reuses, &entries) == SOMA_OK);
    CHECK(builds == 0 && reuses == 0 && entries == 0);

    /* host-side knobs: tuning and the single-launch limit */
    CHECK(soma_opt_set_tuning(opt, 4096, 8192, 0, 0) == SOMA_OK);
    CHECK(soma_opt_set_tuning(opt, 10, 0, 0, 0) == SOMA_ERR_INVALID_ARG);
    CHECK(soma_opt_set_single_launch(opt, 0) == SOMA_OK);
    CHECK(soma_opt_set_single_launch(opt, -1) == SOMA_OK);
    CHECK(soma_opt_set_single_launch(opt, -2) == SOMA_ERR_INVALID_ARG);
    soma_plan_t plan;
    memset(&plan, 0xff, sizeof plan);
    CHECK(soma_opt_get_plan(opt, &plan) == SOMA_OK);
    CHECK(plan.launches_per_step == 0 && plan.single_launch_ctas == 0); /* no step yet */
    CHECK(sizeof(soma_plan_t) == 72);

    soma_opt_destroy(opt);
    CHECK(soma_opt_set_lr(opt, 0, 1e-3) == SOMA_ERR_STATE); /* a destroyed handle is refused */
    puts("c abi ok");
    return 0;
}

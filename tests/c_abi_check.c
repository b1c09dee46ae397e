/*
 * A plain C99 client of include/bf16_linear.h: it must compile as C (not C++),
 * link against the library, and get sensible answers from the host-only entry
 * points (no GPU is touched).  Run by tests/test_c_abi.py; prints one line per
 * check and exits non-zero on the first failure.
 */
#include <stdio.h>
#include <string.h>

#include "bf16_linear.h"

#define CHECK(cond, what)                              \
    do {                                               \
        if (!(cond)) {                                 \
            printf("FAIL %s\n", what);                 \
            return 1;                                  \
        }                                              \
        printf("ok %s\n", what);                       \
    } while (0)

int main(void) {
    bf16l_plan p;
    bf16l_device gb300 = {10, 3, 152};
    bf16l_device hopper = {9, 0, 132};
    memset(&p, 0, sizeof p);

    CHECK(bf16_linear_version() > 0, "version");
    CHECK(bf16_linear_plan(16, 256, 7168, &p) == BF16L_OK && p.grid > 0, "plan for a router shape");
    CHECK(bf16_linear_plan(16, 256, 7168, NULL) == BF16L_EINVAL, "a NULL plan is refused");
    CHECK(bf16_linear_plan_for_device(16, 256, 7168, NULL, &p) == BF16L_OK, "plan for the default device");
    CHECK(bf16_linear_plan_for_device(16, 256, 7168, &gb300, &p) == BF16L_OK, "plan with an explicit GB300 device");
    CHECK(bf16_linear_plan_for_device(16, 256, 7168, &hopper, &p) == BF16L_EARCH, "other architectures are refused");
    CHECK(bf16_linear_plan(-1, 256, 7168, &p) == BF16L_EINVAL, "negative M is refused");
    CHECK(bf16_linear_plan_check(16, 256, 7168, NULL, &p) == BF16L_OK, "the planner's own plan checks");
    p.threads = 33;
    CHECK(bf16_linear_plan_check(16, 256, 7168, NULL, &p) != BF16L_OK, "a broken plan does not");
    CHECK(bf16_linear_plan(16, 256, 7168, &p) == BF16L_OK &&
              bf16_linear_workspace_size(16, 256, 7168, &p) == 0, "the planner's plans need no workspace");
    CHECK(bf16_linear_host_staging_bytes(4, 256, 2048, 0) == 16384 + 1048576 + 2048, "host staging bytes");
    CHECK(bf16_linear_noalloc_scratch_bytes() == 4u << 20, "no-alloc scratch is 4 MiB");
    CHECK(bf16_linear_fp8_split(1, 256, 7168, 152) >= 1, "fp8 split");
    CHECK(strlen(bf16_linear_strerror(BF16L_EALIGN)) > 0, "strerror");
    CHECK(bf16_linear(NULL, NULL, NULL, NULL, 0, 256, 7168, NULL) == BF16L_OK, "M == 0 is a no-op");
    CHECK(bf16_linear(NULL, NULL, NULL, NULL, 4, 0, 7168, NULL) == BF16L_EINVAL, "N == 0 is refused");
    return 0;
}

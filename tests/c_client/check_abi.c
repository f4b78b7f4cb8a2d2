/* A plain C client of the library: includes only include/moe.h (no CUDA or torch
 * headers), links libmoe.so and exercises the entry points that need no GPU -- sizing,
 * validation before any launch, the TP slice rule, status strings. Prints one line per
 * check and exits non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "moe.h"

static int failures = 0;
#define CHECK(cond, what)                                  \
    do {                                                   \
        if (!(cond)) {                                     \
            printf("FAIL %s (%s)\n", (what), moe_last_error()); \
            failures++;                                    \
        } else {                                           \
            printf("ok   %s\n", (what));                   \
        }                                                  \
    } while (0)

static moe_config base_config(void) {
    moe_config c;
    memset(&c, 0, sizeof c);
    c.num_tokens = 8192;
    c.hidden = 2880;
    c.intermediate = 2880;
    c.num_experts = 128;
    c.top_k = 4;
    c.ep_size = 8;
    c.capacity_factor = 0.0f;
    c.mode = MOE_MODE_DISPATCH;
    c.dtype = MOE_DTYPE_BF16;
    return c;
}

int main(void) {
    size_t bytes = 0, train_bytes = 0, packed = 0;
    moe_config c = base_config();
    CHECK(moe_workspace_size(&c, &bytes) == MOE_OK && bytes > 0, "workspace size");
    CHECK(moe_packed_gate_up_size(&c, &packed) == MOE_OK &&
              packed == (size_t)128 * 2 * 2944 * 2880 * 2,
          "packed gate/up size: E x 2 Ipad x H bf16, Ipad = 2944");
    c.training = 1;
    CHECK(moe_workspace_size(&c, &train_bytes) == MOE_OK && train_bytes > bytes,
          "training workspace is larger");
    c = base_config();
    c.ep_size = 7;
    CHECK(moe_workspace_size(&c, &bytes) == MOE_ERR_INVALID_ARG, "ep_size must divide E");
    c = base_config();
    c.hidden = 2881;
    CHECK(moe_workspace_size(&c, &bytes) == MOE_ERR_INVALID_ARG, "hidden multiple of 8");
    c = base_config();
    c.capacity_priority = 5;
    CHECK(moe_workspace_size(&c, &bytes) == MOE_ERR_INVALID_ARG, "capacity priority checked");
    c = base_config();
    /* rejected before any launch: a NULL workspace */
    CHECK(moe_layer_forward(&c, (void *)16, (void *)16, NULL, (void *)16, (void *)16, (void *)16,
                            NULL, NULL, 0, NULL) == MOE_ERR_WORKSPACE,
          "forward without workspace is rejected before any launch");
    int64_t b = -1, e = -1, total = 0;
    int ok_slices = 1;
    for (int r = 0; r < 3; ++r) {
        ok_slices &= moe_tp_slice(7, 3, r, &b, &e) == MOE_OK;
        total += e - b;
    }
    CHECK(ok_slices && total == 7, "TP slices of 7 tokens over 3 ranks cover them");
    CHECK(moe_tp_slice(1, 2, 1, &b, &e) == MOE_OK && b == 1 && e == 1,
          "single decode token: the second TP rank's slice is empty");
    CHECK(moe_tp_slice(4, 2, 2, &b, &e) == MOE_ERR_INVALID_ARG, "TP rank out of range");
    CHECK(strcmp(moe_status_string(MOE_ERR_TIMEOUT), "MOE_ERR_TIMEOUT") == 0, "status strings");
    printf("%d failure(s)\n", failures);
    return failures == 0 ? 0 : 1;
}

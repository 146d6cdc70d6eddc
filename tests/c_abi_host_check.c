/* A plain C caller of libsdpa.so (compiled with gcc, linked to the library):
 * the header must be valid C and the host-side entry points usable without
 * C++ or Python. Only calls that touch no GPU are made: validation,
 * workspace sizes, error strings and host-detected declines.
 * Prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "sdpa.h"

static int fails = 0;
#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            printf("check failed at line %d: %s\n", __LINE__, #cond); \
            ++fails;                                                  \
        }                                                             \
    } while (0)

int main(void) {
    sdpa_problem p;
    memset(&p, 0, sizeof p);
    p.layout = SDPA_THD;
    p.dtype = SDPA_BF16;
    p.mask_type = SDPA_MASK_CAUSAL_TOP_LEFT;
    p.batch = 8;
    p.seqlen_q = p.seqlen_kv = 4096;
    p.total_q = p.total_kv = 19339;
    p.num_heads_q = 32;
    p.num_heads_kv = 8;
    p.head_dim = 128;
    p.window_left = p.window_right = -1;
    p.softmax_scale = 0.08838834764831845f;
    CHECK(sdpa_check_problem(&p) == SDPA_OK);
    CHECK(sdpa_fwd_workspace_size(&p) == 256);
    CHECK(sdpa_bwd_workspace_size(&p) > 0);

    p.head_dim = 64;
    CHECK(sdpa_check_problem(&p) == SDPA_ERR_UNSUPPORTED);
    CHECK(sdpa_bwd_workspace_size(&p) == 0);
    p.head_dim = 192;
    p.head_dim_v = 128;  /* the forward-only pair */
    CHECK(sdpa_check_problem(&p) == SDPA_OK);
    CHECK(sdpa_bwd_workspace_size(&p) == 0);
    p.head_dim = 128;
    p.head_dim_v = 0;
    p.num_heads_kv = 5;
    CHECK(sdpa_check_problem(&p) == SDPA_ERR_INVALID_ARG);
    p.num_heads_kv = 8;

    /* host-detected declines return before any CUDA call */
    CHECK(sdpa_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) == SDPA_ERR_INVALID_ARG);
    CHECK(sdpa_fwd(&p, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) == SDPA_ERR_INVALID_ARG);
    sdpa_merge_problem m = {SDPA_BF16, 10, 128, 0};
    CHECK(sdpa_merge(&m, NULL, NULL, NULL, NULL, NULL) == SDPA_ERR_INVALID_ARG);

    for (int code = SDPA_OK; code <= SDPA_ERR_CUDA; ++code) CHECK(sdpa_error_string(code) != NULL);
    CHECK(strcmp(sdpa_error_string(SDPA_OK), "ok") == 0);

    if (fails) return 1;
    printf("ok\n");
    return 0;
}

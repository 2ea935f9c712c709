/* A plain C11 consumer of include/conv_bn_silu.h: the header must compile as C
 * (no C++ types or keywords), link against libconvbnsilu.so, and its host-only
 * entry points must answer without a GPU.  Exit code 0 when every check holds;
 * otherwise the number of the first failed check. */
#include <stdio.h>
#include <string.h>

#include "conv_bn_silu.h"

#define CHECK(n, cond)                                  \
    do {                                                \
        if (!(cond)) {                                  \
            fprintf(stderr, "check %d failed: %s\n", n, #cond); \
            return n;                                   \
        }                                               \
    } while (0)

int main(void)
{
    int ho = 0, wo = 0;
    CHECK(1, conv_bn_silu_output_dims(640, 640, 3, 3, 2, 2, 1, 1, &ho, &wo) == CBS_OK);
    CHECK(2, ho == 320 && wo == 320);
    CHECK(3, conv_bn_silu_output_dims(2, 2, 3, 3, 1, 1, 0, 0, &ho, &wo) == CBS_ERR_INVALID_ARG);

    cbs_plan_info info;
    memset(&info, 0, sizeof info);
    CHECK(4, conv_bn_silu_plan(32, 20, 20, 512, 512, 3, 3, 1, 1, 1, 1, CBS_ALGO_AUTO, 152, &info) == CBS_OK);
    CHECK(5, info.algo == CBS_ALGO_TCGEN05 && info.stream_k == 1 && info.cluster == 2);
    CHECK(6, info.workspace_bytes > 0);

    cbs_plan_request req;
    memset(&req, 0, sizeof req);
    req.algo = CBS_ALGO_AUTO;
    req.swap_ab = -1;
    req.stream_k = 0;
    req.pair = -1;
    req.block_n = 0;
    CHECK(7, conv_bn_silu_plan_request(32, 20, 20, 512, 512, 3, 3, 1, 1, 1, 1, &req, 152, &info) == CBS_OK);
    CHECK(8, info.stream_k == 0 && info.workspace_bytes == 0);
    req.wait_timeout_ns = -1;
    CHECK(9, conv_bn_silu_plan_request(32, 20, 20, 512, 512, 3, 3, 1, 1, 1, 1, &req, 152, &info) ==
                 CBS_ERR_INVALID_ARG);

    /* argument checks return before any launch */
    CHECK(10, conv_bn_silu_forward(NULL, NULL, NULL, NULL, NULL, 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, NULL) ==
                  CBS_ERR_INVALID_ARG);
    CHECK(11, conv_bn_act_forward(NULL, NULL, NULL, NULL, NULL, NULL, 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, 9,
                                  NULL) == CBS_ERR_INVALID_ARG);
    cbs_fold_layer layer;
    memset(&layer, 0, sizeof layer);
    layer.c_out = 0;
    layer.eps = 1e-3f;
    CHECK(12, conv_bn_silu_fold_batch(&layer, 1, NULL) == CBS_OK);
    CHECK(13, strcmp(conv_bn_silu_status_string(CBS_ERR_TIMEOUT), "kernel pipeline wait timed out") == 0);
    CHECK(14, conv_bn_silu_last_cuda_error() == 0);
    printf("c abi ok\n");
    return 0;
}

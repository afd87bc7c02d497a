/*
 * A plain C caller of libwo (no C++, no torch): the header compiles as C and
 * the host-only entry points work without a GPU.  Built and run by
 * tests/test_c_abi.py; prints one line per check and exits non-zero on the
 * first failure.
 */
#include <stdio.h>
#include <string.h>

#include "wo.h"

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #cond);    \
            return 1;                                                 \
        }                                                             \
        printf("ok %s\n", #cond);                                     \
    } while (0)

int main(void)
{
    /* sizes and status names */
    CHECK(wo_packed_bytes(4608, 3584, 8) == (size_t)4608 * 3584);
    CHECK(wo_packed_bytes(256, 512, 4) == (size_t)256 * 256);
    CHECK(wo_packed_bytes(100, 512, 8) == 0);
    CHECK(strcmp(wo_status_string(WO_ERR_WORKSPACE), "WO_ERR_WORKSPACE") == 0);

    /* the plan: decode on the weight-streaming kernels (4-bit: the persistent
       one), large m on tensor cores */
    wo_gemm_plan_t p;
    CHECK(wo_gemm_plan(1, 4608, 3584, -1, 8, WO_F16, &p) == WO_OK);
    CHECK(p.kernel == WO_KERNEL_STREAM && p.tile_m == 1 && p.ctas > 0);
    CHECK(p.workspace_bytes == wo_workspace_size(1, 4608, 3584, -1, 8));
    CHECK(wo_gemm_plan(1, 131072, 2048, 64, 4, WO_BF16, &p) == WO_OK);
    CHECK(p.kernel == WO_KERNEL_STREAM_PERSISTENT && p.tile_n == 256 && p.ctas > 0);
    CHECK(wo_gemm_plan(4096, 4096, 4096, -1, 8, WO_F16, &p) == WO_OK);
    CHECK(p.kernel == WO_KERNEL_TENSOR_CORE && p.tile_m == 256 && p.tile_n == 256);
    CHECK(wo_gemm_plan(4, 256, 512, 64, 8, WO_F16, &p) == WO_ERR_UNSUPPORTED);

    /* the act-order group sort: channels of group 1 then group 0 */
    int32_t g_idx[128], perm[128];
    for (int c = 0; c < 128; ++c)
        g_idx[c] = c < 64 ? 1 : 0;
    CHECK(wo_act_order_perm(g_idx, 128, 64, perm) == WO_OK);
    CHECK(perm[0] == 64 && perm[63] == 127 && perm[64] == 0 && perm[127] == 63);
    g_idx[0] = 0; /* groups of 65 and 63 channels */
    CHECK(wo_act_order_perm(g_idx, 128, 64, perm) == WO_ERR_UNSUPPORTED);

    /* argument checks return before any CUDA call */
    CHECK(wo_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 4, 256, 512, 64, 4, WO_BF16, NULL, 0,
                  NULL) == WO_ERR_INVALID_ARG);
    CHECK(wo_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 0, 256, 512, 64, 4, WO_BF16, NULL, 0,
                  NULL) == WO_OK);
    CHECK(wo_embed(NULL, 4, NULL, NULL, NULL, NULL, 100, 512, -1, 8, WO_F16, NULL) ==
          WO_ERR_INVALID_ARG);
    printf("all ok\n");
    return 0;
}

// wo_moe.cu -- grouped weight-only MoE FFN (routing, grouped fc1 with the
// gated activation, grouped fc2, routing-weighted combine).
#include "wo_internal.h"

extern "C" {

size_t wo_moe_workspace_size(int T, int hidden, int inter, int experts, int topk)
{
    (void)T; (void)hidden; (void)inter; (void)experts; (void)topk;
    return 0;
}

wo_status wo_moe_ffn(const void* A, const float* gating_logits, const uint8_t* fc1_packed,
                     const void* fc1_scales, const uint8_t* fc2_packed, const void* fc2_scales,
                     void* out, int T, int hidden, int inter, int experts, int topk,
                     int renormalize, wo_dtype act_dtype, void* workspace,
                     size_t workspace_bytes, void* stream)
{
    (void)A; (void)gating_logits; (void)fc1_packed; (void)fc1_scales; (void)fc2_packed;
    (void)fc2_scales; (void)out; (void)T; (void)hidden; (void)inter; (void)experts;
    (void)topk; (void)renormalize; (void)act_dtype; (void)workspace; (void)workspace_bytes;
    (void)stream;
    return WO_ERR_UNSUPPORTED;
}

}  // extern "C"

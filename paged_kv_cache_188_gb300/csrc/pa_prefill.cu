// pa_prefill.cu -- ragged causal prefill over the paged cache (tcgen05 path).
#include "pa_common.cuh"
#include "pa_internal.h"

extern "C" pa_status pa_paged_prefill_attn(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                           const void *v_buf, pa_kv_shape s, int layer_id,
                                           const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                           const int32_t *req_to_token, int req_rows, int max_ctx,
                                           const int32_t *req_pool_indices, float scale, void *workspace,
                                           size_t workspace_bytes, void *out, cudaStream_t st)
{
    return PA_ERR_UNSUPPORTED;
}

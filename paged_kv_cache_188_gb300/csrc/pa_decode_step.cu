// pa_decode_step.cu -- the fused decode step: RoPE + KV store + split-KV
// decode attention of one layer in one launch (the kernel is in
// pa_decode.cuh, instantiated here with FUSED = true).
#include "pa_decode.cuh"

using namespace pa;

extern "C" pa_status pa_decode_step(const void *q, const void *k_new, const void *v_new, int batch, int n_q_heads,
                                    const int32_t *positions, const float *cos_tab, const float *sin_tab,
                                    int max_pos, void *k_buf, void *v_buf, pa_kv_shape s, int layer_id,
                                    const int32_t *loc, const int32_t *req_to_token, int req_rows, int max_ctx,
                                    const int32_t *req_pool_indices, const int32_t *seq_lens, float scale,
                                    void *workspace, size_t workspace_bytes, int max_splits, void *out,
                                    cudaStream_t st)
{
    const StepInputs step{k_new, v_new, positions, loc, cos_tab, sin_tab, max_pos};
    return decode_call<MODE_FUSED>(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                       req_pool_indices, seq_lens, scale, workspace, workspace_bytes, max_splits, out, &step, st);
}


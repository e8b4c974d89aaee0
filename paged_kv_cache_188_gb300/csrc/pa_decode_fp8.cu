// pa_decode_fp8.cu -- the C-ABI entry point of packed split-KV decode
// attention over an e4m3 KV cache with one scale per (layer, kv head) for K
// and one for V (the kernel's fp8 mode, pa_decode.cuh).  Same planning,
// split merge, workspace and error reporting as pa_paged_decode_attn.
#include "pa_decode.cuh"

using namespace pa;

extern "C" pa_status pa_paged_decode_attn_fp8(const void *q, int batch, int n_q_heads, const void *k_buf,
                                              const void *v_buf, pa_kv_shape s, int layer_id,
                                              const int32_t *req_to_token, int req_rows, int max_ctx,
                                              const int32_t *req_pool_indices, const int32_t *seq_lens, float scale,
                                              const float *k_scale, const float *v_scale, void *workspace,
                                              size_t workspace_bytes, int max_splits, void *out, cudaStream_t st)
{
    pa_status rc = check_decode(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                                req_pool_indices, seq_lens, workspace, max_splits, out);
    if (rc != PA_OK) return rc;
    const DecodeWsLayout ws = decode_ws_layout(workspace_bytes, n_q_heads, s.n_kv_heads, s.head_dim, max_splits);
    if (ws.cap_batch < batch || ws.total > workspace_bytes) return PA_ERR_WORKSPACE;
    if (batch == 0) return PA_OK;
    if (!k_scale || !v_scale) return PA_ERR_NULL;
    if (!aligned4(k_scale) || !aligned4(v_scale)) return PA_ERR_ALIGN;
    unsigned char *w = static_cast<unsigned char *>(workspace);
    DecodeArgs a;
    if (!fill_decode_args(a, q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                          req_pool_indices, seq_lens, scale, max_splits, out, reinterpret_cast<int32_t *>(w), ws, w,
                          /*bf16_cache=*/false))
        return PA_ERR_CUDA;
    {
        // page tiles (16 consecutive slots) move as one TMA box of 16 rows per
        // K / V tile: D = 128 rows land 128-byte swizzled, as the ring expects;
        // D = 64 rows land plain
        const cuuint64_t dims[2] = {(cuuint64_t)s.n_kv_heads * s.head_dim, (cuuint64_t)s.n_layers * s.size};
        const cuuint64_t strides[1] = {(cuuint64_t)s.n_kv_heads * s.head_dim};
        const cuuint32_t box[2] = {(cuuint32_t)s.head_dim, kDecTile};
        if (!encode_tmap_u8(&a.tm_k, k_buf, 2, dims, strides, box, s.head_dim == 128) ||
            !encode_tmap_u8(&a.tm_v, v_buf, 2, dims, strides, box, s.head_dim == 128))
            return PA_ERR_CUDA;
    }
    const int64_t layer_bytes = (int64_t)layer_id * s.size * s.n_kv_heads * s.head_dim;   // one byte per element
    a.k8_layer = static_cast<const uint8_t *>(k_buf) + layer_bytes;
    a.v8_layer = static_cast<const uint8_t *>(v_buf) + layer_bytes;
    a.k_scale = k_scale + (int64_t)layer_id * s.n_kv_heads;
    a.v_scale = v_scale + (int64_t)layer_id * s.n_kv_heads;
    return dispatch_mode<MODE_FP8>(a, s.head_dim, st);
}

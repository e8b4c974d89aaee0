// pa_decode.cu -- the C-ABI entry points of packed split-KV decode attention
// (the kernel is in pa_decode.cuh): pa_paged_decode_attn with a caller
// workspace, and pa_paged_decode_attn_noalloc with a fixed scratch array.
#include "pa_decode.cuh"

namespace pa {
// Plain decode on prepared arguments, for the other translation units (the
// cascade's no-group path): its kernel instances are compiled here only.
pa_status decode_plain(const DecodeArgs &a, int head_dim, cudaStream_t st)
{
    return dispatch_mode<MODE_PLAIN>(a, head_dim, st);
}
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_paged_decode_attn(const void *q, int batch, int n_q_heads, const void *k_buf,
                                          const void *v_buf, pa_kv_shape s, int layer_id,
                                          const int32_t *req_to_token, int req_rows, int max_ctx,
                                          const int32_t *req_pool_indices, const int32_t *seq_lens, float scale,
                                          void *workspace, size_t workspace_bytes, int max_splits, void *out,
                                          cudaStream_t st)
{
    return decode_call<MODE_PLAIN>(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                       req_pool_indices, seq_lens, scale, workspace, workspace_bytes, max_splits, out, nullptr, st);
}

// ----------------------------------------------------------------------------
// Allocation-free decode: the same attention as pa_paged_decode_attn, with its
// scratch (split partials, merge tickets, error word) in a fixed device array
// that lives in this library instead of a caller-allocated workspace.
#include <mutex>

namespace pa {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;   // 16 MiB, held per device until exit
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device.  The host-side name is
// only a stand-in, so the address is looked up once per device, with that
// device current, and cached.
static void *noalloc_scratch_address()
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace pa

extern "C" pa_status pa_paged_decode_attn_noalloc(const void *q, int batch, int n_q_heads, const void *k_buf,
                                                  const void *v_buf, pa_kv_shape s, int layer_id,
                                                  const int32_t *req_to_token, int req_rows, int max_ctx,
                                                  const int32_t *req_pool_indices, const int32_t *seq_lens,
                                                  float scale, int max_splits, void *out, int32_t *error_word,
                                                  cudaStream_t st)
{
    using namespace pa;
    // every check runs before the first CUDA call: a call that fails has
    // enqueued nothing and written nothing
    const pa_status rc0 = check_decode_args(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows,
                                            max_ctx, req_pool_indices, seq_lens, max_splits, out);
    if (rc0 != PA_OK) return rc0;
    const DecodeWsLayout ws = decode_ws_layout(kNoAllocScratchBytes, n_q_heads, s.n_kv_heads, s.head_dim, max_splits);
    if (ws.cap_batch < batch || ws.total > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;   // beyond the fixed array
    if (error_word && !aligned4(error_word)) return PA_ERR_ALIGN;
    if (batch == 0) return PA_OK;
    void *scratch = noalloc_scratch_address();
    if (!scratch) return PA_ERR_CUDA;
    // the error word and the merge tickets must start at zero; the partials
    // are always written before they are read
    if (cudaMemsetAsync(scratch, 0, ws.ml_off, st) != cudaSuccess) return PA_ERR_CUDA;
    const pa_status rc = pa_paged_decode_attn(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows,
                                              max_ctx, req_pool_indices, seq_lens, scale, scratch,
                                              kNoAllocScratchBytes, max_splits, out, st);
    if (rc != PA_OK) return rc;
    if (error_word &&
        cudaMemcpyAsync(error_word, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

// pa_decode_cascade.cu -- cascade (shared-prefix) decode: requests grouped by
// a common cached prefix (radix reuse: their page-table rows point at the same
// prefix pages) read that prefix once per chunk of members instead of once per
// request.  Two launches of the kernel in pa_decode.cuh:
//   PREFIX  a virtual request per (group, chunk of up to 16 / G members): the
//           group's prefix tokens against the q rows of the chunk's members
//           (G_v = chunk * G rows per kv head), split-KV + merge as usual,
//           written as a normalised fp32 row and its log-sum-exp;
//   SUFFIX  every request over its tokens after its group's prefix (all of
//           them for requests in no group); the final write folds in the
//           request's prefix row by log-sum-exp.
// The prefix launch's first CTA also writes each request's start token and
// prefix row for the suffix launch, which plans only after waiting for it.
#include "pa_decode.cuh"

namespace pa {
pa_status decode_plain(const DecodeArgs &a, int head_dim, cudaStream_t st);   // pa_decode.cu
}

using namespace pa;

namespace pa {

// Workspace regions, fixed by the capacities alone so the merge tickets of
// both launches keep their places (and their zeros) from call to call.
struct CascadeLayout {
    int C, cpg, Bv, Gv, Hqv;
    size_t start_off, pre_off, preo_off, prelse_off, a_off, a_bytes, b_off, b_bytes, total;
};

static bool cascade_layout(const pa_cascade_caps &c, int n_q_heads, int n_kv_heads, int head_dim, CascadeLayout &L)
{
    if (c.max_batch < 0 || c.max_groups < 0 || c.max_group_size < 1 || c.max_splits < 1 ||
        c.max_splits > kDecMaxSplits || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0)
        return false;
    const int G = n_q_heads / n_kv_heads;
    if (G < 1 || G > 16) return false;
    L.C = 16 / G;
    L.cpg = (c.max_group_size + L.C - 1) / L.C;
    if ((int64_t)c.max_groups * L.cpg > kDecMaxBatch) return false;
    L.Bv = c.max_groups * L.cpg;
    L.Gv = L.C * G;
    L.Hqv = n_kv_heads * L.Gv;
    size_t off = kWorkspaceHeader;
    L.start_off = off;
    off += align_up((size_t)c.max_batch * 4, 256);
    L.pre_off = off;
    off += align_up((size_t)c.max_batch * 4, 256);
    L.preo_off = off;
    off += align_up((size_t)L.Bv * L.Hqv * head_dim * 4, 256);
    L.prelse_off = off;
    off += align_up((size_t)L.Bv * L.Hqv * 4, 256);
    L.a_off = off;
    L.a_bytes = pa_decode_workspace_bytes(L.Bv, L.Hqv, n_kv_heads, head_dim, c.max_splits);
    off += align_up(L.a_bytes, 256);
    L.b_off = off;
    L.b_bytes = pa_decode_workspace_bytes(c.max_batch, n_q_heads, n_kv_heads, head_dim, c.max_splits);
    off += L.b_bytes;
    L.total = off;
    return true;
}

}  // namespace pa

extern "C" size_t pa_cascade_workspace_bytes(pa_cascade_caps caps, int n_q_heads, int n_kv_heads, int head_dim)
{
    CascadeLayout L;
    return cascade_layout(caps, n_q_heads, n_kv_heads, head_dim, L) ? L.total : 0;
}

extern "C" pa_status pa_paged_decode_attn_cascade(const void *q, int batch, int n_q_heads, const void *k_buf,
                                                  const void *v_buf, pa_kv_shape s, int layer_id,
                                                  const int32_t *req_to_token, int req_rows, int max_ctx,
                                                  const int32_t *req_pool_indices, const int32_t *seq_lens,
                                                  const int32_t *group_indptr, const int32_t *group_reqs,
                                                  const int32_t *group_prefix, int n_groups, pa_cascade_caps caps,
                                                  float scale, void *workspace, size_t workspace_bytes, void *out,
                                                  cudaStream_t st)
{
    pa_status rc = check_decode(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                                req_pool_indices, seq_lens, workspace, caps.max_splits, out);
    if (rc != PA_OK) return rc;
    CascadeLayout L;
    if (!cascade_layout(caps, n_q_heads, s.n_kv_heads, s.head_dim, L)) return PA_ERR_SHAPE;
    if (batch > caps.max_batch || n_groups < 0 || n_groups > caps.max_groups) return PA_ERR_SHAPE;
    if (workspace_bytes < L.total) return PA_ERR_WORKSPACE;
    if (batch == 0) return PA_OK;
    if (n_groups > 0) {
        if (!group_indptr || !group_reqs || !group_prefix) return PA_ERR_NULL;
        if (!aligned4(group_indptr) || !aligned4(group_reqs) || !aligned4(group_prefix)) return PA_ERR_ALIGN;
    }
    unsigned char *w = static_cast<unsigned char *>(workspace);
    int32_t *err = reinterpret_cast<int32_t *>(w);
    const DecodeWsLayout wb = decode_ws_layout(L.b_bytes, n_q_heads, s.n_kv_heads, s.head_dim, caps.max_splits);
    if (n_groups == 0) {   // nothing shared: plain decode in the suffix region
        DecodeArgs b;
        if (!fill_decode_args(b, q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                              req_pool_indices, seq_lens, scale, caps.max_splits, out, err, wb, w + L.b_off))
            return PA_ERR_CUDA;
        return decode_plain(b, s.head_dim, st);
    }
    const DecodeWsLayout wa = decode_ws_layout(L.a_bytes, L.Hqv, s.n_kv_heads, s.head_dim, caps.max_splits);
    int32_t *req_start = reinterpret_cast<int32_t *>(w + L.start_off);
    int32_t *req_pre = reinterpret_cast<int32_t *>(w + L.pre_off);
    float *pre_o = reinterpret_cast<float *>(w + L.preo_off);
    float *pre_lse = reinterpret_cast<float *>(w + L.prelse_off);
    auto cascade_fields = [&](DecodeArgs &a) {
        a.grp_indptr = group_indptr;
        a.grp_reqs = group_reqs;
        a.grp_prefix = group_prefix;
        a.n_groups = n_groups;
        a.cpg = L.cpg;
        a.C = L.C;
        a.G_real = n_q_heads / s.n_kv_heads;
        a.Hq_real = n_q_heads;
        a.B_real = batch;
        a.req_start = req_start;
        a.req_pre = req_pre;
        a.pre_o = pre_o;
        a.pre_lse = pre_lse;
    };
    // launch 1: the groups' prefixes, one virtual request per (group, chunk)
    DecodeArgs pa;
    if (!fill_decode_args(pa, q, n_groups * L.cpg, L.Hqv, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                          req_pool_indices, seq_lens, scale, caps.max_splits, nullptr, err, wa, w + L.a_off))
        return PA_ERR_CUDA;
    cascade_fields(pa);
    rc = s.head_dim == 128 ? dispatch_decode<128, 2, MODE_PREFIX>(pa, st) : dispatch_decode<64, 2, MODE_PREFIX>(pa, st);
    if (rc != PA_OK) return rc;
    // launch 2: every request after its prefix, folding in the prefix rows
    DecodeArgs sb;
    if (!fill_decode_args(sb, q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                          req_pool_indices, seq_lens, scale, caps.max_splits, out, err, wb, w + L.b_off))
        return PA_ERR_CUDA;
    cascade_fields(sb);
    return dispatch_mode<MODE_SUFFIX>(sb, s.head_dim, st);
}

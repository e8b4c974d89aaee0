// pa_store_rope.cu -- the two bandwidth-bound elementwise steps of the path:
//   pa_kv_store    : new tokens' K/V written at buffer[layer_id, loc]
//                    (AstrAI commit 398e8a3, tests/inference/test_cache.py:
//                    single advanced indexing buffer[layer_id, loc], int32 loc)
//   pa_rope_packed : rotary embedding on packed [T, H, D] q and k from a cos/sin
//                    table (commit 398e8a3: rotary extended to packed 3-D
//                    inputs; commit e58a728, docs/developer/architecture.md:
//                    a real cos/sin freqs_cis table)
//   pa_kv_store_fp8: the same store into an e4m3 cache, each row divided by
//                    its (layer, kv head) scale and rounded to e4m3
// All move 16-byte vectors: one thread per 16 bytes of a row, rows contiguous
// in memory, so every warp touches whole 128-byte lines.  Launched behind
// another kernel (launch overlap on), each thread waits for it before reading
// data; in early-metadata mode its first loc / position entry is read first.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// One thread copies one 16-byte chunk of one token's K row and the same chunk
// of its V row.  row_chunks = Hkv * D / 8 chunks per token.
__global__ void __launch_bounds__(256) kv_store_kernel(uint4 *__restrict__ k_layer, uint4 *__restrict__ v_layer,
                                                       const uint4 *__restrict__ k_new,
                                                       const uint4 *__restrict__ v_new,
                                                       const int32_t *__restrict__ loc, int64_t n_chunks,
                                                       int row_chunks, int size, int32_t *err, int early_meta)
{
    // early-metadata mode: this thread's first cache location is read before
    // waiting for the preceding kernel, everything else after
    const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int32_t slot0 = (early_meta && i0 < n_chunks) ? __ldg(loc + i0 / row_chunks) : 0;
    pdl_wait();
    pdl_launch_dependents();
    const bool small = n_chunks < (1LL << 31);   // 32-bit index arithmetic suffices
    for (int64_t i = i0; i < n_chunks; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t t;
        int c;
        if (small) {
            const uint32_t t32 = (uint32_t)i / (uint32_t)row_chunks;
            c = (int)((uint32_t)i - t32 * (uint32_t)row_chunks);
            t = t32;
        } else {
            t = i / row_chunks;
            c = (int)(i - t * row_chunks);
        }
        const int32_t slot = (early_meta && i == i0) ? slot0 : __ldg(loc + t);
        if (slot < 0 || slot >= size) {
            if (c == 0) set_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const uint4 kv = __ldcs(k_new + i);
        const uint4 vv = __ldcs(v_new + i);
        const int64_t dst = (int64_t)slot * row_chunks + c;
        k_layer[dst] = kv;
        v_layer[dst] = vv;
    }
}

// One thread quantises 16 consecutive elements (one 16-byte e4m3 chunk) of one
// token's K row and the same elements of its V row.  row_chunks = Hkv * D / 16
// chunks per token, head_chunks = D / 16 per head; scales are the layer's
// [Hkv] K and V scales.
__global__ void __launch_bounds__(256) kv_store_fp8_kernel(uint4 *__restrict__ k_layer, uint4 *__restrict__ v_layer,
                                                           const uint4 *__restrict__ k_new,
                                                           const uint4 *__restrict__ v_new,
                                                           const int32_t *__restrict__ loc,
                                                           const float *__restrict__ k_scale,
                                                           const float *__restrict__ v_scale, int64_t n_chunks,
                                                           int row_chunks, int head_chunks, int size, int32_t *err,
                                                           int early_meta)
{
    const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int32_t slot0 = (early_meta && i0 < n_chunks) ? __ldg(loc + i0 / row_chunks) : 0;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t i = i0; i < n_chunks; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / row_chunks;
        const int c = (int)(i - t * row_chunks);
        const int32_t slot = (early_meta && i == i0) ? slot0 : __ldg(loc + t);
        if (slot < 0 || slot >= size) {
            if (c == 0) set_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const int h = c / head_chunks;
        const uint4 k0 = __ldcs(k_new + 2 * i), k1 = __ldcs(k_new + 2 * i + 1);
        const uint4 v0 = __ldcs(v_new + 2 * i), v1 = __ldcs(v_new + 2 * i + 1);
        const float ks = __ldg(k_scale + h), vs = __ldg(v_scale + h);
        float kx[16], vx[16];
        const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            kx[2 * j] = __uint_as_float(kw[j] << 16);
            kx[2 * j + 1] = __uint_as_float(kw[j] & 0xFFFF0000u);
            vx[2 * j] = __uint_as_float(vw[j] << 16);
            vx[2 * j + 1] = __uint_as_float(vw[j] & 0xFFFF0000u);
        }
        const int64_t dst = (int64_t)slot * row_chunks + c;
        k_layer[dst] = quant_e4m3x16(kx, ks);
        v_layer[dst] = quant_e4m3x16(vx, vs);
    }
}

// One thread rotates 8 consecutive elements (4 interleaved pairs) of one head
// vector.  Heads [0, Hq) index q, heads [Hq, Hq + Hkv) index k.
__global__ void __launch_bounds__(256) rope_kernel(uint4 *__restrict__ q, uint4 *__restrict__ k, int Hq, int Hkv,
                                                   int head_chunks, const int32_t *__restrict__ positions,
                                                   int64_t n_chunks, const float4 *__restrict__ cos_tab,
                                                   const float4 *__restrict__ sin_tab, int max_pos,
                                                   int32_t *err, int early_meta)
{
    const int heads = Hq + Hkv;
    // early-metadata mode: this thread's first position is read before waiting
    // for the preceding kernel, everything else after
    const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int32_t p0 = (early_meta && i0 < n_chunks) ? __ldg(positions + i0 / head_chunks / heads) : 0;
    pdl_wait();
    pdl_launch_dependents();
    // 32-bit index arithmetic when the chunk count allows it (64-bit
    // divisions had cost this kernel 7 % of its throughput)
    const bool small = n_chunks < (1LL << 31);
    for (int64_t i = i0; i < n_chunks; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t t;
        int c, h;
        if (small) {
            const uint32_t i32 = (uint32_t)i, th = i32 / (uint32_t)head_chunks;   // token * heads + head
            c = (int)(i32 - th * (uint32_t)head_chunks);
            const uint32_t t32 = th / (uint32_t)heads;
            h = (int)(th - t32 * (uint32_t)heads);
            t = t32;
        } else {
            const int64_t th = i / head_chunks;
            c = (int)(i - th * head_chunks);
            t = th / heads;
            h = (int)(th - t * heads);
        }
        const int32_t p = (early_meta && i == i0) ? p0 : __ldg(positions + t);
        if (p < 0 || p >= max_pos) {
            if (h == 0 && c == 0) set_error(err, PA_DEVERR_POS);
            continue;
        }
        uint4 *ptr = h < Hq ? q + (t * Hq + h) * head_chunks + c : k + (t * Hkv + (h - Hq)) * head_chunks + c;
        // pairs 4c .. 4c+3 of this head: table row p, columns 4c .. 4c+3
        const float4 cs = __ldg(cos_tab + (int64_t)p * head_chunks + c);
        const float4 sn = __ldg(sin_tab + (int64_t)p * head_chunks + c);
        const uint4 x = *ptr;
        *ptr = make_uint4(rope_pair_bf16(x.x, cs.x, sn.x), rope_pair_bf16(x.y, cs.y, sn.y),
                          rope_pair_bf16(x.z, cs.z, sn.z), rope_pair_bf16(x.w, cs.w, sn.w));
    }
}

static int grid_for(int64_t n_threads, int block)
{
    int64_t g = (n_threads + block - 1) / block;
    const int cap = num_sms() * 16;
    return (int)(g < cap ? (g > 0 ? g : 1) : cap);
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_kv_store(void *k_buf, void *v_buf, pa_kv_shape s, int layer_id, const void *k_new,
                                 const void *v_new, const int32_t *loc, int n_tokens, int32_t *error_word,
                                 cudaStream_t st)
{
    if (n_tokens < 0 || s.n_layers <= 0 || s.size <= 0 || s.n_kv_heads <= 0 || s.head_dim <= 0)
        return PA_ERR_SHAPE;
    if (layer_id < 0 || layer_id >= s.n_layers) return PA_ERR_SHAPE;
    if (s.head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return PA_OK;
    if (!k_buf || !v_buf || !k_new || !v_new || !loc) return PA_ERR_NULL;
    if (!aligned16(k_buf) || !aligned16(v_buf) || !aligned16(k_new) || !aligned16(v_new) || !aligned4(loc))
        return PA_ERR_ALIGN;
    if (error_word && !aligned4(error_word)) return PA_ERR_ALIGN;
    const int row_chunks = s.n_kv_heads * s.head_dim / 8;
    const int64_t layer_off = (int64_t)layer_id * s.size * row_chunks;
    const int64_t n_chunks = (int64_t)n_tokens * row_chunks;
    if (launch_kernel(kv_store_kernel, dim3(grid_for(n_chunks, 256)), dim3(256), 0, st,
                      static_cast<uint4 *>(k_buf) + layer_off, static_cast<uint4 *>(v_buf) + layer_off,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), loc, n_chunks,
                      row_chunks, s.size, error_word,
                      (int)early_metadata()) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_kv_store_fp8(void *k_buf, void *v_buf, pa_kv_shape s, int layer_id, const void *k_new,
                                     const void *v_new, const int32_t *loc, int n_tokens, const float *k_scale,
                                     const float *v_scale, int32_t *error_word, cudaStream_t st)
{
    if (n_tokens < 0 || s.n_layers <= 0 || s.size <= 0 || s.n_kv_heads <= 0 || s.head_dim <= 0)
        return PA_ERR_SHAPE;
    if (layer_id < 0 || layer_id >= s.n_layers) return PA_ERR_SHAPE;
    if (s.head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return PA_OK;
    if (!k_buf || !v_buf || !k_new || !v_new || !loc || !k_scale || !v_scale) return PA_ERR_NULL;
    if (!aligned16(k_buf) || !aligned16(v_buf) || !aligned16(k_new) || !aligned16(v_new) || !aligned4(loc) ||
        !aligned4(k_scale) || !aligned4(v_scale))
        return PA_ERR_ALIGN;
    if (error_word && !aligned4(error_word)) return PA_ERR_ALIGN;
    const int row_chunks = s.n_kv_heads * s.head_dim / 16;
    const int64_t layer_off = (int64_t)layer_id * s.size * row_chunks;
    const int64_t n_chunks = (int64_t)n_tokens * row_chunks;
    const int64_t scale_off = (int64_t)layer_id * s.n_kv_heads;
    if (launch_kernel(kv_store_fp8_kernel, dim3(grid_for(n_chunks, 256)), dim3(256), 0, st,
                      static_cast<uint4 *>(k_buf) + layer_off, static_cast<uint4 *>(v_buf) + layer_off,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), loc, k_scale + scale_off,
                      v_scale + scale_off, n_chunks, row_chunks, s.head_dim / 16, s.size, error_word,
                      (int)early_metadata()) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_rope_packed(void *q, int n_q_heads, void *k, int n_kv_heads, int head_dim,
                                    const int32_t *positions, int n_tokens, const float *cos_tab,
                                    const float *sin_tab, int max_pos, int32_t *error_word, cudaStream_t st)
{
    if (n_tokens < 0 || n_q_heads < 0 || n_kv_heads < 0 || head_dim <= 0 || max_pos <= 0) return PA_ERR_SHAPE;
    if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (n_tokens == 0 || n_q_heads + n_kv_heads == 0) return PA_OK;
    if ((n_q_heads > 0 && !q) || (n_kv_heads > 0 && !k) || !positions || !cos_tab || !sin_tab) return PA_ERR_NULL;
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || !aligned4(positions) || !aligned16(cos_tab) ||
        !aligned16(sin_tab))
        return PA_ERR_ALIGN;
    if (error_word && !aligned4(error_word)) return PA_ERR_ALIGN;
    const int head_chunks = head_dim / 8;
    const int64_t n_chunks = (int64_t)n_tokens * (n_q_heads + n_kv_heads) * head_chunks;
    if (launch_kernel(rope_kernel, dim3(grid_for(n_chunks, 256)), dim3(256), 0, st, static_cast<uint4 *>(q),
                      static_cast<uint4 *>(k), n_q_heads, n_kv_heads, head_chunks, positions, n_chunks,
                      reinterpret_cast<const float4 *>(cos_tab), reinterpret_cast<const float4 *>(sin_tab), max_pos,
                      error_word, (int)early_metadata()) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

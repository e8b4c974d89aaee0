/*
 * oracle.c -- plain, slow, single-threaded float64 statement of what the
 * paged-KV attention hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * measured against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the product path never calls it, and it shares
 * no code, header, table or helper with the CUDA sources.
 *
 * Source of the definitions: the AstrAI commit pages on packed 3-D inference
 * with a paged KV cache --
 *   "398e8a3 / tests/inference/test_cache.py": packed 3-D q/k/v for inference,
 *     rotary embedding extended to packed 3-D inputs, int32 page-table /
 *     request-row / cache-location indices, KV written at buffer[layer_id, loc]
 *     of per-layer [n_layers, size, n_kv_heads, head_dim] buffers, a
 *     ReqToTokenPool, split-KV decode with workspace-owned partials;
 *   "e58a728 / docs/developer/architecture.md": rotary from a cos/sin
 *     freqs_cis table, packed shared-prefix prefill addressed by cumulative
 *     query lengths (qo_indptr), paged prefill (attn_paged_prefill), decode
 *     gathering flat K/V through req_to_token.
 * The pages carry no formulas.  Every function below is the textbook
 * definition of the named operation written out; the readings taken where the
 * pages are silent are listed at each function.
 *
 * bf16 values travel as their 16-bit patterns (uint16_t).  All arithmetic is
 * IEEE double; build without -ffast-math and with -ffp-contract=off so x86
 * and Arm give identical results.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_SHAPE 2
#define ORA_ERR_INDEX 7
#define ORA_ERR_NOMEM 8

/* ---------------------------------------------------------------- bf16 */

/* Exact widening of a bfloat16 bit pattern (the upper half of an IEEE
 * binary32) to double. */
double ora_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bfloat16 (8 significant bits, binary32
 * exponent range, subnormal spacing 2^-133), ties to even; one rounding
 * straight from double.  NaN -> canonical quiet NaN 0x7FC0. */
uint16_t ora_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;         /* spacing of 8-significant-bit numbers near a */
    if (qexp < -133)
        qexp = -133;          /* subnormal range has fixed spacing */
    double r = nearbyint(ldexp(a, -qexp)); /* default mode: nearest, ties even */
    double v = ldexp(r, qexp);
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)v;       /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void ora_f64_to_bf16_array(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_f64_to_bf16(x[i]);
}

/* ---------------------------------------------------------------- RoPE */

/* Rotary embedding of packed [T, H, D] vectors (page "398e8a3": rotary
 * extended to packed 3-D inputs; page "e58a728": the table is a real cos/sin
 * pair, not a complex buffer).
 *
 * Reading (pair convention): element pairs are (2i, 2i+1), the interleaved
 * form that a complex freqs_cis table multiplies.  For token t at position
 * p = pos[t], head h, pair i < D/2, with c = cos_tab[p, i], s = sin_tab[p, i]:
 *     y[2i]   = x[2i] * c - x[2i+1] * s
 *     y[2i+1] = x[2i] * s + x[2i+1] * c
 * computed in double from the exact fp32 table values.  y_f64 (optional)
 * receives the unrounded results, y_bf16 (optional) their bf16 rounding.
 * Returns ORA_ERR_INDEX if a position is outside [0, max_pos). */
int ora_rope(const uint16_t *x, int64_t T, int H, int D, const int32_t *pos,
             const float *cos_tab, const float *sin_tab, int max_pos,
             uint16_t *y_bf16, double *y_f64)
{
    if (D <= 0 || D % 2 != 0 || H <= 0 || T < 0)
        return ORA_ERR_SHAPE;
    const int half = D / 2;
    for (int64_t t = 0; t < T; ++t) {
        int32_t p = pos[t];
        if (p < 0 || p >= max_pos)
            return ORA_ERR_INDEX;
        for (int h = 0; h < H; ++h) {
            const int64_t base = (t * H + h) * (int64_t)D;
            for (int i = 0; i < half; ++i) {
                double c = (double)cos_tab[(int64_t)p * half + i];
                double s = (double)sin_tab[(int64_t)p * half + i];
                double x0 = ora_bf16_to_f64(x[base + 2 * i]);
                double x1 = ora_bf16_to_f64(x[base + 2 * i + 1]);
                double y0 = x0 * c - x1 * s;
                double y1 = x0 * s + x1 * c;
                if (y_f64) {
                    y_f64[base + 2 * i] = y0;
                    y_f64[base + 2 * i + 1] = y1;
                }
                if (y_bf16) {
                    y_bf16[base + 2 * i] = ora_f64_to_bf16(y0);
                    y_bf16[base + 2 * i + 1] = ora_f64_to_bf16(y1);
                }
            }
        }
    }
    return ORA_OK;
}

/* ------------------------------------------------------------ KV store */

/* Store the new tokens' K and V at their cache locations (page "398e8a3":
 * buffer[layer_id, loc] single advanced indexing into per-layer
 * [n_layers, size, n_kv_heads, head_dim] buffers; int32 cache locations):
 *     k_buf[layer, loc[t], h, :] = k_new[t, h, :]   (same for v)
 * A pure copy of bit patterns.  Reading: duplicate locations within one call
 * are not meaningful; the copy runs in token order so the last one wins.
 * All locations are checked before anything is written. */
int ora_kv_store(uint16_t *k_buf, uint16_t *v_buf, int n_layers, int64_t size,
                 int Hkv, int D, int layer, const uint16_t *k_new,
                 const uint16_t *v_new, const int32_t *loc, int64_t T)
{
    if (layer < 0 || layer >= n_layers || Hkv <= 0 || D <= 0 || T < 0)
        return ORA_ERR_SHAPE;
    for (int64_t t = 0; t < T; ++t)
        if (loc[t] < 0 || (int64_t)loc[t] >= size)
            return ORA_ERR_INDEX;
    const int64_t row = (int64_t)Hkv * D;
    for (int64_t t = 0; t < T; ++t) {
        int64_t dst = ((int64_t)layer * size + loc[t]) * row;
        for (int64_t j = 0; j < row; ++j) {
            k_buf[dst + j] = k_new[t * row + j];
            v_buf[dst + j] = v_new[t * row + j];
        }
    }
    return ORA_OK;
}

/* ----------------------------------------------------------- attention */

/* Softmax attention of one query vector over n keys given by their cache
 * slots:  s_j = scale * <q, K[slot_j]>,  out = sum_j softmax(s)_j V[slot_j].
 * The maximum is subtracted before exponentiation (exact in real arithmetic).
 * n == 0 gives a zero vector (reading: the pages do not define an empty
 * softmax; zeros keep the output finite).  scores must hold n doubles. */
static void attend_one(const uint16_t *qv, const uint16_t *k_head0,
                       const uint16_t *v_head0, int64_t slot_stride,
                       const int32_t *slots, int64_t n, int D, double scale,
                       double *scores, double *out)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return;
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        const uint16_t *kr = k_head0 + (int64_t)slots[j] * slot_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += ora_bf16_to_f64(qv[d]) * ora_bf16_to_f64(kr[d]);
        scores[j] = scale * dot;
        if (scores[j] > m)
            m = scores[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        scores[j] = exp(scores[j] - m);
        denom += scores[j];
    }
    for (int64_t j = 0; j < n; ++j) {
        const uint16_t *vr = v_head0 + (int64_t)slots[j] * slot_stride;
        double w = scores[j] / denom;
        for (int d = 0; d < D; ++d)
            out[d] += w * ora_bf16_to_f64(vr[d]);
    }
}

/* Packed decode attention over the paged cache (page "398e8a3": per-request
 * rows of a ReqToTokenPool, int32 indices, GQA split-KV decode; page
 * "e58a728": decode gathers flat K/V via req_to_token).
 *
 * For request b with n = seq_lens[b] and row = req_pool_indices[b], its token
 * j < n lives at cache slot req_to_token[row, j].  Query head hq reads kv
 * head hq / (Hq / Hkv) (reading: contiguous GQA grouping).  The output for
 * (b, hq) is the softmax attention of q[b, hq, :] over those n keys.
 * Reading: seq_lens counts the current token, whose K/V are already stored;
 * entries req_to_token[row, j >= n] are never read.
 *
 * If sel_b is NULL every (b, hq) pair is computed into out[B, Hq, D];
 * otherwise only the n_sel pairs (sel_b[i], sel_h[i]) into out[n_sel, D].
 * Slots and rows are range-checked first (ORA_ERR_INDEX). */
int ora_decode(const uint16_t *q, int B, int Hq, const uint16_t *k_buf,
               const uint16_t *v_buf, int n_layers, int64_t size, int Hkv,
               int D, int layer, const int32_t *req_to_token, int req_rows,
               int max_ctx, const int32_t *req_pool_indices,
               const int32_t *seq_lens, double scale, const int32_t *sel_b,
               const int32_t *sel_h, int64_t n_sel, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || layer < 0 || layer >= n_layers || D <= 0)
        return ORA_ERR_SHAPE;
    const int G = Hq / Hkv;
    const int64_t npairs = sel_b ? n_sel : (int64_t)B * Hq;
    for (int64_t i = 0; i < npairs; ++i) {
        int b = sel_b ? sel_b[i] : (int)(i / Hq);
        int hq = sel_b ? sel_h[i] : (int)(i % Hq);
        if (b < 0 || b >= B || hq < 0 || hq >= Hq)
            return ORA_ERR_SHAPE;
        int row = req_pool_indices[b];
        int n = seq_lens[b];
        if (row < 0 || row >= req_rows || n < 0 || n > max_ctx)
            return ORA_ERR_INDEX;
        for (int j = 0; j < n; ++j) {
            int32_t s = req_to_token[(int64_t)row * max_ctx + j];
            if (s < 0 || (int64_t)s >= size)
                return ORA_ERR_INDEX;
        }
    }
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!scores)
        return ORA_ERR_NOMEM;
    const int64_t slot_stride = (int64_t)Hkv * D;
    for (int64_t i = 0; i < npairs; ++i) {
        int b = sel_b ? sel_b[i] : (int)(i / Hq);
        int hq = sel_b ? sel_h[i] : (int)(i % Hq);
        int h = hq / G;
        int row = req_pool_indices[b];
        const uint16_t *k0 = k_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        const uint16_t *v0 = v_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        attend_one(q + ((int64_t)b * Hq + hq) * D, k0, v0, slot_stride,
                   req_to_token + (int64_t)row * max_ctx, seq_lens[b], D, scale,
                   scores, out + i * D);
    }
    free(scores);
    return ORA_OK;
}

/* Ragged causal prefill over packed tokens (page "e58a728": prompts packed
 * into one forward, per-request rows located by cumulative query lengths,
 * attn_paged_prefill; page "398e8a3": request mappings rebuilt for cached
 * prefix pages).
 *
 * Request r owns packed query rows qo_indptr[r] .. qo_indptr[r+1]-1 (n_r of
 * them) and L_r = kv_indptr[r+1] - kv_indptr[r] cached tokens, of which the
 * first p_r = L_r - n_r are an already-cached prefix (reading: kv_indptr
 * counts tokens, the new tokens are the last n_r of the request).  Query i of
 * request r sits at position p_r + i and attends to positions 0 .. p_r + i
 * (causal mask aligned to the end), read through
 * req_to_token[req_pool_indices[r], position].
 *
 * If sel_t is NULL every (t, hq) is computed into out[T, Hq, D]; otherwise the
 * n_sel pairs (sel_t[i], sel_h[i]) into out[n_sel, D].  Checks the indptr
 * arrays and every slot read first. */
int ora_prefill(const uint16_t *q, int64_t T, int Hq, const uint16_t *k_buf,
                const uint16_t *v_buf, int n_layers, int64_t size, int Hkv,
                int D, int layer, const int32_t *qo_indptr,
                const int32_t *kv_indptr, int R, const int32_t *req_to_token,
                int req_rows, int max_ctx, const int32_t *req_pool_indices,
                double scale, const int32_t *sel_t, const int32_t *sel_h,
                int64_t n_sel, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || layer < 0 || layer >= n_layers || D <= 0 || R < 0)
        return ORA_ERR_SHAPE;
    if (qo_indptr[0] != 0 || qo_indptr[R] != T || kv_indptr[0] != 0)
        return ORA_ERR_SHAPE;
    for (int r = 0; r < R; ++r) {
        int n_r = qo_indptr[r + 1] - qo_indptr[r];
        int L_r = kv_indptr[r + 1] - kv_indptr[r];
        if (n_r < 0 || L_r < n_r || L_r > max_ctx)
            return ORA_ERR_SHAPE;
        int row = req_pool_indices[r];
        if (row < 0 || row >= req_rows)
            return ORA_ERR_INDEX;
        for (int j = 0; j < L_r; ++j) {
            int32_t s = req_to_token[(int64_t)row * max_ctx + j];
            if (s < 0 || (int64_t)s >= size)
                return ORA_ERR_INDEX;
        }
    }
    const int G = Hq / Hkv;
    const int64_t slot_stride = (int64_t)Hkv * D;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!scores)
        return ORA_ERR_NOMEM;
    const int64_t npairs = sel_t ? n_sel : T * Hq;
    for (int64_t i = 0; i < npairs; ++i) {
        int64_t t = sel_t ? sel_t[i] : i / Hq;
        int hq = sel_t ? sel_h[i] : (int)(i % Hq);
        if (t < 0 || t >= T || hq < 0 || hq >= Hq) {
            free(scores);
            return ORA_ERR_SHAPE;
        }
        int r = 0;
        while (!(qo_indptr[r] <= t && t < qo_indptr[r + 1]))
            ++r;
        int n_r = qo_indptr[r + 1] - qo_indptr[r];
        int L_r = kv_indptr[r + 1] - kv_indptr[r];
        int p_r = L_r - n_r;
        int64_t qi = t - qo_indptr[r];
        int h = hq / G;
        int row = req_pool_indices[r];
        const uint16_t *k0 = k_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        const uint16_t *v0 = v_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        attend_one(q + (t * Hq + hq) * D, k0, v0, slot_stride,
                   req_to_token + (int64_t)row * max_ctx, p_r + qi + 1, D, scale,
                   scores, out + i * D);
    }
    free(scores);
    return ORA_OK;
}

/* ------------------------------------------------------ fp8 (e4m3) cache */

/* fp8 e4m3 KV cache with per-head scales.  The only mention on the pages is
 * page "e58a728 / docs/developer/architecture.md", whose change list names an
 * fp8 test among the CUDA kernel sources; everything below is a reading.
 * Format: the OCP 8-bit float E4M3 -- 1 sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448.
 * Reading (the pages give no scheme): one fp32 scale per (layer, kv head) for
 * K and one for V, supplied by the caller; stored byte =
 * e4m3(fp32(x) / scale) with the division in fp32 (IEEE, nearest) and the
 * conversion rounding to nearest, ties to even, finite values beyond 448
 * saturating to +-448; the value read back is e4m3_value(byte) * scale. */

/* Exact value of an e4m3 byte (NaN for the two NaN codes). */
double ora_e4m3_to_f64(uint8_t b)
{
    int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = e == 0 ? ldexp((double)m, -9)             /* subnormal: m/8 * 2^-6 */
                      : ldexp(8.0 + m, e - 10);          /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest e4m3 byte to a float, ties to even, saturating finite overflow
 * (and infinities) to +-448; NaN -> 0x7F. */
uint8_t ora_f32_to_e4m3(float xf)
{
    double x = (double)xf;
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);             /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    int qexp = e - 4;         /* spacing of 4-significant-bit numbers near a */
    if (qexp < -9)
        qexp = -9;            /* subnormal range: fixed spacing 2^-9 */
    double r = nearbyint(ldexp(a, -qexp)); /* exact scaling, then nearest-even */
    double v = ldexp(r, qexp);             /* <= 448 since a < 448 */
    if (v == 0.0)
        return sign;
    int ev;
    frexp(v, &ev);
    int E = ev - 1 + 7;       /* biased exponent of v = 2^(ev-1) * (1 + m/8) */
    if (E <= 0)               /* subnormal: v = m * 2^-9 */
        return (uint8_t)(sign | (uint8_t)ldexp(v, 9));
    int m = (int)(ldexp(v, -(ev - 1)) * 8.0) - 8;
    return (uint8_t)(sign | (E << 3) | m);
}

void ora_f32_to_e4m3_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_f32_to_e4m3(x[i]);
}

/* Quantising KV store: k8_buf[layer, loc[t], h, :] = e4m3(k_new[t, h, :] /
 * k_scale[layer, h]), the same for V; buffers [n_layers, size, Hkv, D] bytes,
 * scales [n_layers, Hkv] fp32.  Locations are checked before anything is
 * written. */
int ora_kv_store_fp8(uint8_t *k_buf, uint8_t *v_buf, int n_layers, int64_t size,
                     int Hkv, int D, int layer, const uint16_t *k_new,
                     const uint16_t *v_new, const int32_t *loc, int64_t T,
                     const float *k_scale, const float *v_scale)
{
    if (layer < 0 || layer >= n_layers || Hkv <= 0 || D <= 0 || T < 0)
        return ORA_ERR_SHAPE;
    for (int64_t t = 0; t < T; ++t)
        if (loc[t] < 0 || (int64_t)loc[t] >= size)
            return ORA_ERR_INDEX;
    const int64_t row = (int64_t)Hkv * D;
    for (int64_t t = 0; t < T; ++t) {
        int64_t dst = ((int64_t)layer * size + loc[t]) * row;
        for (int h = 0; h < Hkv; ++h) {
            float ks = k_scale[(int64_t)layer * Hkv + h], vs = v_scale[(int64_t)layer * Hkv + h];
            for (int d = 0; d < D; ++d) {
                int64_t j = (int64_t)h * D + d;
                float kx = (float)ora_bf16_to_f64(k_new[t * row + j]);
                float vx = (float)ora_bf16_to_f64(v_new[t * row + j]);
                k_buf[dst + j] = ora_f32_to_e4m3(kx / ks);
                v_buf[dst + j] = ora_f32_to_e4m3(vx / vs);
            }
        }
    }
    return ORA_OK;
}

/* Packed decode attention over an fp8 cache: as ora_decode, with key j of kv
 * head h read as e4m3_value(K8[slot_j, h, :]) * k_scale[layer, h] and value
 * rows likewise with v_scale.  Same output, selection and checks. */
int ora_decode_fp8(const uint16_t *q, int B, int Hq, const uint8_t *k_buf,
                   const uint8_t *v_buf, int n_layers, int64_t size, int Hkv,
                   int D, int layer, const int32_t *req_to_token, int req_rows,
                   int max_ctx, const int32_t *req_pool_indices,
                   const int32_t *seq_lens, double scale, const float *k_scale,
                   const float *v_scale, const int32_t *sel_b,
                   const int32_t *sel_h, int64_t n_sel, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || layer < 0 || layer >= n_layers || D <= 0)
        return ORA_ERR_SHAPE;
    const int G = Hq / Hkv;
    const int64_t npairs = sel_b ? n_sel : (int64_t)B * Hq;
    for (int64_t i = 0; i < npairs; ++i) {
        int b = sel_b ? sel_b[i] : (int)(i / Hq);
        int hq = sel_b ? sel_h[i] : (int)(i % Hq);
        if (b < 0 || b >= B || hq < 0 || hq >= Hq)
            return ORA_ERR_SHAPE;
        int row = req_pool_indices[b];
        int n = seq_lens[b];
        if (row < 0 || row >= req_rows || n < 0 || n > max_ctx)
            return ORA_ERR_INDEX;
        for (int j = 0; j < n; ++j) {
            int32_t s = req_to_token[(int64_t)row * max_ctx + j];
            if (s < 0 || (int64_t)s >= size)
                return ORA_ERR_INDEX;
        }
    }
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!scores)
        return ORA_ERR_NOMEM;
    const int64_t slot_stride = (int64_t)Hkv * D;
    for (int64_t i = 0; i < npairs; ++i) {
        int b = sel_b ? sel_b[i] : (int)(i / Hq);
        int hq = sel_b ? sel_h[i] : (int)(i % Hq);
        int h = hq / G;
        int n = seq_lens[b];
        const int32_t *slots = req_to_token + (int64_t)req_pool_indices[b] * max_ctx;
        const uint16_t *qv = q + ((int64_t)b * Hq + hq) * D;
        const uint8_t *k0 = k_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        const uint8_t *v0 = v_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        const double ks = (double)k_scale[(int64_t)layer * Hkv + h];
        const double vs = (double)v_scale[(int64_t)layer * Hkv + h];
        double *o = out + i * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (n <= 0)
            continue;
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            const uint8_t *kr = k0 + (int64_t)slots[j] * slot_stride;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += ora_bf16_to_f64(qv[d]) * (ora_e4m3_to_f64(kr[d]) * ks);
            scores[j] = scale * dot;
            if (scores[j] > m)
                m = scores[j];
        }
        double denom = 0.0;
        for (int j = 0; j < n; ++j) {
            scores[j] = exp(scores[j] - m);
            denom += scores[j];
        }
        for (int j = 0; j < n; ++j) {
            const uint8_t *vr = v0 + (int64_t)slots[j] * slot_stride;
            double w = scores[j] / denom;
            for (int d = 0; d < D; ++d)
                o[d] += w * (ora_e4m3_to_f64(vr[d]) * vs);
        }
    }
    free(scores);
    return ORA_OK;
}

/* Ragged causal prefill over an fp8 cache: as ora_prefill (same request
 * layout, bottom-right aligned causal mask, selection and checks), with key j
 * of kv head h read as e4m3_value(K8[slot_j, h, :]) * k_scale[layer, h] and
 * value rows likewise with v_scale.  The scheme is the reading stated above
 * ora_kv_store_fp8 (page "e58a728" names only an fp8 test). */
int ora_prefill_fp8(const uint16_t *q, int64_t T, int Hq, const uint8_t *k_buf,
                    const uint8_t *v_buf, int n_layers, int64_t size, int Hkv,
                    int D, int layer, const int32_t *qo_indptr,
                    const int32_t *kv_indptr, int R, const int32_t *req_to_token,
                    int req_rows, int max_ctx, const int32_t *req_pool_indices,
                    double scale, const float *k_scale, const float *v_scale,
                    const int32_t *sel_t, const int32_t *sel_h, int64_t n_sel,
                    double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || layer < 0 || layer >= n_layers || D <= 0 || R < 0)
        return ORA_ERR_SHAPE;
    if (qo_indptr[0] != 0 || qo_indptr[R] != T || kv_indptr[0] != 0)
        return ORA_ERR_SHAPE;
    for (int r = 0; r < R; ++r) {
        int n_r = qo_indptr[r + 1] - qo_indptr[r];
        int L_r = kv_indptr[r + 1] - kv_indptr[r];
        if (n_r < 0 || L_r < n_r || L_r > max_ctx)
            return ORA_ERR_SHAPE;
        int row = req_pool_indices[r];
        if (row < 0 || row >= req_rows)
            return ORA_ERR_INDEX;
        for (int j = 0; j < L_r; ++j) {
            int32_t s = req_to_token[(int64_t)row * max_ctx + j];
            if (s < 0 || (int64_t)s >= size)
                return ORA_ERR_INDEX;
        }
    }
    const int G = Hq / Hkv;
    const int64_t slot_stride = (int64_t)Hkv * D;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    if (!scores)
        return ORA_ERR_NOMEM;
    const int64_t npairs = sel_t ? n_sel : T * Hq;
    for (int64_t i = 0; i < npairs; ++i) {
        int64_t t = sel_t ? sel_t[i] : i / Hq;
        int hq = sel_t ? sel_h[i] : (int)(i % Hq);
        if (t < 0 || t >= T || hq < 0 || hq >= Hq) {
            free(scores);
            return ORA_ERR_SHAPE;
        }
        int r = 0;
        while (!(qo_indptr[r] <= t && t < qo_indptr[r + 1]))
            ++r;
        int n_r = qo_indptr[r + 1] - qo_indptr[r];
        int L_r = kv_indptr[r + 1] - kv_indptr[r];
        int64_t n = (L_r - n_r) + (t - qo_indptr[r]) + 1;   /* positions 0 .. p_r + i */
        int h = hq / G;
        const int32_t *slots = req_to_token + (int64_t)req_pool_indices[r] * max_ctx;
        const uint16_t *qv = q + (t * Hq + hq) * D;
        const uint8_t *k0 = k_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        const uint8_t *v0 = v_buf + (int64_t)layer * size * slot_stride + (int64_t)h * D;
        const double ks = (double)k_scale[(int64_t)layer * Hkv + h];
        const double vs = (double)v_scale[(int64_t)layer * Hkv + h];
        double *o = out + i * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            const uint8_t *kr = k0 + (int64_t)slots[j] * slot_stride;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += ora_bf16_to_f64(qv[d]) * (ora_e4m3_to_f64(kr[d]) * ks);
            scores[j] = scale * dot;
            if (scores[j] > m)
                m = scores[j];
        }
        double denom = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            scores[j] = exp(scores[j] - m);
            denom += scores[j];
        }
        for (int64_t j = 0; j < n; ++j) {
            const uint8_t *vr = v0 + (int64_t)slots[j] * slot_stride;
            double w = scores[j] / denom;
            for (int d = 0; d < D; ++d)
                o[d] += w * (ora_e4m3_to_f64(vr[d]) * vs);
        }
    }
    free(scores);
    return ORA_OK;
}

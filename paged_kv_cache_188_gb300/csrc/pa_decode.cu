// pa_decode.cu -- packed GQA split-KV decode attention over the paged cache.
//
// What it computes (AstrAI commit 398e8a3, tests/inference/test_cache.py:
// packed decode with int32 req_to_token / req_pool_indices / seq_lens and
// workspace-owned split partials decode_o_part / decode_ml_part; commit
// e58a728, docs/developer/architecture.md: decode reads K/V via req_to_token):
// for request b and query head hq, softmax(scale * q K^T) V over the request's
// seq_lens[b] cached tokens, K/V rows gathered through req_to_token.
//
// How (one kernel, persistent grid of (#SM x resident CTAs)):
//  * Planning on the device, redundantly in every CTA: sum of seq_lens ->
//    split length; per request the split count s_b (<= max_splits); a prefix
//    sum over s_b * Hkv enumerates work items (b, split, kv head).  The grid
//    never depends on device lengths, so a captured graph stays valid.
//  * An item loads its token range's slots from req_to_token into shared
//    memory once, then each of the 4 warps streams 16-token tiles of K and V
//    (one kv head: 16 rows x 256 B, rows anywhere in the cache) through its own
//    cp.async ring.  Rows are stored with a 16-byte-chunk XOR swizzle so the
//    ldmatrix reads below are bank-conflict free.
//  * QK^T and PV use the warp-level bf16 MMA (m16n8k16): the G query heads of
//    one kv head form the M=16 rows, so K/V bytes are read once for all G
//    heads and the fp32 FMA count does not grow with G.  Online softmax in the
//    log2 domain (exp2), fp32 state per warp.
//  * The warps' states merge in shared memory; a request with one split writes
//    bf16 output directly, otherwise the item writes fp32 (o, m, l) partials
//    and the CTA that completes a (request, kv head) -- an integer atomic
//    ticket, no waiting -- merges all splits in split order (deterministic),
//    writes bf16 and re-arms the ticket to zero.
#include <math.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecTile = 16;        // tokens per warp tile
constexpr int kDecIdxWin = 1024;    // req_to_token entries staged per window
constexpr int kDecMinChunk = 64;    // split length bounds (tokens)
constexpr int kDecMaxChunk = 1024;
constexpr int kDecMaxBatch = 4096;
constexpr int kDecMaxSplits = 256;

struct DecodeArgs {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_layer;
    const __nv_bfloat16 *v_layer;
    const int32_t *req_to_token;
    const int32_t *req_pool_indices;
    const int32_t *seq_lens;
    __nv_bfloat16 *out;
    int32_t *err;
    int32_t *counters;
    float *ml_part;
    float *o_part;
    int batch, Hq, Hkv, G;
    int size, req_rows, max_ctx;
    int cap_batch, max_splits;
    float scale_log2;
};

__device__ __forceinline__ int clamp_len(int n, int max_ctx) { return n < 0 ? 0 : (n > max_ctx ? max_ctx : n); }

// split count and split length (tokens) of a request of n tokens
__device__ __forceinline__ void split_of(int n, int chunk, int max_splits, int &sb, int &len)
{
    if (n <= 0) {
        sb = 1;
        len = 0;
        return;
    }
    int s = (n + chunk - 1) / chunk;
    if (s > max_splits) s = max_splits;
    len = ((n + s - 1) / s + 15) & ~15;
    sb = (n + len - 1) / len;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D, int STAGES>
struct DecodeSmem {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kDecTile * kRowBytes;          // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;               // K + V
    static constexpr int kRingBytes = STAGES * kStageBytes;          // per warp
    static constexpr int kKvBytes = kDecWarps * kRingBytes;
    static constexpr int kIdxOff = kKvBytes;
    static constexpr int kPrefOff = kIdxOff + kDecIdxWin * 4;
    static size_t bytes(int batch) { return (size_t)kPrefOff + (size_t)(batch + 1) * 4; }
};

template <int D, int STAGES>
__global__ void __launch_bounds__(kDecThreads, 1) paged_decode_kernel(const DecodeArgs a)
{
    using L = DecodeSmem<D, STAGES>;
    constexpr int CPR = D / 8;            // 16-byte chunks per row
    constexpr int TPI = 32 / CPR;         // rows covered by one warp-wide copy instruction
    constexpr int COPIES = kDecTile / TPI;
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;             // n-tiles of the output

    extern __shared__ __align__(128) unsigned char smem[];
    int32_t *s_idx = reinterpret_cast<int32_t *>(smem + L::kIdxOff);
    int32_t *s_pref = reinterpret_cast<int32_t *>(smem + L::kPrefOff);
    __shared__ float s_m[kDecWarps][16], s_l[kDecWarps][16];
    __shared__ int s_red[kDecWarps];
    __shared__ int s_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int B = a.batch, Hkv = a.Hkv, G = a.G;

    // ---------------------------------------------------------- planning
    int my_tot = 0;
    for (int b = tid; b < B; b += kDecThreads) my_tot += clamp_len(__ldg(a.seq_lens + b), a.max_ctx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_tot += __shfl_xor_sync(0xffffffffu, my_tot, o);
    if (lane == 0) s_red[warp] = my_tot;
    __syncthreads();
    long long tot = 0;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) tot += s_red[w];
    long long want = (tot * Hkv + gridDim.x - 1) / gridDim.x;
    int chunk = (int)((want + kDecMinChunk - 1) / kDecMinChunk * kDecMinChunk);
    chunk = chunk < kDecMinChunk ? kDecMinChunk : (chunk > kDecMaxChunk ? kDecMaxChunk : chunk);

    // exclusive prefix of s_b * Hkv over requests; each thread scans a contiguous run
    const int per = (B + kDecThreads - 1) / kDecThreads;
    const int b_lo = tid * per, b_hi = min(B, b_lo + per);
    int run = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        int sb, len;
        split_of(clamp_len(__ldg(a.seq_lens + b), a.max_ctx), chunk, a.max_splits, sb, len);
        run += sb * Hkv;
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    __syncthreads();   // s_red reuse
    if (lane == 31) s_red[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_red[w];
    int excl = base + incl - run;
    for (int b = b_lo; b < b_hi; ++b) {
        s_pref[b] = excl;
        int sb, len;
        split_of(clamp_len(__ldg(a.seq_lens + b), a.max_ctx), chunk, a.max_splits, sb, len);
        excl += sb * Hkv;
    }
    if (tid == kDecThreads - 1) s_pref[B] = base + incl;
    __syncthreads();
    const int total_items = s_pref[B];

    const uint32_t ring = smem_u32(smem) + warp * L::kRingBytes;

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        // ------------------------------------------------ item -> (b, s, h)
        int lo = 0, hi = B;   // largest b with s_pref[b] <= item
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (s_pref[mid] <= item) lo = mid; else hi = mid;
        }
        const int b = lo;
        const int local = item - s_pref[b];
        const int s = local / Hkv, h = local - s * Hkv;
        int n = __ldg(a.seq_lens + b);
        if (n < 0 || n > a.max_ctx) {
            if (tid == 0 && s == 0 && h == 0) set_error(a.err, PA_DEVERR_LEN);
            n = clamp_len(n, a.max_ctx);
        }
        int sb, len;
        split_of(n, chunk, a.max_splits, sb, len);
        const int row = __ldg(a.req_pool_indices + b);
        if (row < 0 || row >= a.req_rows) {
            if (tid == 0 && s == 0 && h == 0) set_error(a.err, PA_DEVERR_ROW);
            n = 0;    // treated as empty: zeros out
        }
        const int t0 = s * len, t1 = min(n, t0 + len);
        const int32_t *r2t = a.req_to_token + (int64_t)(row < 0 || row >= a.req_rows ? 0 : row) * a.max_ctx;

        // query fragments: rows = the G heads of kv head h, zero beyond G
        uint32_t qa[KSTEPS][4];
        {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(a.q + ((int64_t)b * a.Hq + h * G) * D);
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int c0 = kk * 8 + t4;     // 32-bit column index (pairs of bf16)
                qa[kk][0] = g < G ? __ldg(q32 + g * (D / 2) + c0) : 0u;
                qa[kk][1] = g + 8 < G ? __ldg(q32 + (g + 8) * (D / 2) + c0) : 0u;
                qa[kk][2] = g < G ? __ldg(q32 + g * (D / 2) + c0 + 4) : 0u;
                qa[kk][3] = g + 8 < G ? __ldg(q32 + (g + 8) * (D / 2) + c0 + 4) : 0u;
            }
        }

        float o_acc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        const __nv_bfloat16 *kh = a.k_layer + (int64_t)h * D;
        const __nv_bfloat16 *vh = a.v_layer + (int64_t)h * D;
        const int64_t slot_stride = (int64_t)Hkv * D;

        for (int w0 = t0; w0 < t1; w0 += kDecIdxWin) {
            const int nwin = min(kDecIdxWin, t1 - w0);
            __syncthreads();
            for (int i = tid; i < nwin; i += kDecThreads) {
                int sl = __ldg(r2t + w0 + i);
                if (sl < 0 || sl >= a.size) {
                    set_error(a.err, PA_DEVERR_SLOT);
                    sl = -1;
                }
                s_idx[i] = sl;
            }
            __syncthreads();

            const int n_tiles = (nwin + kDecTile - 1) / kDecTile;
            const int my_tiles = n_tiles > warp ? (n_tiles - warp + kDecWarps - 1) / kDecWarps : 0;

            auto issue = [&](int it) {
                const int tile = warp + it * kDecWarps;
                const uint32_t st_base = ring + (it % STAGES) * L::kStageBytes;
#pragma unroll
                for (int c = 0; c < COPIES; ++c) {
                    const int r = c * TPI + lane / CPR;     // row within tile
                    const int ch = lane % CPR;
                    const int tok = tile * kDecTile + r;
                    const int sl = tok < nwin ? s_idx[tok] : -1;
                    const int64_t off = sl >= 0 ? (int64_t)sl * slot_stride + ch * 8 : 0;
                    const int nb = sl >= 0 ? 16 : 0;
                    const uint32_t dst = st_base + r * L::kRowBytes + ((ch ^ (r & 7)) << 4);
                    cp_async_16(dst, kh + off, nb);
                    cp_async_16(dst + L::kTileBytes, vh + off, nb);
                }
            };

#pragma unroll
            for (int i = 0; i < STAGES - 1; ++i) {
                if (i < my_tiles) issue(i);
                cp_async_commit();
            }
            for (int it = 0; it < my_tiles; ++it) {
                if (it + STAGES - 1 < my_tiles) issue(it + STAGES - 1);
                cp_async_commit();
                cp_async_wait<STAGES - 1>();
                __syncwarp();

                const int tile = warp + it * kDecWarps;
                const uint32_t kb = ring + (it % STAGES) * L::kStageBytes;
                const uint32_t vb = kb + L::kTileBytes;

                // S = Q K^T for 16 tokens (two n-tiles of 8)
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int r = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        const int ch = kk * 2 + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(kb + r * L::kRowBytes + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
                        mma_bf16_16816(sc[0], qa[kk], b0, b1);
                        mma_bf16_16816(sc[1], qa[kk], b2, b3);
                    }
                }
                // mask + online softmax (log2 domain)
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = tile * kDecTile + nt * 8 + 2 * t4 + e;
                        const bool ok = tok < nwin && s_idx[tok] >= 0;
                        sc[nt][e] = ok ? sc[nt][e] * a.scale_log2 : -INFINITY;
                        sc[nt][e + 2] = ok ? sc[nt][e + 2] * a.scale_log2 : -INFINITY;
                        mx0 = fmaxf(mx0, sc[nt][e]);
                        mx1 = fmaxf(mx1, sc[nt][e + 2]);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float mr0 = mn0 == -INFINITY ? 0.f : mn0;
                const float mr1 = mn1 == -INFINITY ? 0.f : mn1;
                const float al0 = ex2(m0 - mr0), al1 = ex2(m1 - mr1);
                m0 = mn0;
                m1 = mn1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    sc[nt][0] = ex2(sc[nt][0] - mr0);
                    sc[nt][1] = ex2(sc[nt][1] - mr0);
                    sc[nt][2] = ex2(sc[nt][2] - mr1);
                    sc[nt][3] = ex2(sc[nt][3] - mr1);
                    ps0 += sc[nt][0] + sc[nt][1];
                    ps1 += sc[nt][2] + sc[nt][3];
                }
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    o_acc[i][0] *= al0;
                    o_acc[i][1] *= al0;
                    o_acc[i][2] *= al1;
                    o_acc[i][3] *= al1;
                }
                uint32_t pa_[4];
                pa_[0] = pack_bf16x2(sc[0][0], sc[0][1]);
                pa_[1] = pack_bf16x2(sc[0][2], sc[0][3]);
                pa_[2] = pack_bf16x2(sc[1][0], sc[1][1]);
                pa_[3] = pack_bf16x2(sc[1][2], sc[1][3]);
                // O += P V
                {
                    const int mi = lane >> 3;
                    const int r = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int np = 0; np < D / 16; ++np) {
                        const int ch = np * 2 + (mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4_trans(vb + r * L::kRowBytes + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
                        mma_bf16_16816(o_acc[2 * np], pa_, b0, b1);
                        mma_bf16_16816(o_acc[2 * np + 1], pa_, b2, b3);
                    }
                }
                __syncwarp();
            }
            cp_async_wait<0>();
        }

        // ---------------------------------------- merge the warps' states
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        __syncthreads();   // every warp is done with its ring: reuse it as scratch
        float *s_o = reinterpret_cast<float *>(smem);   // [warps][G][D]
        if (t4 == 0) {
            if (g < G) {
                s_m[warp][g] = m0;
                s_l[warp][g] = l0;
            }
            if (g + 8 < G) {
                s_m[warp][g + 8] = m1;
                s_l[warp][g + 8] = l1;
            }
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int d = i * 8 + 2 * t4;
            if (g < G) {
                s_o[(warp * G + g) * D + d] = o_acc[i][0];
                s_o[(warp * G + g) * D + d + 1] = o_acc[i][1];
            }
            if (g + 8 < G) {
                s_o[(warp * G + g + 8) * D + d] = o_acc[i][2];
                s_o[(warp * G + g + 8) * D + d + 1] = o_acc[i][3];
            }
        }
        __syncthreads();
        const int hq0 = h * G;
        for (int e = tid; e < G * D; e += kDecThreads) {
            const int gg = e / D, d = e - gg * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w][gg]);
            const float Mr = M == -INFINITY ? 0.f : M;
            float lsum = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                const float wt = ex2(s_m[w][gg] - Mr);
                lsum += wt * s_l[w][gg];
                acc += wt * s_o[(w * G + gg) * D + d];
            }
            if (sb == 1) {
                a.out[((int64_t)b * a.Hq + hq0 + gg) * D + d] = __float2bfloat16_rn(lsum > 0.f ? acc / lsum : 0.f);
            } else {
                const int64_t pr = ((int64_t)s * a.cap_batch + b) * a.Hq + hq0 + gg;
                a.o_part[pr * D + d] = acc;
                if (d == 0) {
                    a.ml_part[pr * 2] = M;
                    a.ml_part[pr * 2 + 1] = lsum;
                }
            }
        }

        if (sb > 1) {
            // ------------------------- last CTA of (b, h) merges the splits
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int prev = atomicAdd(a.counters + b * Hkv + h, 1);
                s_flag = prev == sb - 1;
                __threadfence();
            }
            __syncthreads();
            if (s_flag) {
                float *s_ml = reinterpret_cast<float *>(smem);            // [sb][G][2]
                float *s_w = s_ml + 2 * kDecMaxSplits * 16;                // [sb][G]
                float *s_lt = s_w + kDecMaxSplits * 16;                    // [G]
                for (int i = tid; i < sb * G; i += kDecThreads) {
                    const int ss = i / G, gg = i - ss * G;
                    const int64_t pr = ((int64_t)ss * a.cap_batch + b) * a.Hq + hq0 + gg;
                    s_ml[i * 2] = __ldcg(a.ml_part + pr * 2);
                    s_ml[i * 2 + 1] = __ldcg(a.ml_part + pr * 2 + 1);
                }
                __syncthreads();
                for (int gg = tid; gg < G; gg += kDecThreads) {
                    float M = -INFINITY;
                    for (int ss = 0; ss < sb; ++ss) M = fmaxf(M, s_ml[(ss * G + gg) * 2]);
                    const float Mr = M == -INFINITY ? 0.f : M;
                    float lt = 0.f;
                    for (int ss = 0; ss < sb; ++ss) {
                        const float wt = ex2(s_ml[(ss * G + gg) * 2] - Mr);
                        s_w[ss * G + gg] = wt;
                        lt += wt * s_ml[(ss * G + gg) * 2 + 1];
                    }
                    s_lt[gg] = lt;
                }
                __syncthreads();
                const int64_t split_stride = (int64_t)a.cap_batch * a.Hq * D;
                for (int e = tid; e < G * D; e += kDecThreads) {
                    const int gg = e / D, d = e - gg * D;
                    const float *src = a.o_part + ((int64_t)b * a.Hq + hq0 + gg) * D + d;
                    float acc = 0.f;
                    int ss = 0;
                    // eight independent loads in flight, summed in split order
                    for (; ss + 8 <= sb; ss += 8) {
                        float v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (ss + j) * split_stride);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc += s_w[(ss + j) * G + gg] * v[j];
                    }
                    for (; ss < sb; ++ss) acc += s_w[ss * G + gg] * __ldcg(src + ss * split_stride);
                    const float lt = s_lt[gg];
                    a.out[((int64_t)b * a.Hq + hq0 + gg) * D + d] = __float2bfloat16_rn(lt > 0.f ? acc / lt : 0.f);
                }
                if (tid == 0) a.counters[b * Hkv + h] = 0;
            }
        }
        __syncthreads();
    }
}

template <int D, int STAGES>
static pa_status launch_decode(const DecodeArgs &a, cudaStream_t st)
{
    auto kern = paged_decode_kernel<D, STAGES>;
    const size_t smem = DecodeSmem<D, STAGES>::bytes(a.batch);
    static size_t configured = 0;
    if (smem > configured) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return PA_ERR_CUDA;
        configured = smem;
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDecThreads, smem) != cudaSuccess || occ < 1)
        return PA_ERR_CUDA;
    const int grid = num_sms() * occ;
    kern<<<grid, kDecThreads, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
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
    if (batch < 0 || batch > kDecMaxBatch || n_q_heads <= 0 || s.n_layers <= 0 || s.size <= 0 ||
        s.n_kv_heads <= 0 || req_rows <= 0 || max_ctx <= 0 || max_splits < 1 || max_splits > kDecMaxSplits)
        return PA_ERR_SHAPE;
    if (layer_id < 0 || layer_id >= s.n_layers) return PA_ERR_SHAPE;
    if (n_q_heads % s.n_kv_heads != 0) return PA_ERR_SHAPE;
    const int G = n_q_heads / s.n_kv_heads;
    if (G > 16 || (s.head_dim != 64 && s.head_dim != 128)) return PA_ERR_UNSUPPORTED;
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    const DecodeWsLayout ws = decode_ws_layout(workspace_bytes, n_q_heads, s.n_kv_heads, s.head_dim, max_splits);
    if (ws.cap_batch < batch || ws.total > workspace_bytes) return PA_ERR_WORKSPACE;
    if (batch == 0) return PA_OK;
    if (!q || !k_buf || !v_buf || !req_to_token || !req_pool_indices || !seq_lens || !out) return PA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_buf) || !aligned16(v_buf) || !aligned16(out) || !aligned4(req_to_token) ||
        !aligned4(req_pool_indices) || !aligned4(seq_lens))
        return PA_ERR_ALIGN;

    DecodeArgs a{};
    const int64_t layer_off = (int64_t)layer_id * s.size * s.n_kv_heads * s.head_dim;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k_layer = static_cast<const __nv_bfloat16 *>(k_buf) + layer_off;
    a.v_layer = static_cast<const __nv_bfloat16 *>(v_buf) + layer_off;
    a.req_to_token = req_to_token;
    a.req_pool_indices = req_pool_indices;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    unsigned char *w = static_cast<unsigned char *>(workspace);
    a.err = reinterpret_cast<int32_t *>(w);
    a.counters = reinterpret_cast<int32_t *>(w + ws.counters_off);
    a.ml_part = reinterpret_cast<float *>(w + ws.ml_off);
    a.o_part = reinterpret_cast<float *>(w + ws.o_off);
    a.batch = batch;
    a.Hq = n_q_heads;
    a.Hkv = s.n_kv_heads;
    a.G = G;
    a.size = s.size;
    a.req_rows = req_rows;
    a.max_ctx = max_ctx;
    a.cap_batch = ws.cap_batch;
    a.max_splits = max_splits;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    if (s.head_dim == 128) return launch_decode<128, 3>(a, st);
    return launch_decode<64, 4>(a, st);
}

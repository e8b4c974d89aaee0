// pa_prefill.cu -- ragged causal prefill over the paged KV cache on tcgen05.
//
// What it computes (AstrAI commit e58a728, docs/developer/architecture.md:
// prompts packed into one forward with cumulative query lengths qo_indptr,
// attn_paged_prefill over cached prefix pages; commit 398e8a3,
// tests/inference/test_cache.py: int32 request rows / page table): query i of
// request r (position p_r + i, p_r = cached prefix) attends to positions
// 0 .. p_r + i of the request, K/V rows read through req_to_token.
//
// How (persistent, one CTA per SM, warp-specialised, 320 threads):
//  * Work item = (request, q-tile, kv head).  A q-tile packs the G query heads
//    of one kv head into the MMA's M = 128 rows: 128/G consecutive tokens x G
//    heads (token-major), so each K/V tile fetched serves all G heads.
//  * warp 8 (producer): TMA.  Q tile via a 3-D tensor map (d, head, token);
//    K/V tiles of 128 positions gathered through req_to_token: a group of 16
//    positions on 16 consecutive slots (one page) is one 16-row box per 64-wide
//    half, anything else falls back to 1-row boxes; positions past the item's
//    last visible key load zeros (out-of-range rows).  128-byte swizzle, the
//    layout the UMMA descriptors below expect.  Two K and two V stages.
//  * warp 9 (MMA issuer, one thread): S = Q K^T into one of two TMEM buffers
//    (128 lanes x 128 fp32 columns), O += P V into a third; commits signal the
//    other warps.  S(t+1) is issued before PV(t) so the tensor core works on
//    the next scores while the softmax warps finish the current tile.
//  * warps 0-7 (softmax + epilogue): row i = TMEM lane i, warpgroup h owns
//    columns [64h, 64h+64) of S, O and P; the two halves of a row exchange
//    their maxima (and at the end their sums) through shared memory.  Causal
//    mask (bottom-right aligned) only on diagonal tiles, online softmax in the
//    log2 domain with a lazy running max (O in TMEM is rescaled only when the
//    max grows by more than 2^8), P rounded to bf16 into shared memory as the
//    A operand of the PV MMA.  Epilogue: O / l to bf16, rows of padding tokens
//    are not written.
//  * Every mbarrier wait is bounded in time; on a time-out the CTA raises an
//    abort flag, sets PA_DEVERR_TIMEOUT and unwinds, freeing its TMEM.
#include <cuda.h>
#include <math.h>

#include "pa_internal.h"
#include "pa_sm100.cuh"

namespace pa {
using namespace sm100;

constexpr int kPfRows = 128;           // MMA M: rows of a q tile
constexpr int kPfKeys = 128;           // keys per kv tile
constexpr int kPfD = 128;              // head dim
constexpr int kPfSoftmaxThreads = 256;  // warps 0-7: two warpgroups, one per 64-column half
constexpr int kPfThreads = 320;         // + warp 8 (TMA producer) + warp 9 (MMA issuer)
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr int kPfMaxReqs = 2048;
constexpr int kHalf = 128 * 128;       // one 128-row x 128-byte swizzled half tile (16 KB)
constexpr int kOffQ = 0;               // 2 halves
constexpr int kOffK = 2 * kHalf;       // 2 stages x 2 halves
constexpr int kOffV = 6 * kHalf;       // 2 stages x 2 halves
constexpr int kOffP = 10 * kHalf;      // 2 halves
constexpr int kOffBar = 12 * kHalf;
enum { Q_FULL, Q_EMPTY, K_FULL, K_FULL1, K_EMPTY, K_EMPTY1, V_FULL, V_FULL1, V_EMPTY, V_EMPTY1,
       S_FULL, S_FULL1, S_EMPTY, S_EMPTY1, P_FULL, O_DONE, O_EMPTY, XCH0, XCH1, XCH2, XCH3, N_BARS };
constexpr int kOffMisc = kOffBar + 32 * 8;
constexpr int kOffXch = kOffMisc + 64;            // row max / sum exchange between the two halves
constexpr int kOffPref = kOffXch + 3 * 128 * 4 * 2;
constexpr uint32_t kTmemCols = 512;    // S0 | S1 | O | unused
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);   // Q (K-major) x K (K-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);  // P (K-major) x V (MN-major)

struct PrefillParams {
    CUtensorMap tm_q;     // 3-D (d, head, token) over q [T, Hq, 128]
    CUtensorMap tm_k16;   // 2-D (element, row) over k_buf rows, 64 x 16 boxes
    CUtensorMap tm_k1;    //                                  64 x 1 boxes
    CUtensorMap tm_v16;
    CUtensorMap tm_v1;
    const int32_t *qo_indptr;
    const int32_t *kv_indptr;
    const int32_t *req_to_token;
    const int32_t *req_pool_indices;
    __nv_bfloat16 *out;
    int32_t *err;
    int T, Hq, Hkv, G, TQ, R;
    int size, layer_row0, total_rows, req_rows, max_ctx;
    float scale_log2;
};

struct PfItem {
    int h, qs, q0, nq, p, row, n_keys, ntiles;
};

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ PfItem pf_item(const PrefillParams &p, const int *s_pref, int item)
{
    int lo = 0, hi = p.R;   // largest r with s_pref[r] <= item
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] <= item) lo = mid; else hi = mid;
    }
    const int r = lo;
    const int local = item - s_pref[r];
    const int tiles_r = (s_pref[r + 1] - s_pref[r]) / p.Hkv;
    const int jj = local / p.Hkv;
    PfItem I;
    I.h = local - jj * p.Hkv;
    const int j = tiles_r - 1 - jj;            // later (heavier) q tiles first
    I.qs = __ldg(p.qo_indptr + r);
    const int n_r = __ldg(p.qo_indptr + r + 1) - I.qs;
    const int L_r = __ldg(p.kv_indptr + r + 1) - __ldg(p.kv_indptr + r);
    I.p = L_r - n_r;
    I.q0 = j * p.TQ;
    I.nq = min(p.TQ, n_r - I.q0);
    I.row = __ldg(p.req_pool_indices + r);
    I.n_keys = I.p + I.q0 + I.nq;
    I.ntiles = (I.n_keys + kPfKeys - 1) / kPfKeys;
    return I;
}

__global__ void __launch_bounds__(kPfThreads, 1) paged_prefill_kernel(const __grid_constant__ PrefillParams p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *sb = smem_raw + (base - raw);
    const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sP = base + kOffP;
    volatile int *s_abort = reinterpret_cast<volatile int *>(sb + kOffMisc);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sb + kOffMisc + 4);
    int *s_wsum = reinterpret_cast<int *>(sb + kOffMisc + 8);    // one int per warp
    int *s_pref = reinterpret_cast<int *>(sb + kOffPref);
    auto bar = [&](int i) -> uint32_t { return base + kOffBar + i * 8; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *err = p.err;

    if (tid == 0) {
        *s_abort = 0;
        for (int i = 0; i < N_BARS; ++i) {
            const uint32_t cnt = (i == S_EMPTY || i == S_EMPTY1 || i == P_FULL || i == O_EMPTY)
                                     ? (uint32_t)kPfSoftmaxThreads
                                     : (i >= XCH0 ? 64u : 1u);
            mbar_init(bar(i), cnt);
        }
        fence_mbar_init();
    }
    if (warp == kWarpMma) tmem_alloc(smem_u32(s_tmem), kTmemCols);
    if (warp == kWarpProducer && lane == 0) {
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k16);
        prefetch_tmap(&p.tm_k1);
        prefetch_tmap(&p.tm_v16);
        prefetch_tmap(&p.tm_v1);
    }

    // ---------------------------------------------------------- planning
    // q tiles per request (0 for an invalid request), exclusive prefix of
    // tiles * Hkv; every thread scans a contiguous run of requests
    {
        const int per = (p.R + kPfThreads - 1) / kPfThreads;
        const int r_lo = min(p.R, tid * per), r_hi = min(p.R, r_lo + per);
        auto tiles_of = [&](int r) -> int {
            const int qa = __ldg(p.qo_indptr + r), qb = __ldg(p.qo_indptr + r + 1);
            const int n_r = qb - qa;
            const int L_r = __ldg(p.kv_indptr + r + 1) - __ldg(p.kv_indptr + r);
            const int row = __ldg(p.req_pool_indices + r);
            if (n_r <= 0) {
                if (n_r < 0) set_error(err, PA_DEVERR_LEN);
                return 0;
            }
            if (qa < 0 || qb > p.T || L_r < n_r || L_r > p.max_ctx) {
                set_error(err, PA_DEVERR_LEN);
                return 0;
            }
            if (row < 0 || row >= p.req_rows) {
                set_error(err, PA_DEVERR_ROW);
                return 0;
            }
            return (n_r + p.TQ - 1) / p.TQ;
        };
        int run = 0;
        for (int r = r_lo; r < r_hi; ++r) run += tiles_of(r) * p.Hkv;
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int wbase = 0;
        for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
        int excl = wbase + incl - run;
        for (int r = r_lo; r < r_hi; ++r) {
            s_pref[r] = excl;
            excl += tiles_of(r) * p.Hkv;
        }
        if (tid == kPfThreads - 1) s_pref[p.R] = wbase + incl;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int total_items = s_pref[p.R];
    const int G = p.G;

    if (warp == kWarpProducer) {
        // ================================================== TMA producer
        int kt = 0, it = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x, ++it) {
            const PfItem I = pf_item(p, s_pref, item);
            if (it > 0 && !mbar_wait(bar(Q_EMPTY), (it - 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(Q_FULL), 2 * kHalf);
                tma_load_3d(sQ, &p.tm_q, 0, I.h * G, I.qs + I.q0, bar(Q_FULL));
                tma_load_3d(sQ + kHalf, &p.tm_q, 64, I.h * G, I.qs + I.q0, bar(Q_FULL));
            }
            const int32_t *r2t = p.req_to_token + (int64_t)I.row * p.max_ctx;
            const int col0 = I.h * kPfD;
            const int gi = lane >> 2, sub = lane & 3;
            for (int t = 0; t < I.ntiles; ++t, ++kt) {
                const int st = kt & 1;
                const uint32_t ph_prev = ((kt >> 1) - 1) & 1;
                // slots of positions k0 + 4*lane + e
                const int k0 = t * kPfKeys;
                int slot[4];
                bool okp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = k0 + 4 * lane + e;
                    okp[e] = pos < I.n_keys;
                    slot[e] = okp[e] ? __ldg(r2t + pos) : -1;
                    if (okp[e] && (slot[e] < 0 || slot[e] >= p.size)) {
                        set_error(err, PA_DEVERR_SLOT);
                        okp[e] = false;
                    }
                }
                const int s0 = __shfl_sync(0xffffffffu, slot[0], lane & ~3);
                const bool mine = okp[0] && okp[1] && okp[2] && okp[3] && slot[0] == s0 + 4 * sub &&
                                  slot[1] == slot[0] + 1 && slot[2] == slot[0] + 2 && slot[3] == slot[0] + 3;
                const unsigned contig = __ballot_sync(0xffffffffu, mine);
                const unsigned anyok = __ballot_sync(0xffffffffu, okp[0] || okp[1] || okp[2] || okp[3]);
                const bool g_contig = ((contig >> (lane & ~3)) & 0xFu) == 0xFu;
                const bool g_empty = ((anyok >> (lane & ~3)) & 0xFu) == 0u;

                auto issue = [&](const CUtensorMap *m16, const CUtensorMap *m1, uint32_t dst, uint32_t b) {
                    if (g_contig || g_empty) {
                        if (sub == 0) {
                            const int row = g_empty ? p.total_rows : p.layer_row0 + s0;
                            tma_load_2d(dst + gi * 16 * 128, m16, col0, row, b);
                            tma_load_2d(dst + kHalf + gi * 16 * 128, m16, col0 + 64, row, b);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int rr = 16 * gi + 4 * sub + e;
                            const int row = okp[e] ? p.layer_row0 + slot[e] : p.total_rows;
                            tma_load_2d(dst + rr * 128, m1, col0, row, b);
                            tma_load_2d(dst + kHalf + rr * 128, m1, col0 + 64, row, b);
                        }
                    }
                };
                if (kt >= 2 && !mbar_wait(bar(K_EMPTY + st), ph_prev, s_abort, err, PA_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(bar(K_FULL + st), 2 * kHalf);
                __syncwarp();
                issue(&p.tm_k16, &p.tm_k1, sK + st * 2 * kHalf, bar(K_FULL + st));
                if (kt >= 2 && !mbar_wait(bar(V_EMPTY + st), ph_prev, s_abort, err, PA_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(bar(V_FULL + st), 2 * kHalf);
                __syncwarp();
                issue(&p.tm_v16, &p.tm_v1, sV + st * 2 * kHalf, bar(V_FULL + st));
            }
        }
    } else if (warp == kWarpMma) {
        // ================================================== MMA issuer
        if (lane == 0) {
            int kt = 0, it = 0;
            int pend_kt = -1, pend_it = 0;
            bool pend_first = false, ok = true;
            auto issue_pv = [&](int pkt, bool first, int pit) -> bool {
                const int st = pkt & 1;
                if (!mbar_wait(bar(P_FULL), pkt & 1, s_abort, err, PA_DEVERR_TIMEOUT)) return false;
                if (!mbar_wait(bar(V_FULL + st), (pkt >> 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT)) return false;
                if (first && pit > 0 && !mbar_wait(bar(O_EMPTY), (pit - 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(sP + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(sV + st * 2 * kHalf + kk * 2048, kHalf, 1024);
                    umma_ss(tmem + 256, a, b, kIdescPV, (kk > 0 || !first) ? 1u : 0u);
                }
                umma_commit(bar(V_EMPTY + st));
                umma_commit(bar(O_DONE));
                return true;
            };
            for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x, ++it) {
                const PfItem I = pf_item(p, s_pref, item);
                if (!mbar_wait(bar(Q_FULL), it & 1, s_abort, err, PA_DEVERR_TIMEOUT)) break;
                for (int t = 0; t < I.ntiles; ++t, ++kt) {
                    const int st = kt & 1;
                    if (!mbar_wait(bar(K_FULL + st), (kt >> 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT) ||
                        (kt >= 2 &&
                         !mbar_wait(bar(S_EMPTY + st), ((kt >> 1) - 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kPfD / 16; ++kk) {
                        const uint64_t a = smem_desc_sw128(sQ + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                        const uint64_t b =
                            smem_desc_sw128(sK + st * 2 * kHalf + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                        umma_ss(tmem + st * 128, a, b, kIdescS, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(K_EMPTY + st));
                    umma_commit(bar(S_FULL + st));
                    if (t == I.ntiles - 1) umma_commit(bar(Q_EMPTY));
                    if (pend_kt >= 0 && !issue_pv(pend_kt, pend_first, pend_it)) {
                        ok = false;
                        break;
                    }
                    pend_kt = kt;
                    pend_first = (t == 0);
                    pend_it = it;
                }
            }
            if (ok && pend_kt >= 0) issue_pv(pend_kt, pend_first, pend_it);
        }
        __syncwarp();
    } else {
        // ============================ softmax + epilogue (row, column half)
        // thread -> row (TMEM lane) and one 64-column half of S, O and P
        const int half = warp >> 2;
        const int row = tid & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t o_addr = tmem + lane_base + 256 + half * 64;
        float *xmax = reinterpret_cast<float *>(sb + kOffXch);     // [parity][half][row]
        float *xsum = xmax + 4 * 128;                              // [half][row]
        const uint32_t xbar = bar(XCH0 + (warp & 3));
        uint32_t xph = 0;
        const float sl2 = p.scale_log2;
        int kt = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x) {
            const PfItem I = pf_item(p, s_pref, item);
            const int tok = row / G;                    // token of this row within the q tile
            const int qpos = I.p + I.q0 + tok;           // its position in the request
            float m_run = -INFINITY, l_run = 0.f;
            for (int t = 0; t < I.ntiles; ++t, ++kt) {
                const int st = kt & 1;
                if (!mbar_wait(bar(S_FULL + st), (kt >> 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r[64];
                {
                    uint32_t (&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
                    uint32_t (&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
                    const uint32_t s_addr = tmem + lane_base + st * 128 + half * 64;
                    tmem_ld32(s_addr, r0);
                    tmem_ld32(s_addr + 32, r1);
                    tmem_wait_ld();
                }
                const int limit = qpos - t * kPfKeys - half * 64;    // columns <= limit are visible
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
                if (limit >= 63) {
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        mx0 = fmaxf(mx0, __uint_as_float(r[c]));
                        mx1 = fmaxf(mx1, __uint_as_float(r[c + 1]));
                        mx2 = fmaxf(mx2, __uint_as_float(r[c + 2]));
                        mx3 = fmaxf(mx3, __uint_as_float(r[c + 3]));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const float v = c <= limit ? __uint_as_float(r[c]) : -INFINITY;
                        r[c] = __float_as_uint(v);
                        if ((c & 3) == 0) mx0 = fmaxf(mx0, v);
                        if ((c & 3) == 1) mx1 = fmaxf(mx1, v);
                        if ((c & 3) == 2) mx2 = fmaxf(mx2, v);
                        if ((c & 3) == 3) mx3 = fmaxf(mx3, v);
                    }
                }
                float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                // row maximum across the two halves
                xmax[((kt & 1) * 2 + half) * 128 + row] = mx;
                mbar_arrive(xbar);
                if (!mbar_wait(xbar, xph & 1, s_abort, err, PA_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                ++xph;
                mx = fmaxf(mx, xmax[((kt & 1) * 2 + (half ^ 1)) * 128 + row]);
                float m_new = m_run;
                bool rescale = false;
                if (mx > m_run && (m_run == -INFINITY || (mx - m_run) * sl2 > 8.f)) {
                    rescale = m_run != -INFINITY;
                    m_new = mx;
                }
                const float alpha = rescale ? ex2f((m_run - m_new) * sl2) : 1.f;
                m_run = m_new;
                const float mb = m_new == -INFINITY ? 0.f : m_new * sl2;
                uint32_t pk[32];
                float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float v0 = ex2f(fmaf(__uint_as_float(r[c]), sl2, -mb));
                    const float v1 = ex2f(fmaf(__uint_as_float(r[c + 1]), sl2, -mb));
                    sum0 += v0;
                    sum1 += v1;
                    pk[c / 2] = pack_bf16x2(v0, v1);
                }
                l_run = l_run * alpha + (sum0 + sum1);
                tc_fence_before();
                mbar_arrive(bar(S_EMPTY + st));
                // the previous PV must be done: P's buffer is free and O is stable
                if (kt > 0 && !mbar_wait(bar(O_DONE), (kt - 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (t > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + ch * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(o_addr + ch * 32, o);
                    }
                    tmem_wait_st();
                }
                // P: this half's 64 keys of the row -> its K-major 128-byte swizzled region
                unsigned char *prow = sb + kOffP + half * kHalf + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(prow + ((c ^ (row & 7)) << 4)) =
                        make_uint4(pk[c * 4], pk[c * 4 + 1], pk[c * 4 + 2], pk[c * 4 + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(P_FULL));
            }
            if (!ok) break;
            // ------------------------------------------------ epilogue
            if (!mbar_wait(bar(O_DONE), (kt - 1) & 1, s_abort, err, PA_DEVERR_TIMEOUT)) break;
            tc_fence_after();
            xsum[half * 128 + row] = l_run;
            mbar_arrive(xbar);
            if (!mbar_wait(xbar, xph & 1, s_abort, err, PA_DEVERR_TIMEOUT)) break;
            ++xph;
            const float l_tot = l_run + xsum[(half ^ 1) * 128 + row];
            const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const bool row_ok = tok < I.nq;
            __nv_bfloat16 *dst =
                p.out + ((int64_t)(I.qs + I.q0 + tok) * p.Hq + I.h * G + (row - tok * G)) * kPfD + half * 64;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t o[32];
                tmem_ld32(o_addr + ch * 32, o);
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[q * 8 + 0]) * inv_l, __uint_as_float(o[q * 8 + 1]) * inv_l);
                        v.y = pack_bf16x2(__uint_as_float(o[q * 8 + 2]) * inv_l, __uint_as_float(o[q * 8 + 3]) * inv_l);
                        v.z = pack_bf16x2(__uint_as_float(o[q * 8 + 4]) * inv_l, __uint_as_float(o[q * 8 + 5]) * inv_l);
                        v.w = pack_bf16x2(__uint_as_float(o[q * 8 + 6]) * inv_l, __uint_as_float(o[q * 8 + 7]) * inv_l);
                        *reinterpret_cast<uint4 *>(dst + ch * 32 + q * 8) = v;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(O_EMPTY));
        }
    }

    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host
static bool encode(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box)
{
    return encode_tmap_bf16(m, ptr, rank, dims, strides, box);
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_paged_prefill_attn(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                           const void *v_buf, pa_kv_shape s, int layer_id,
                                           const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                           const int32_t *req_to_token, int req_rows, int max_ctx,
                                           const int32_t *req_pool_indices, float scale, void *workspace,
                                           size_t workspace_bytes, void *out, cudaStream_t st)
{
    if (n_tokens < 0 || n_reqs < 0 || n_reqs > kPfMaxReqs || n_q_heads <= 0 || s.n_layers <= 0 || s.size <= 0 ||
        s.n_kv_heads <= 0 || req_rows <= 0 || max_ctx <= 0)
        return PA_ERR_SHAPE;
    if (layer_id < 0 || layer_id >= s.n_layers) return PA_ERR_SHAPE;
    if (n_q_heads % s.n_kv_heads != 0) return PA_ERR_SHAPE;
    const int G = n_q_heads / s.n_kv_heads;
    if (s.head_dim != kPfD || (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)) return PA_ERR_UNSUPPORTED;
    if ((int64_t)s.n_layers * s.size >= (int64_t)INT32_MAX - 16) return PA_ERR_SHAPE;
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    if (workspace_bytes < pa_prefill_workspace_bytes()) return PA_ERR_WORKSPACE;
    if (n_tokens == 0 || n_reqs == 0) return PA_OK;
    if (!q || !k_buf || !v_buf || !qo_indptr || !kv_indptr || !req_to_token || !req_pool_indices || !out)
        return PA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_buf) || !aligned16(v_buf) || !aligned16(out) || !aligned4(qo_indptr) ||
        !aligned4(kv_indptr) || !aligned4(req_to_token) || !aligned4(req_pool_indices))
        return PA_ERR_ALIGN;

    PrefillParams prm;
    memset(&prm, 0, sizeof prm);
    const int TQ = kPfRows / G;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kPfD, (cuuint64_t)n_q_heads, (cuuint64_t)n_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)kPfD * 2, (cuuint64_t)n_q_heads * kPfD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
        if (!encode(&prm.tm_q, q, 3, dims, strides, box)) return PA_ERR_CUDA;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)s.n_kv_heads * kPfD, (cuuint64_t)s.n_layers * s.size};
        const cuuint64_t strides[1] = {(cuuint64_t)s.n_kv_heads * kPfD * 2};
        const cuuint32_t box16[2] = {64, 16}, box1[2] = {64, 1};
        if (!encode(&prm.tm_k16, k_buf, 2, dims, strides, box16) || !encode(&prm.tm_k1, k_buf, 2, dims, strides, box1) ||
            !encode(&prm.tm_v16, v_buf, 2, dims, strides, box16) || !encode(&prm.tm_v1, v_buf, 2, dims, strides, box1))
            return PA_ERR_CUDA;
    }
    prm.qo_indptr = qo_indptr;
    prm.kv_indptr = kv_indptr;
    prm.req_to_token = req_to_token;
    prm.req_pool_indices = req_pool_indices;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.err = static_cast<int32_t *>(workspace);
    prm.T = n_tokens;
    prm.Hq = n_q_heads;
    prm.Hkv = s.n_kv_heads;
    prm.G = G;
    prm.TQ = TQ;
    prm.R = n_reqs;
    prm.size = s.size;
    prm.layer_row0 = layer_id * s.size;
    prm.total_rows = s.n_layers * s.size;
    prm.req_rows = req_rows;
    prm.max_ctx = max_ctx;
    prm.scale_log2 = (float)((double)scale * 1.4426950408889634);

    const size_t smem = (size_t)kOffPref + (size_t)(n_reqs + 1) * 4 + 1024;
    static size_t configured = 0;
    if (smem > configured) {
        if (cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        configured = smem;
    }
    paged_prefill_kernel<<<num_sms(), kPfThreads, smem, st>>>(prm);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

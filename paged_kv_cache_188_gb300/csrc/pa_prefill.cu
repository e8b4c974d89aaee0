// pa_prefill.cu -- ragged causal prefill over the paged KV cache on tcgen05.
//
// What it computes (AstrAI commit e58a728, docs/developer/architecture.md:
// prompts packed into one forward with cumulative query lengths qo_indptr,
// attn_paged_prefill over cached prefix pages; commit 398e8a3,
// tests/inference/test_cache.py: int32 request rows / page table): query i of
// request r (position p_r + i, p_r = cached prefix) attends to positions
// 0 .. p_r + i of the request, K/V rows read through req_to_token.
//
// How (persistent, one CTA per SM, warp-specialised, 352 threads):
//  * Work item = (request, pair of q tiles, kv head).  A q tile packs the G
//    query heads of one kv head into the MMA's M = 128 rows: 128/G
//    consecutive tokens x G heads (token-major).  The two tiles A and B of a
//    pair are consecutive and share every K/V tile the CTA fetches.
//  * Items are claimed from a counter in the workspace (heaviest pairs of a
//    request first), so CTAs that drew short items take more of them; the
//    producer hands each claim to the other roles through a small ring.
//  * warps 8 and 10 (producers): TMA; warp 8 claims the items and loads Q
//    and K, warp 10 loads V (fp8: warp 8 loads all three).  Q tiles via a
//    3-D tensor map (d, head, token); K/V tiles of 128 positions gathered
//    through req_to_token (the next tile's entries requested ahead): a group of 16
//    positions on 16 consecutive slots (one page) is one 16-row box per 64-wide
//    half, anything else falls back to 1-row boxes; positions past the pair's
//    last visible key load zeros (out-of-range rows).  128-byte swizzle, the
//    layout the UMMA descriptors below expect.  Two K and two V stages.
//  * warp 9 (MMA issuer, one thread), tensor memory S_A | S_B | O_A | O_B
//    (128 fp32 columns each):  S_X = Q_X K^T, then O_X += P_X V with P_X read
//    from tensor memory, where the softmax left it over S_X (bf16 pairs).  The
//    order S_A(t), S_B(t), PV_A(t), S_A(t+1), PV_B(t), S_B(t+1), ... gives each
//    softmax warpgroup two MMA groups' time for its tile while the tensor core
//    works on the other tile (ping-pong).
//  * warps 0-3 own tile A's rows, warps 4-7 tile B's (row i = TMEM lane i):
//    read S with tcgen05.ld, causal mask (bottom-right aligned) on diagonal
//    tiles only, online softmax in the log2 domain with a lazy running max (O
//    is rescaled in tensor memory only when the max grows by more than 2^8),
//    P rounded to bf16 and stored back with tcgen05.st.  Epilogue: O / l to
//    bf16, rows of padding tokens are not written.
//  * Launched behind another kernel (launch overlap on), the CTA waits for it
//    after its barrier and tensor-memory setup, or -- early-metadata mode --
//    after planning.
//  * Every mbarrier wait is bounded in time; on a time-out the CTA raises an
//    abort flag, sets PA_DEVERR_TIMEOUT and unwinds, freeing its TMEM.
#include <cuda.h>
#include <math.h>

#include "pa_internal.h"
#include "pa_sm100.cuh"

namespace pa {
using namespace sm100;

constexpr int kPfRows = 128;            // MMA M: rows of a q tile
constexpr int kPfKeys = 128;            // keys per kv tile
constexpr int kPfThreads = 352;         // 8 softmax warps + K producer + MMA issuer + V producer
constexpr int kPfThreadsF8 = 384;       // e4m3 cache: + two warps widening K / V tiles to bf16
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpCvtK = 10, kWarpCvtV = 11;
constexpr int kWarpProducerV = 10;      // bf16 kernels: V tiles are issued by a warp of their own
constexpr int kPfMaxReqs = 2048;
constexpr int kHalf = 128 * 128;        // one 128-row x 128-byte swizzled half tile (16 KB): 64 of D columns
constexpr int kRing = 4;               // claimed work items handed from the producer to the other roles
// K_RAW / V_RAW: an e4m3 tile has landed (fp8 mode; K_FULL / V_FULL then
// mean "widened to bf16").  DRAIN: the MMA issuer's last commit on abort.
enum { Q_FULL, Q_EMPTY, K_FULL, K_FULL1, K_EMPTY, K_EMPTY1, V_FULL, V_FULL1, V_EMPTY, V_EMPTY1,
       SA_FULL, SB_FULL, PA_FULL, PB_FULL, OA_FINAL, OB_FINAL, OA_EMPTY, OB_EMPTY,
       K_RAW, K_RAW1, V_RAW, V_RAW1, DRAIN,
       ITEM_FULL, ITEM_EMPTY = ITEM_FULL + kRing, N_BARS = ITEM_EMPTY + kRing };
static_assert(N_BARS <= 32, "barrier area holds 32 barriers");
constexpr int kItemReaders = 1 + 8;     // the MMA warp and the eight softmax warps (+ 2 widening warps in fp8 mode)
constexpr int kStageBytes = 32 * 64;    // per softmax warp: 32 rows x 32 bf16 of the output
constexpr uint32_t kTmemCols = 512;     // S_A | S_B | O_A | O_B
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);   // Q (K-major) x K (K-major)

// Shared-memory layout for head dimension D (64 or 128): a q, K or V tile is
// D / 64 halves; Q tiles A and B, two K and two V stages, (fp8, D = 64) the
// e4m3 tiles as loaded, then barriers, the misc words, the item ring, the
// output staging and the plan's prefix array.  An e4m3 tile is 128 rows of D
// bytes at a 128-byte pitch (a tensor copy's shared-memory destination must be
// 128-byte aligned, so single-row boxes need that pitch): for D = 128 it lands
// in the upper half of the bf16 stage it is widened into, where e4m3 row r
// shares its 128 bytes with bf16 row r of half 1 and with nothing else.
template <int D, bool F8 = false>
struct PfLayout {
    static constexpr int kHalves = D / 64;
    static constexpr int kOffQA = 0;
    static constexpr int kOffQB = kHalves * kHalf;
    static constexpr int kOffK = 2 * kHalves * kHalf;   // 2 stages
    static constexpr int kOffV = 4 * kHalves * kHalf;   // 2 stages
    static constexpr int kRawPitch = 128;                // bytes per e4m3 row as loaded
    static constexpr int kRawBytes = kPfKeys * kRawPitch;   // one e4m3 tile
    static constexpr int kOffRaw = 6 * kHalves * kHalf;
    static constexpr int kRawArea = (F8 && D == 64) ? 4 * kRawBytes : 0;   // K stages 0, 1, then V
    static constexpr int kOffBar = kOffRaw + kRawArea;
    static constexpr int kOffMisc = kOffBar + 32 * 8;
    static constexpr int kOffRing = kOffMisc + 64;      // kRing work-item descriptions
    static constexpr int kOffStage = kOffMisc + 256;
    static constexpr int kOffPref = kOffStage + 8 * kStageBytes;
    // tensor-memory columns: S_A | S_B | O_A | O_B
    static constexpr uint32_t kColOA = 256, kColOB = 256 + D;
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);  // P (tensor memory) x V (MN-major)
};

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
    int32_t *queue;       // [0]: next item to claim, [done]: CTAs finished (kept at 0 between launches)
    int T, Hq, Hkv, G, TQ, R;
    int size, layer_row0, total_rows, req_rows, max_ctx;
    int early_meta;       // launched behind another kernel: plan before waiting for it
    __nv_bfloat16 *last_out;   // optional [R, Hq, D]: each request's last row of out
    float scale_log2;
    const float *k_scale;      // fp8 mode: the layer's per-kv-head K / V scales [Hkv]
    const float *v_scale;
    const __nv_bfloat16 *k_rows;   // bf16 K / V rows (row r at r * row_elems): the cp.async gather
    const __nv_bfloat16 *v_rows;
    int row_elems;
    uint64_t wait_ns;          // time limit of the pipeline waits
};

struct alignas(16) PfItem {
    int h, qs, q0, nqa, nqb, p, row, n_keys, ntiles;   // q0: first token of tile A; nqb == 0: no tile B
    int end;                                           // 1: no more items for this CTA
    int r, nr;                                         // request and its number of new tokens
};
static_assert(PfLayout<128>::kOffRing + kRing * (int)sizeof(PfItem) <= PfLayout<128>::kOffMisc + 256,
              "item ring fits the misc area");
static_assert(N_BARS <= 32, "barrier area holds 32 barriers");

// Widen one e4m3 tile (128 rows of D bytes at a 128-byte pitch at `src`) to bf16 in the
// 128-byte-swizzled K/V stage layout at `dst` (16-byte chunk c of row r at
// (c / 8) halves + r * 128 + ((c % 8) ^ (r % 8)) * 16).  D / 16 lanes share a
// row, each widening one 16-byte chunk into two; every row's bytes are read
// (and the warp synchronised) before any of its bf16 chunks is written, so
// the in-place D = 128 layout is safe.  Exact: e4m3 values are bf16 numbers.
template <int D>
__device__ __forceinline__ void widen_e4m3_tile(uint32_t src, uint32_t dst, int lane)
{
    constexpr int LPR = D / 16;     // lanes per row
    constexpr int RPP = 32 / LPR;   // rows per pass of the warp
    constexpr int U = 4;            // passes whose loads are in flight together
    const int rr = lane / LPR, j = lane % LPR;
#pragma unroll 1
    for (int r0 = 0; r0 < kPfKeys; r0 += RPP * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = ld_shared_v4(src + (uint32_t)((r0 + u * RPP + rr) * 128 + j * 16));
        __syncwarp();
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * RPP + rr;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t a = half ? v[u].z : v[u].x, b = half ? v[u].w : v[u].y;
                const int c = 2 * j + half;   // bf16 chunk: d = 8 c .. 8 c + 7
                st_shared_v4(dst + (uint32_t)((c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)),
                             e4m3x2_to_bf16x2(a), e4m3x2_to_bf16x2(a >> 16), e4m3x2_to_bf16x2(b),
                             e4m3x2_to_bf16x2(b >> 16));
            }
        }
        __syncwarp();
    }
}

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool DENSE>
__device__ __forceinline__ PfItem pf_item(const PrefillParams &p, const int *s_pref, int item)
{
    int lo = 0, hi = p.R;   // largest r with s_pref[r] <= item
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] <= item) lo = mid; else hi = mid;
    }
    const int r = lo;
    const int local = item - s_pref[r];
    const int pairs_r = (s_pref[r + 1] - s_pref[r]) / p.Hkv;
    const int jj = local / p.Hkv;
    PfItem I;
    I.h = local - jj * p.Hkv;
    const int jp = pairs_r - 1 - jj;            // later (heavier) pairs first
    I.qs = __ldg(p.qo_indptr + r);
    const int n_r = __ldg(p.qo_indptr + r + 1) - I.qs;
    const int L_r = DENSE ? n_r : __ldg(p.kv_indptr + r + 1) - __ldg(p.kv_indptr + r);
    I.p = L_r - n_r;
    I.r = r;
    I.nr = n_r;
    I.q0 = 2 * jp * p.TQ;
    I.nqa = min(p.TQ, n_r - I.q0);
    I.nqb = max(0, min(p.TQ, n_r - I.q0 - p.TQ));
    I.row = DENSE ? 0 : __ldg(p.req_pool_indices + r);
    I.n_keys = I.p + I.q0 + I.nqa + I.nqb;
    I.ntiles = (I.n_keys + kPfKeys - 1) / kPfKeys;
    return I;
}

template <int D, bool DENSE, bool LAST, bool F8>
__global__ void __launch_bounds__(F8 ? kPfThreadsF8 : kPfThreads, 1)
    paged_prefill_kernel(const __grid_constant__ PrefillParams p)
{
    using PL = PfLayout<D, F8>;
    constexpr int QH = PL::kHalves;   // 64-column halves of a q, K or V row
    constexpr int NT = F8 ? kPfThreadsF8 : kPfThreads;
    static_assert(!(F8 && (DENSE || LAST)), "the e4m3 mode is paged prefill only");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *sb = smem_raw + (base - raw);
    const uint32_t sQA = base + PL::kOffQA, sQB = base + PL::kOffQB, sK = base + PL::kOffK, sV = base + PL::kOffV;
    // fp8: where stage st's e4m3 K / V tile lands
    auto raw_tile = [&](bool isv, int st) -> uint32_t {
        if (D == 128) return (isv ? sV : sK) + st * QH * kHalf + kHalf;
        return base + PL::kOffRaw + ((isv ? 2 : 0) + st) * PL::kRawBytes;
    };
    volatile int *s_abort = reinterpret_cast<volatile int *>(sb + PL::kOffMisc);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sb + PL::kOffMisc + 4);
    int *s_wsum = reinterpret_cast<int *>(sb + PL::kOffMisc + 8);    // one int per warp (at most 12)
    PfItem *s_ring = reinterpret_cast<PfItem *>(sb + PL::kOffRing);
    int *s_pref = reinterpret_cast<int *>(sb + PL::kOffPref);
    auto bar = [&](int i) -> uint32_t { return base + PL::kOffBar + i * 8; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *err = p.err;

    if (tid == 0) {
        *s_abort = 0;
        for (int i = 0; i < N_BARS; ++i) {
            const bool softmax_arrive = i == PA_FULL || i == PB_FULL || i == OA_EMPTY || i == OB_EMPTY;
            const bool item_read = i >= ITEM_EMPTY && i < ITEM_EMPTY + kRing;
            mbar_init(bar(i), softmax_arrive ? 128u : item_read ? (uint32_t)(kItemReaders + (F8 ? 2 : 1)) : 1u);
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
    if (!p.early_meta) pdl_wait();

    // ---------------------------------------------------------- planning
    // q-tile pairs per request (0 for an invalid request), exclusive prefix of
    // pairs * Hkv; every thread scans a contiguous run of requests.  Error
    // bits are held until the wait for a preceding kernel.
    int pend_err = 0;
    {
        const int per = (p.R + NT - 1) / NT;
        const int r_lo = min(p.R, tid * per), r_hi = min(p.R, r_lo + per);
        auto pairs_of = [&](int r) -> int {
            const int qa = __ldg(p.qo_indptr + r), qb = __ldg(p.qo_indptr + r + 1);
            const int n_r = qb - qa;
            const int L_r = DENSE ? n_r : __ldg(p.kv_indptr + r + 1) - __ldg(p.kv_indptr + r);
            const int row = DENSE ? 0 : __ldg(p.req_pool_indices + r);
            if (n_r <= 0) {
                if (n_r < 0) pend_err |= PA_DEVERR_LEN;
                return 0;
            }
            if (qa < 0 || qb > p.T || L_r < n_r || L_r > p.max_ctx) {
                pend_err |= PA_DEVERR_LEN;
                return 0;
            }
            if (row < 0 || row >= p.req_rows) {
                pend_err |= PA_DEVERR_ROW;
                return 0;
            }
            return (n_r + 2 * p.TQ - 1) / (2 * p.TQ);
        };
        int run = 0;
        for (int r = r_lo; r < r_hi; ++r) run += pairs_of(r) * p.Hkv;
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
            excl += pairs_of(r) * p.Hkv;
        }
        if (tid == NT - 1) s_pref[p.R] = wbase + incl;
    }
    __syncthreads();
    // the plan read only index arrays; everything below waits for the
    // preceding kernel
    if (p.early_meta) pdl_wait();
    pdl_launch_dependents();
    if (pend_err) set_error(err, pend_err);
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int total_items = s_pref[p.R];
    const int G = p.G;

    if (warp == kWarpProducer || (!F8 && warp == kWarpProducerV)) {
        // ================================================== TMA producers
        // Items are claimed one at a time from a global counter, so a CTA that
        // drew short items takes more of them; each claim (and finally the
        // first index past the end) goes to the other roles through a ring.
        // bf16: warp 8 claims items and loads Q and the K tiles, warp 10 reads
        // the ring and loads the V tiles, so the two tiles' copies are issued
        // in parallel (each 16-row box is a TMA instruction of its own, and
        // one warp issuing both tiles had become the step's critical path).
        // fp8: warp 8 loads everything.
        const bool doK = warp == kWarpProducer;
        const bool doV = F8 || warp == kWarpProducerV;
        int kt = 0;
        int nq = 0, nk = 0, nv = 0;   // Q, K and V loads armed (for the drain on abort)
        bool ok = true;
        // every lane waits; the warp continues only if all saw the phase
        auto wait1 = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar(b), parity, s_abort, err, PA_DEVERR_TIMEOUT, p.wait_ns));
        };
        for (int it = 0; ok; ++it) {
            const int slot = it % kRing;
            PfItem I;
            if (doK) {
                if (it >= kRing && !wait1(ITEM_EMPTY + slot, (it / kRing - 1) & 1)) break;
                int item = 0;
                if (lane == 0) item = atomicAdd(p.queue, 1);
                item = __shfl_sync(0xffffffffu, item, 0);
                if (item < total_items) {
                    I = pf_item<DENSE>(p, s_pref, item);
                    I.end = 0;
                } else {
                    I.end = 1;
                }
                if (lane == 0) {
                    s_ring[slot] = I;
                    mbar_arrive(bar(ITEM_FULL + slot));
                }
            } else {
                // the V producer reads the claim like the other roles
                if (!wait1(ITEM_FULL + slot, (it / kRing) & 1)) break;
                I = s_ring[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + slot));
            }
            if (I.end) break;
            if (doK && it > 0 && !wait1(Q_EMPTY, (it - 1) & 1)) break;
            if (doK) ++nq;
            if (doK && lane == 0) {
                mbar_arrive_expect_tx(bar(Q_FULL), 2 * QH * kHalf);
#pragma unroll
                for (int hh = 0; hh < QH; ++hh) {
                    tma_load_3d(sQA + hh * kHalf, &p.tm_q, 64 * hh, I.h * G, I.qs + I.q0, bar(Q_FULL));
                    tma_load_3d(sQB + hh * kHalf, &p.tm_q, 64 * hh, I.h * G, I.qs + I.q0 + p.TQ, bar(Q_FULL));
                }
            }
            const int32_t *r2t = DENSE ? nullptr : p.req_to_token + (int64_t)I.row * p.max_ctx;
            // tensor-map row of slot / position 0: the layer's first slot, or
            // (dense) the request's first packed token
            const int row0 = DENSE ? I.qs : p.layer_row0;
            const int col0 = I.h * D;
            const int gi = lane >> 2, sub = lane & 3;
            // page-table entries of positions 128 t + 4 lane + e: the next
            // tile's are requested while this one's copies are issued, so a
            // tile's K copy waits for no table round trip (after the item's
            // first tile)
            int nraw[4];
            auto load_raw = [&](int tt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = tt * kPfKeys + 4 * lane + e;
                    nraw[e] = DENSE ? pos : ld_nc_ordered_s32_if(pos < I.n_keys, r2t + pos);
                }
            };
            if (I.ntiles > 0) load_raw(0);
            for (int t = 0; t < I.ntiles; ++t, ++kt) {
                const int st = kt & 1;
                const uint32_t ph_prev = ((kt >> 1) - 1) & 1;
                const int raw[4] = {nraw[0], nraw[1], nraw[2], nraw[3]};
                if (t + 1 < I.ntiles) load_raw(t + 1);
                // slots of positions k0 + 4*lane + e
                const int k0 = t * kPfKeys;
                int slot[4];
                bool okp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = k0 + 4 * lane + e;
                    okp[e] = pos < I.n_keys;
                    slot[e] = okp[e] ? raw[e] : -1;
                    if (okp[e] && !DENSE && (slot[e] < 0 || slot[e] >= p.size)) {   // skipped: zeros, flagged
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
                    if constexpr (F8) {
                        // e4m3 rows of D bytes at a 128-byte pitch: D = 128,
                        // one 16-row box per page group, else a box per row;
                        // D = 64 always a box per row (a 16-row box would pack
                        // the rows at a 64-byte pitch)
                        if (D == 128 && (g_contig || g_empty)) {
                            if (sub == 0)
                                tma_load_2d(dst + gi * 16 * 128, m16, col0, g_empty ? p.total_rows : row0 + s0, b);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int rr = 16 * gi + 4 * sub + e;
                                tma_load_2d(dst + rr * 128, m1, col0, okp[e] ? row0 + slot[e] : p.total_rows, b);
                            }
                        }
                        return;
                    }
                    if (g_contig || g_empty) {
                        if (sub == 0) {
                            const int row = g_empty ? p.total_rows : row0 + s0;
#pragma unroll
                            for (int hh = 0; hh < QH; ++hh)
                                tma_load_2d(dst + hh * kHalf + gi * 16 * 128, m16, col0 + 64 * hh, row, b);
                        }
                    }   // other groups: gathered by cp.async before the barrier arrival
                };
                // bf16: the tile lands in its stage; fp8: its e4m3 bytes land
                // for the widening warp
                const int kb = F8 ? K_RAW : K_FULL, vb = F8 ? V_RAW : V_FULL;
                constexpr uint32_t kTileBytes = F8 ? (uint32_t)(kPfKeys * D) : (uint32_t)(QH * kHalf);   // bytes landing
                // bf16 groups not on one page (page sizes below 16, ragged
                // ends) are gathered by cp.async, K and V together: the
                // group's 4 lanes copy 64 contiguous bytes of a row per
                // instruction into the swizzled tile, the producer waits for
                // its own copies and fences them for the tensor core's async
                // proxy before arming the barriers.  Tiles whose groups all
                // move as TMA boxes (page 16) skip this entirely.
                const bool gathered = !F8 && !(g_contig || g_empty);
                const bool any_gathered = __any_sync(0xffffffffu, gathered);
                uint32_t tile_bytes = kTileBytes;
                if (any_gathered)
                    tile_bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, sub == 0 && (g_contig || g_empty))) * 16u *
                                 (uint32_t)(QH * 128);
                auto gather = [&](const __nv_bfloat16 *rows, uint32_t dst) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int src_lane = (lane & ~3) + (i >> 2);
                        const int sl = __shfl_sync(0xffffffffu, slot[i & 3], src_lane);
                        const bool ok_row = __shfl_sync(0xffffffffu, okp[i & 3], src_lane);
                        if (!gathered) continue;
                        const int rr = 16 * gi + i;
                        const __nv_bfloat16 *src = rows + (int64_t)(row0 + (ok_row ? sl : 0)) * p.row_elems + col0;
#pragma unroll
                        for (int q4 = 0; q4 < 2 * QH; ++q4) {
                            const int ch = q4 * 4 + sub;            // 16-byte chunk of the row (8 per 64 columns)
                            const int hh = ch >> 3, c = ch & 7;
                            cp_async_16(dst + hh * kHalf + rr * 128 + ((c ^ (rr & 7)) << 4), src + ch * 8,
                                        ok_row ? 16 : 0);
                        }
                    }
                };
                if (doK) {
                    if (kt >= 2 && !wait1(K_EMPTY + st, ph_prev)) {
                        ok = false;
                        break;
                    }
                    if (any_gathered) {
                        gather(p.k_rows, sK + st * QH * kHalf);
                        cp_async_wait_all();
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    ++nk;
                    if (lane == 0) mbar_arrive_expect_tx(bar(kb + st), tile_bytes);
                    __syncwarp();
                    issue(&p.tm_k16, &p.tm_k1, F8 ? raw_tile(false, st) : sK + st * QH * kHalf, bar(kb + st));
                }
                if (doV) {
                    if (kt >= 2 && !wait1(V_EMPTY + st, ph_prev)) {
                        ok = false;
                        break;
                    }
                    if (any_gathered) {
                        gather(p.v_rows, sV + st * QH * kHalf);
                        cp_async_wait_all();
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    ++nv;
                    if (lane == 0) mbar_arrive_expect_tx(bar(vb + st), tile_bytes);
                    __syncwarp();
                    issue(&p.tm_v16, &p.tm_v1, F8 ? raw_tile(true, st) : sV + st * QH * kHalf, bar(vb + st));
                }
            }
        }
        if (*s_abort && lane == 0) {
            // aborted: every copy this warp issued lands before the CTA's
            // shared memory goes away (each barrier's last armed phase)
            if (nq > 0) mbar_drain(bar(Q_FULL), (nq - 1) & 1);
            const int kb = F8 ? K_RAW : K_FULL, vb = F8 ? V_RAW : V_FULL;
            for (int st = 0; st < 2; ++st) {
                const int ck = (nk - st + 1) / 2, cv = (nv - st + 1) / 2;   // arms of stage st
                if (ck > 0) mbar_drain(bar(kb + st), (ck - 1) & 1);
                if (cv > 0) mbar_drain(bar(vb + st), (cv - 1) & 1);
            }
        }
        __syncwarp();
    } else if (F8 && (warp == kWarpCvtK || warp == kWarpCvtV)) {
        // =========================================== e4m3 -> bf16 widening
        // One warp per operand: each e4m3 tile that lands is widened into its
        // bf16 stage, then handed to the MMA issuer (generic-proxy writes made
        // visible to the tensor core's async proxy first).
        const bool isv = warp == kWarpCvtV;
        int kt = 0;
        bool ok = true;
        auto wait1 = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar(b), parity, s_abort, err, PA_DEVERR_TIMEOUT, p.wait_ns));
        };
        for (int n = 0; ok; ++n) {
            if (!wait1(ITEM_FULL + n % kRing, (n / kRing) & 1)) break;
            const PfItem I = s_ring[n % kRing];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + n % kRing));
            if (I.end) break;
            for (int t = 0; t < I.ntiles; ++t, ++kt) {
                const int st = kt & 1;
                if (!wait1((isv ? V_RAW : K_RAW) + st, (kt >> 1) & 1)) {
                    ok = false;
                    break;
                }
                widen_e4m3_tile<D>(raw_tile(isv, st), (isv ? sV : sK) + st * QH * kHalf, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar((isv ? V_FULL : K_FULL) + st));
            }
        }
    } else if (warp == kWarpMma) {
        // ================================================== MMA issuer
        // The whole warp runs the loop and waits (uniform control flow); one
        // elected lane issues the MMAs and commits.  A tcgen05.mma is accepted
        // only about one MMA ahead of the tensor core, so each wait between
        // groups idles the pipe for its latency: every iteration waits at two
        // points only, each testing all the barriers it needs at once.
        int kt = 0, ia = 0, ib = 0, ta = 0, tb = 0;   // tiles / items seen by tile A and B
        bool ok = true;
        auto waitn = [&](auto const &bars, auto const &pars) -> bool {
            ok = __all_sync(0xffffffffu, mbar_wait_all(bars, pars, s_abort, err, PA_DEVERR_TIMEOUT, p.wait_ns));
            return ok;
        };
        auto qk = [&](uint32_t sQ, int st, uint32_t d_col) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = smem_desc_sw128(sQ + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                const uint64_t b = smem_desc_sw128(sK + st * QH * kHalf + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                umma_ss(tmem + d_col, a, b, kIdescS, kk > 0 ? 1u : 0u);
            }
        };
        auto pv = [&](uint32_t p_col, uint32_t o_col, int st, bool first) {
#pragma unroll
            for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                const uint64_t b = smem_desc_sw128(sV + st * QH * kHalf + kk * 2048, kHalf, 1024);
                umma_ts(tmem + o_col, tmem + p_col + kk * 8, b, PL::kIdescPV, (kk > 0 || !first) ? 1u : 0u);
            }
        };
        for (int n = 0; ok; ++n) {
            const int slot = n % kRing;
            {
                const uint32_t b1[1] = {bar(ITEM_FULL + slot)}, p1[1] = {(uint32_t)(n / kRing) & 1u};
                if (!waitn(b1, p1)) break;
            }
            const PfItem I = s_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + slot));
            if (I.end) break;
            const bool hasB = I.nqb > 0;
            // S_A(0), S_B(0)
            {
                const uint32_t b2[2] = {bar(Q_FULL), bar(K_FULL + (kt & 1))};
                const uint32_t p2[2] = {(uint32_t)ia & 1u, (uint32_t)(kt >> 1) & 1u};
                if (!waitn(b2, p2)) break;
            }
            tc_fence_after();
            if (elect_one()) {
                qk(sQA, kt & 1, 0);
                umma_commit(bar(SA_FULL));
                if (hasB) {
                    qk(sQB, kt & 1, 128);
                    umma_commit(bar(SB_FULL));
                }
                umma_commit(bar(K_EMPTY + (kt & 1)));
                if (I.ntiles == 1) umma_commit(bar(Q_EMPTY));   // the item's last QK^T: Q may be refilled
            }
            __syncwarp();
            for (int t = 0; t < I.ntiles; ++t, ++kt) {
                const int st = kt & 1, st1 = (kt + 1) & 1;
                const bool more = t + 1 < I.ntiles;
                // wait point 1: P_A(t), V(t), K(t+1), and O_A free at an item's first tile
                {
                    const uint32_t b4[4] = {bar(PA_FULL), bar(V_FULL + st), bar(more ? K_FULL + st1 : V_FULL + st),
                                            bar(t == 0 && ia > 0 ? OA_EMPTY : V_FULL + st)};
                    const uint32_t p4[4] = {(uint32_t)ta & 1u, (uint32_t)(kt >> 1) & 1u,
                                            (uint32_t)(more ? (kt + 1) >> 1 : kt >> 1) & 1u,
                                            (uint32_t)(t == 0 && ia > 0 ? ia - 1 : kt >> 1) & 1u};
                    if (!waitn(b4, p4)) break;
                }
                tc_fence_after();
                if (elect_one()) {
                    pv(0, PL::kColOA, st, t == 0);                            // PV_A(t)
                    if (!more) umma_commit(bar(OA_FINAL));
                    if (more) {
                        qk(sQA, st1, 0);                                      // S_A(t+1)
                        umma_commit(bar(SA_FULL));
                    }
                }
                __syncwarp();
                ++ta;
                // wait point 2: P_B(t), and O_B free at an item's first tile
                if (hasB) {
                    const uint32_t b2[2] = {bar(PB_FULL), bar(t == 0 && ib > 0 ? OB_EMPTY : PB_FULL)};
                    const uint32_t p2[2] = {(uint32_t)tb & 1u, (uint32_t)(t == 0 && ib > 0 ? ib - 1 : tb) & 1u};
                    if (!waitn(b2, p2)) break;
                    tc_fence_after();
                }
                if (elect_one()) {
                    if (hasB) {
                        pv(128, PL::kColOB, st, t == 0);                      // PV_B(t)
                        if (!more) umma_commit(bar(OB_FINAL));
                    }
                    umma_commit(bar(V_EMPTY + st));
                    if (more) {
                        if (hasB) {
                            qk(sQB, st1, 128);                                // S_B(t+1)
                            umma_commit(bar(SB_FULL));
                        }
                        umma_commit(bar(K_EMPTY + st1));
                        if (t + 2 == I.ntiles) umma_commit(bar(Q_EMPTY));   // last QK^T of the item issued
                    }
                }
                __syncwarp();
                if (hasB) ++tb;
            }
            ++ia;
            if (hasB) ++ib;
        }
        if (*s_abort) {
            // aborted: one more commit, which arrives once every MMA this
            // lane issued has completed, before tensor memory is freed
            if (elect_one()) umma_commit(bar(DRAIN));
            __syncwarp();
            mbar_drain(bar(DRAIN), 0);
            __syncwarp();
        }
    } else {
        // ======================= softmax + epilogue: warpgroup X owns tile X
        const int X = warp >> 2;                  // 0: tile A, 1: tile B
        const int row = tid & 127;                // TMEM lane = row of the tile
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + X * 128;     // S_X, later P_X (bf16 pairs)
        const uint32_t o_addr = tmem + lane_base + (X ? PL::kColOB : PL::kColOA);
        const int b_s_full = X ? SB_FULL : SA_FULL, b_p_full = X ? PB_FULL : PA_FULL;
        const int b_o_final = X ? OB_FINAL : OA_FINAL, b_o_empty = X ? OB_EMPTY : OA_EMPTY;
        float sl2 = p.scale_log2;
        int tx = 0, ix = 0;       // tiles and items this warpgroup has processed
        bool ok = true;
        for (int n = 0; ok; ++n) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar(ITEM_FULL + n % kRing), (n / kRing) & 1, s_abort, err,
                                                   PA_DEVERR_TIMEOUT, p.wait_ns)))
                break;
            const PfItem I = s_ring[n % kRing];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + n % kRing));
            if (I.end) break;
            if (p.wait_ns == 0) {
                // a wait limit of 0: give up at the first item, as a timed-out
                // wait would; the other roles then find their next phase
                // incomplete and see the abort flag
                *s_abort = 1;
                set_error(err, PA_DEVERR_TIMEOUT);
                break;
            }
            const int nq = X ? I.nqb : I.nqa;
            if (nq <= 0) continue;                // no tile B in this pair
            const int q0 = I.q0 + X * p.TQ;
            if constexpr (F8) sl2 = p.scale_log2 * __ldg(p.k_scale + I.h);   // the head's K scale joins the softmax scale
            const int tok = row / G;              // token of this row within the tile
            const int qpos = I.p + q0 + tok;      // its position in the request
            float m_run = -INFINITY, l_run = 0.f;
            for (int t = 0; t < I.ntiles; ++t, ++tx) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(bar(b_s_full), tx & 1, s_abort, err, PA_DEVERR_TIMEOUT, p.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int limit = qpos - t * kPfKeys;    // columns <= limit are visible
                // the whole row of S in registers: four loads, one wait
                uint32_t r[128];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    tmem_ld32(s_addr + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[ch * 32]));
                tmem_wait_ld();
                const bool diag = limit < kPfKeys - 1;
                if (diag) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > limit) r[c] = __float_as_uint(-INFINITY);
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 4) {
                    mx0 = fmaxf(mx0, __uint_as_float(r[c]));
                    mx1 = fmaxf(mx1, __uint_as_float(r[c + 1]));
                    mx2 = fmaxf(mx2, __uint_as_float(r[c + 2]));
                    mx3 = fmaxf(mx3, __uint_as_float(r[c + 3]));
                }
                const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                float m_new = m_run;
                bool rescale = false;
                if (mx > m_run && (m_run == -INFINITY || (mx - m_run) * sl2 > 8.f)) {
                    rescale = m_run != -INFINITY;
                    m_new = mx;
                }
                const float alpha = rescale ? ex2f((m_run - m_new) * sl2) : 1.f;
                m_run = m_new;
                const float mb = m_new == -INFINITY ? 0.f : m_new * sl2;
                // P = exp2(s*scale - m) (masked entries are -inf -> 0), written
                // back as bf16 pairs over the first 64 columns of S_X
                // column pairs in packed two-float FMAs and adds (each lane an
                // IEEE round-to-nearest op: the same values as scalar code)
                const uint64_t sl2x2 = f32x2_pack(sl2, sl2), nmb2 = f32x2_pack(-mb, -mb);
                uint64_t sum2 = f32x2_pack(0.f, 0.f);   // even and odd columns' sums
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const uint64_t x = fma_f32x2(f32x2_pack(__uint_as_float(r[hh * 64 + c]),
                                                                __uint_as_float(r[hh * 64 + c + 1])),
                                                     sl2x2, nmb2);
                        const float v0 = ex2f(f32x2_lo(x)), v1 = ex2f(f32x2_hi(x));
                        const uint64_t v2 = f32x2_pack(v0, v1);
                        sum2 = add_f32x2(sum2, v2);
                        pk[c / 2] = pack_bf16x2(v0, v1);
                    }
                    tmem_st32(s_addr + hh * 32, pk);
                }
                l_run = l_run * alpha + (f32x2_lo(sum2) + f32x2_hi(sum2));
                // O_X is stable here: S_X(t) completing implies PV_X(t-1) completed
                if (t > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + ch * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(o_addr + ch * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(b_p_full));
            }
            if (!ok) break;
            // ------------------------------------------------ epilogue
            if (!__all_sync(0xffffffffu, mbar_wait(bar(b_o_final), ix & 1, s_abort, err, PA_DEVERR_TIMEOUT, p.wait_ns)))
                break;
            tc_fence_after();
            uint32_t o[D];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch)
                tmem_ld32(o_addr + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[ch * 32]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(b_o_empty));          // O_X is in registers: the next item may overwrite it
            // fp8: the head's V scale multiplies the normalised output
            const float inv_l = l_run > 0.f ? (F8 ? __ldg(p.v_scale + I.h) : 1.f) / l_run : 0.f;
            uint32_t ob[D / 2];                   // O / l as bf16 pairs
#pragma unroll
            for (int c = 0; c < D / 2; ++c)
                ob[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l, __uint_as_float(o[2 * c + 1]) * inv_l);
            // 32 columns at a time through this warp's staging buffer (row
            // lane, 16-byte chunks XOR-swizzled by row so neither side
            // conflicts), then out with four lanes on 64 contiguous bytes
            const uint32_t stg = base + PL::kOffStage + warp * kStageBytes;
            const int rr0 = lane >> 2, cc = lane & 3;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t *v = &ob[ch * 16 + c * 4];
                    st_shared_v4(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), v[0], v[1], v[2], v[3]);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = 8 * i + rr0;                 // staged row = tile row (warp & 3) * 32 + rr
                    const uint4 v = ld_shared_v4(stg + rr * 64 + ((cc ^ ((rr >> 1) & 3)) << 4));
                    const int trow = (warp & 3) * 32 + rr;
                    const int ttok = trow / G;
                    if (ttok < nq) {
                        __nv_bfloat16 *dst = p.out + ((int64_t)(I.qs + q0 + ttok) * p.Hq + I.h * G + (trow - ttok * G)) * D;
                        *reinterpret_cast<uint4 *>(dst + ch * 32 + cc * 8) = v;
                        if (LAST && q0 + ttok == I.nr - 1) {   // the request's last row, gathered
                            __nv_bfloat16 *lst = p.last_out + ((int64_t)I.r * p.Hq + I.h * G + (trow - ttok * G)) * D;
                            *reinterpret_cast<uint4 *>(lst + ch * 32 + cc * 8) = v;
                        }
                    }
                }
                __syncwarp();
            }
            ++ix;
        }
    }

    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // the last CTA to finish returns the queue to zero for the next launch;
    // every CTA's claims precede its increment here
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(p.queue + (kPrefillDoneWord - kPrefillQueueWord), 1) == (int)gridDim.x - 1) {
            atomicExch(p.queue, 0);
            atomicExch(p.queue + (kPrefillDoneWord - kPrefillQueueWord), 0);
        }
    }
}

}  // namespace pa

using namespace pa;

namespace pa {

template <int D, bool DENSE, bool LAST, bool F8 = false>
static pa_status launch_prefill(const PrefillParams &prm, cudaStream_t st)
{
    auto kern = paged_prefill_kernel<D, DENSE, LAST, F8>;
    const size_t smem = (size_t)PfLayout<D, F8>::kOffPref + (size_t)(prm.R + 1) * 4 + 1024;
    if (!ensure_dynamic_smem(reinterpret_cast<const void *>(kern), smem)) return PA_ERR_CUDA;
    if (launch_kernel(kern, dim3(num_sms()), dim3(F8 ? kPfThreadsF8 : kPfThreads), smem, st, prm) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
static_assert(PfLayout<128>::kOffPref + (kPfMaxReqs + 1) * 4 + 1024 <= 232448, "bf16 prefill smem");
static_assert(PfLayout<128, true>::kOffPref + (kPfMaxReqs + 1) * 4 + 1024 <= 232448, "fp8 prefill smem");
static_assert(PfLayout<64, true>::kOffPref + (kPfMaxReqs + 1) * 4 + 1024 <= 232448, "fp8 prefill smem, D = 64");

// Shared host path of the paged and dense entry points.  Paged: K/V rows are
// slots of layer `layer_id` of [n_layers, size, Hkv, D] buffers, reached
// through req_to_token (bf16, or e4m3 bytes with per-kv-head scales when
// k_scale != NULL).  Dense: K/V are the packed new tokens' rows
// [n_tokens, Hkv, D] (no prefix: kv length = query length).
static pa_status prefill_call(const void *q, int n_tokens, int n_q_heads, const void *k_rows, const void *v_rows,
                              int n_kv_heads, int D, int64_t total_rows, int layer_row0, int size,
                              const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                              const int32_t *req_to_token, int req_rows, int max_ctx,
                              const int32_t *req_pool_indices, float scale, void *workspace, size_t workspace_bytes,
                              void *out, void *last_out, bool dense, cudaStream_t st,
                              const float *k_scale = nullptr, const float *v_scale = nullptr)
{
    PrefillParams prm;
    memset(&prm, 0, sizeof prm);
    const bool f8 = k_scale != nullptr;
    const int G = n_q_heads / n_kv_heads;
    const int TQ = kPfRows / G;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n_q_heads, (cuuint64_t)n_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)n_q_heads * D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
        if (!encode_tmap_bf16(&prm.tm_q, q, 3, dims, strides, box)) return PA_ERR_CUDA;
    }
    if (f8) {
        // e4m3 rows: D bytes per (slot, kv head), plain boxes of 16 rows or 1
        const cuuint64_t dims[2] = {(cuuint64_t)n_kv_heads * D, (cuuint64_t)total_rows};
        const cuuint64_t strides[1] = {(cuuint64_t)n_kv_heads * D};
        const cuuint32_t box16[2] = {(cuuint32_t)D, 16}, box1[2] = {(cuuint32_t)D, 1};
        if (!encode_tmap_u8(&prm.tm_k16, k_rows, 2, dims, strides, box16) ||
            !encode_tmap_u8(&prm.tm_k1, k_rows, 2, dims, strides, box1) ||
            !encode_tmap_u8(&prm.tm_v16, v_rows, 2, dims, strides, box16) ||
            !encode_tmap_u8(&prm.tm_v1, v_rows, 2, dims, strides, box1))
            return PA_ERR_CUDA;
    } else {
        const cuuint64_t dims[2] = {(cuuint64_t)n_kv_heads * D, (cuuint64_t)total_rows};
        const cuuint64_t strides[1] = {(cuuint64_t)n_kv_heads * D * 2};
        const cuuint32_t box16[2] = {64, 16}, box1[2] = {64, 1};
        if (!encode_tmap_bf16(&prm.tm_k16, k_rows, 2, dims, strides, box16) ||
            !encode_tmap_bf16(&prm.tm_k1, k_rows, 2, dims, strides, box1) ||
            !encode_tmap_bf16(&prm.tm_v16, v_rows, 2, dims, strides, box16) ||
            !encode_tmap_bf16(&prm.tm_v1, v_rows, 2, dims, strides, box1))
            return PA_ERR_CUDA;
    }
    prm.qo_indptr = qo_indptr;
    prm.kv_indptr = kv_indptr;
    prm.req_to_token = req_to_token;
    prm.req_pool_indices = req_pool_indices;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.last_out = static_cast<__nv_bfloat16 *>(last_out);
    prm.err = static_cast<int32_t *>(workspace);
    prm.queue = static_cast<int32_t *>(workspace) + kPrefillQueueWord;
    prm.T = n_tokens;
    prm.Hq = n_q_heads;
    prm.Hkv = n_kv_heads;
    prm.G = G;
    prm.TQ = TQ;
    prm.R = n_reqs;
    prm.size = size;
    prm.layer_row0 = layer_row0;
    prm.total_rows = (int)total_rows;
    prm.req_rows = req_rows;
    prm.max_ctx = max_ctx;
    prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
    prm.early_meta = early_metadata();
    prm.k_scale = k_scale;
    prm.v_scale = v_scale;
    prm.k_rows = static_cast<const __nv_bfloat16 *>(k_rows);
    prm.v_rows = static_cast<const __nv_bfloat16 *>(v_rows);
    prm.row_elems = n_kv_heads * D;
    prm.wait_ns = wait_limit_ns();

    if (f8) return D == 64 ? launch_prefill<64, false, false, true>(prm, st) : launch_prefill<128, false, false, true>(prm, st);
    if (D == 64) {
        if (dense) return last_out ? launch_prefill<64, true, true>(prm, st) : launch_prefill<64, true, false>(prm, st);
        return last_out ? launch_prefill<64, false, true>(prm, st) : launch_prefill<64, false, false>(prm, st);
    }
    if (dense) return last_out ? launch_prefill<128, true, true>(prm, st) : launch_prefill<128, true, false>(prm, st);
    return last_out ? launch_prefill<128, false, true>(prm, st) : launch_prefill<128, false, false>(prm, st);
}

// Host checks shared by the paged entry points (bf16 or e4m3 cache).
static pa_status check_paged(const void *q, int n_tokens, int n_q_heads, const void *k_buf, const void *v_buf,
                             pa_kv_shape s, int layer_id, const int32_t *qo_indptr, const int32_t *kv_indptr,
                             int n_reqs, const int32_t *req_to_token, int req_rows, int max_ctx,
                             const int32_t *req_pool_indices, void *workspace, size_t workspace_bytes, void *out,
                             void *last_out)
{
    if (n_tokens < 0 || n_reqs < 0 || n_reqs > kPfMaxReqs || n_q_heads <= 0 || s.n_layers <= 0 || s.size <= 0 ||
        s.n_kv_heads <= 0 || req_rows <= 0 || max_ctx <= 0)
        return PA_ERR_SHAPE;
    if (layer_id < 0 || layer_id >= s.n_layers) return PA_ERR_SHAPE;
    if (n_q_heads % s.n_kv_heads != 0) return PA_ERR_SHAPE;
    const int G = n_q_heads / s.n_kv_heads;
    if ((s.head_dim != 64 && s.head_dim != 128) || (G != 1 && G != 2 && G != 4 && G != 8 && G != 16))
        return PA_ERR_UNSUPPORTED;
    if ((int64_t)s.n_layers * s.size >= (int64_t)INT32_MAX - 16) return PA_ERR_SHAPE;
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    if (workspace_bytes < pa_prefill_workspace_bytes()) return PA_ERR_WORKSPACE;
    if (n_tokens == 0 || n_reqs == 0) return PA_OK;
    if (!q || !k_buf || !v_buf || !qo_indptr || !kv_indptr || !req_to_token || !req_pool_indices || !out)
        return PA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_buf) || !aligned16(v_buf) || !aligned16(out) || !aligned4(qo_indptr) ||
        !aligned4(kv_indptr) || !aligned4(req_to_token) || !aligned4(req_pool_indices) ||
        (last_out && !aligned16(last_out)))
        return PA_ERR_ALIGN;
    return PA_OK;
}

static pa_status paged_call(const void *q, int n_tokens, int n_q_heads, const void *k_buf, const void *v_buf,
                            pa_kv_shape s, int layer_id, const int32_t *qo_indptr, const int32_t *kv_indptr,
                            int n_reqs, const int32_t *req_to_token, int req_rows, int max_ctx,
                            const int32_t *req_pool_indices, float scale, void *workspace, size_t workspace_bytes,
                            void *out, void *last_out, cudaStream_t st)
{
    const pa_status rc = check_paged(q, n_tokens, n_q_heads, k_buf, v_buf, s, layer_id, qo_indptr, kv_indptr, n_reqs,
                                     req_to_token, req_rows, max_ctx, req_pool_indices, workspace, workspace_bytes,
                                     out, last_out);
    if (rc != PA_OK || n_tokens == 0 || n_reqs == 0) return rc;
    return prefill_call(q, n_tokens, n_q_heads, k_buf, v_buf, s.n_kv_heads, s.head_dim, (int64_t)s.n_layers * s.size,
                        layer_id * s.size, s.size, qo_indptr, kv_indptr, n_reqs, req_to_token, req_rows, max_ctx,
                        req_pool_indices, scale, workspace, workspace_bytes, out, last_out, false, st);
}

}  // namespace pa

extern "C" pa_status pa_paged_prefill_attn(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                           const void *v_buf, pa_kv_shape s, int layer_id,
                                           const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                           const int32_t *req_to_token, int req_rows, int max_ctx,
                                           const int32_t *req_pool_indices, float scale, void *workspace,
                                           size_t workspace_bytes, void *out, cudaStream_t st)
{
    return paged_call(q, n_tokens, n_q_heads, k_buf, v_buf, s, layer_id, qo_indptr, kv_indptr, n_reqs, req_to_token,
                      req_rows, max_ctx, req_pool_indices, scale, workspace, workspace_bytes, out, nullptr, st);
}

extern "C" pa_status pa_paged_prefill_attn_last(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                                const void *v_buf, pa_kv_shape s, int layer_id,
                                                const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                                const int32_t *req_to_token, int req_rows, int max_ctx,
                                                const int32_t *req_pool_indices, float scale, void *workspace,
                                                size_t workspace_bytes, void *out, void *last_out, cudaStream_t st)
{
    if (!last_out && n_tokens > 0 && n_reqs > 0) return PA_ERR_NULL;
    return paged_call(q, n_tokens, n_q_heads, k_buf, v_buf, s, layer_id, qo_indptr, kv_indptr, n_reqs, req_to_token,
                      req_rows, max_ctx, req_pool_indices, scale, workspace, workspace_bytes, out, last_out, st);
}

extern "C" pa_status pa_paged_prefill_attn_fp8(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                               const void *v_buf, pa_kv_shape s, int layer_id,
                                               const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                               const int32_t *req_to_token, int req_rows, int max_ctx,
                                               const int32_t *req_pool_indices, float scale, const float *k_scale,
                                               const float *v_scale, void *workspace, size_t workspace_bytes,
                                               void *out, cudaStream_t st)
{
    pa_status rc = check_paged(q, n_tokens, n_q_heads, k_buf, v_buf, s, layer_id, qo_indptr, kv_indptr, n_reqs,
                               req_to_token, req_rows, max_ctx, req_pool_indices, workspace, workspace_bytes, out,
                               nullptr);
    if (rc != PA_OK || n_tokens == 0 || n_reqs == 0) return rc;
    if (!k_scale || !v_scale) return PA_ERR_NULL;
    if (!aligned4(k_scale) || !aligned4(v_scale)) return PA_ERR_ALIGN;
    const int64_t sc_off = (int64_t)layer_id * s.n_kv_heads;   // the layer's [Hkv] scales
    return prefill_call(q, n_tokens, n_q_heads, k_buf, v_buf, s.n_kv_heads, s.head_dim, (int64_t)s.n_layers * s.size,
                        layer_id * s.size, s.size, qo_indptr, kv_indptr, n_reqs, req_to_token, req_rows, max_ctx,
                        req_pool_indices, scale, workspace, workspace_bytes, out, nullptr, false, st,
                        k_scale + sc_off, v_scale + sc_off);
}

extern "C" pa_status pa_dense_prefill_attn(const void *q, int n_tokens, int n_q_heads, const void *k, const void *v,
                                           int n_kv_heads, int head_dim, const int32_t *qo_indptr, int n_reqs,
                                           float scale, void *workspace, size_t workspace_bytes, void *out,
                                           void *last_out, cudaStream_t st)
{
    if (n_tokens < 0 || n_reqs < 0 || n_reqs > kPfMaxReqs || n_q_heads <= 0 || n_kv_heads <= 0)
        return PA_ERR_SHAPE;
    if (n_q_heads % n_kv_heads != 0) return PA_ERR_SHAPE;
    const int G = n_q_heads / n_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (G != 1 && G != 2 && G != 4 && G != 8 && G != 16))
        return PA_ERR_UNSUPPORTED;
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    if (workspace_bytes < pa_prefill_workspace_bytes()) return PA_ERR_WORKSPACE;
    if (n_tokens == 0 || n_reqs == 0) return PA_OK;
    if (!q || !k || !v || !qo_indptr || !out) return PA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(qo_indptr) ||
        (last_out && !aligned16(last_out)))
        return PA_ERR_ALIGN;
    // qo_indptr doubles as kv_indptr (kv length = query length); max_ctx bounds a request by the pack
    return prefill_call(q, n_tokens, n_q_heads, k, v, n_kv_heads, head_dim, n_tokens, 0, n_tokens, qo_indptr, qo_indptr,
                        n_reqs, nullptr, 1, n_tokens, nullptr, scale, workspace, workspace_bytes, out, last_out, true,
                        st);
}

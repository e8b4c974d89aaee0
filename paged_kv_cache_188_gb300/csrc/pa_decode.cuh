#pragma once
// pa_decode.cuh -- packed GQA split-KV decode attention over the paged cache:
// the kernel and its launch, shared by pa_decode.cu (decode attention, and
// the allocation-free entry point) and pa_decode_step.cu (the fused step).
//
// What it computes (AstrAI commit 398e8a3, tests/inference/test_cache.py:
// packed decode with int32 req_to_token / req_pool_indices / seq_lens and
// workspace-owned split partials decode_o_part / decode_ml_part; commit
// e58a728, docs/developer/architecture.md: decode reads K/V via req_to_token):
// for request b and query head hq, softmax(scale * q K^T) V over the request's
// seq_lens[b] cached tokens, K/V rows gathered through req_to_token.
//
// How (one kernel, one persistent CTA of 8 warps per SM):
//  * Planning on the device, redundantly in every CTA: sum of seq_lens ->
//    per request the split count s_b (<= max_splits): splits of a common
//    length (at most 2048 tokens), or -- when batch x Hkv is at most half the
//    grid and that length would pass 2048 -- counts proportional to the
//    lengths that fill the grid in one wave; a prefix sum over s_b * Hkv
//    enumerates work items (b, split, kv head).  The grid never depends on
//    device lengths, so a captured graph stays valid.
//  * The CTA's 8 warps share each item: 16-token tile i of the item belongs to
//    warp i % 8.  Every warp streams its own tiles -- K and V rows of one kv
//    head, D*2 bytes each wherever the page table puts them -- through a
//    private ring of S shared-memory stages with 16-byte cp.async copies (D/8
//    lanes per row, so an instruction reads whole rows).  The ring runs across
//    item boundaries: while a warp computes its last tiles of one item it is
//    already loading its first tiles of the next.  Page-table entries of the
//    next tile to load are prefetched into registers one tile ahead.  Rows are
//    stored with a 16-byte-chunk XOR swizzle so ldmatrix is conflict free.
//    (A gather microbenchmark on this GPU: 8 warps x 3 cp.async stages per SM
//    read these rows at 7.2 TB/s; a single TMA-issuing thread per SM tops out
//    near 4.4 TB/s.)
//  * Per tile, warp-level bf16 MMAs (m16n8k16) with tokens as the M dimension:
//      S^T[tok, head] = K[tok, :] . Q[head, :]       (Q^T held in registers)
//      online softmax per head column, log2 domain (exp2)
//      O^T[d, head]  += V^T[d, tok] . P^T[tok, head]   (P^T by movmatrix)
//    so K/V bytes are read once for all G heads of the kv head.
//  * At the end of an item the warps' states merge in shared memory; a
//    request with one split writes bf16 output directly, otherwise the item
//    writes fp32 (o, m, l) partials and the CTA that completes a (request, kv
//    head) -- an integer atomic ticket, no waiting -- merges all splits in
//    split order (deterministic), writes bf16 and re-arms the ticket to zero.
//    The ticket is an acquire-release atomic, so the merging CTA needs no
//    separate fence; the first 20 splits' partials (8 when G > 8) travel with
//    the (m, l) pairs, the weights are warp-parallel, further splits follow
//    in batches of the same size.
//  * Fused decode step (FUSED = true, pa_decode_step): q is rotated (RoPE)
//    in registers as it is loaded.  The warp that computes the last tile of
//    a (request, kv head)'s last split loads that head's new K and V rows
//    with q, writes them at loc[b] (K rotated) and puts them over the newest
//    token's row of its landed tile, so no CTA reads them from the cache and
//    no tile waits for the store.
//  * fp8 cache (MODE_FP8, pa_paged_decode_attn_fp8): K/V rows are D bytes of
//    e4m3 with one scale per (layer, kv head).  Rows reach the ring by
//    cp.async only.  Keys feed f16 MMAs straight from shared memory: lane t4
//    takes bytes [t4 D/4, (t4+1) D/4) of rows g and g+8, four per k-step, so
//    the head dimension is permuted inside the dot product and q is loaded in
//    the same order (as f16).  Values are widened to f16 into a per-warp
//    staging tile in the bf16 tile layout and read by the same transposing
//    ldmatrix.  The K scale joins the softmax scale; the V scale multiplies
//    the item's output state.
//  * Launched behind another kernel (launch overlap on), the CTA waits for it
//    at the start, or -- early-metadata mode -- after planning and the first
//    page-table reads, just before its first K/V load.
//  * Ring waits are bounded in time (PA_DEVERR_TIMEOUT, then the CTA drains
//    and exits).
#include <math.h>

#include "pa_internal.h"
#include "pa_sm100.cuh"

namespace pa {
using namespace sm100;

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecTile = 16;        // tokens per ring stage
constexpr int kDecMinChunk = 64;    // split length bounds (tokens)
constexpr int kDecMaxChunk = 2048;
constexpr int kDecMaxBatch = 4096;
constexpr int kDecMaxSplits = 128;

// Kernel modes.  PLAIN: decode attention.  FUSED: the decode step (RoPE +
// KV store + attention).  PREFIX / SUFFIX: the two launches of cascade
// decode -- PREFIX runs "virtual requests" (a group's shared prefix against
// the q rows of up to 16 / G members at once) and writes each row's
// normalised output and log-sum-exp; SUFFIX runs every request over its
// tokens after its group's prefix and folds the prefix result into its
// output by log-sum-exp.
// FP8: decode attention over an e4m3 cache.
enum DecMode { MODE_PLAIN = 0, MODE_FUSED = 1, MODE_PREFIX = 2, MODE_SUFFIX = 3, MODE_FP8 = 4 };

struct DecodeArgs {
    CUtensorMap tm_k;    // 2-D (element, row) over k_buf rows, 64 x 16 boxes, 128-byte swizzle
    CUtensorMap tm_v;
    const __nv_bfloat16 *q;
    union {   // the layer's K / V rows: bf16, or e4m3 bytes in FP8 mode
        const __nv_bfloat16 *k_layer;
        const uint8_t *k8_layer;
    };
    union {
        const __nv_bfloat16 *v_layer;
        const uint8_t *v8_layer;
    };
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
    int layer_row0;      // layer_id * size: tensor-map row of slot 0 of the layer
    int early_meta;      // launched behind another kernel: plan and page table before waiting for it
    int early_kv;        // ... and copy K/V tiles (not the requests' newest rows) before waiting for it
    int defer_merge;     // large batch: every split's partials written, merged by a second kernel (no tickets)
    uint64_t wait_ns;    // time limit of the ring waits
    float scale_log2;
    // fused decode step (k_new != null): RoPE on q as it is loaded, and the new
    // token's rotated K and its V written at loc[b] and into the newest tile
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    const int32_t *positions;
    const int32_t *loc;
    union {   // fused step: the RoPE tables; FP8: the layer's per-kv-head K / V scales [Hkv]
        const float *cos_tab;
        const float *k_scale;
    };
    union {
        const float *sin_tab;
        const float *v_scale;
    };
    __nv_bfloat16 *k_layer_w;   // the layer's K / V rows, writable
    __nv_bfloat16 *v_layer_w;
    int max_pos;
    // cascade (PREFIX / SUFFIX)
    const int32_t *grp_indptr;  // [n_groups + 1]: members of group g are grp_reqs[grp_indptr[g] ..)
    const int32_t *grp_reqs;
    const int32_t *grp_prefix;  // [n_groups]: tokens shared by every member
    int n_groups, cpg, C;       // chunks per group, members per chunk (virtual request = (group, chunk))
    int G_real, Hq_real, B_real;
    int32_t *req_start;         // [B_real]: first token of the request's own part (PREFIX writes, SUFFIX reads)
    int32_t *req_pre;           // [B_real]: virtual request * 16 + member slot, or -1
    float *pre_o;               // [virtual batch, Hkv * G_v, D]: normalised prefix outputs
    float *pre_lse;             // [virtual batch, Hkv * G_v]: their log2-sum-exp (scaled-score units)
};

__device__ __forceinline__ int clamp_len(int n, int max_ctx) { return n < 0 ? 0 : (n > max_ctx ? max_ctx : n); }

// How requests are cut into splits.  Large batches: splits of about `chunk`
// tokens, many items per CTA.  Small batches (budget > 0): one wave -- request
// b gets floor(budget * n_b / tot) splits, budget = CTAs per kv head, so the
// items of all requests fill the grid once.
struct DecPlan {
    int chunk;
    int budget;
    float inv_tot;   // budget / total tokens (every CTA computes the same value)
    int bal;         // balanced large-batch plan (below)
    int W;           // bal: tiles per CTA
};

// Balanced plan for large batches whose merges are deferred: the (kv head,
// request) segments, head-major, are laid end to end as 16-token tiles (at
// least one per segment, so an empty request still writes its zero output),
// and CTA c takes tiles [c W, (c + 1) W).  Each piece of a segment inside one
// CTA's range is an item; a segment's pieces are its splits, in CTA order.
// Every CTA then streams the same number of tiles, whatever the mix of
// lengths (round-robin items of a common length left CTAs up to 15 % above
// the mean), and one CTA reads consecutive requests of one kv head, so pages
// that requests share are read again while they are in L2.
__device__ __forceinline__ int seg_tiles(int n) { return n > 0 ? (n + kDecTile - 1) / kDecTile : 1; }

// The plan of a launch of `grid` CTAs over B requests of `tot` tokens in all
// (every CTA, and the deferred merge, computes the same values).
__device__ __forceinline__ DecPlan make_plan(long long tot, int B, int Hkv, int grid, long long tiles = 0,
                                             int tb_max = 0, int max_splits = 0, bool allow_bal = false)
{
    const long long want = (tot * Hkv + grid - 1) / grid;
    DecPlan p;
    p.chunk = (int)((want + kDecMinChunk - 1) / kDecMinChunk * kDecMinChunk);
    p.chunk = p.chunk < kDecMinChunk ? kDecMinChunk : (p.chunk > kDecMaxChunk ? kDecMaxChunk : p.chunk);
    // one wave for small batches whose common split length would hit the cap
    p.budget = (2 * B * Hkv <= grid && want > kDecMaxChunk) ? grid / Hkv : 0;
    p.inv_tot = p.budget > 0 ? (float)p.budget / (float)tot : 0.f;
    // balanced: W tiles per CTA, a multiple of the warp count; a segment of
    // tb tiles has at most ceil(tb / W) + 1 pieces, which must fit max_splits
    p.bal = 0;
    p.W = 0;
    const long long T = tiles * Hkv;
    if (allow_bal && 2 * B * Hkv > grid && T < (1LL << 30)) {
        const long long W = ((T + grid - 1) / grid + kDecWarps - 1) / kDecWarps * kDecWarps;
        if ((tb_max + W - 1) / W + 1 <= max_splits) {
            p.bal = 1;
            p.W = (int)W;
        }
    }
    return p;
}

// split count and split length (tokens) of a request of n tokens
__device__ __forceinline__ void split_of(int n, const DecPlan &pl, int max_splits, int &sb, int &len)
{
    if (n <= 0) {
        sb = 1;
        len = 0;
        return;
    }
    int s;
    if (pl.budget > 0) {
        s = min((int)((float)n * pl.inv_tot), pl.budget);
        s = min(max(s, 1), (n + kDecMinChunk - 1) / kDecMinChunk);
    } else {
        s = (n + pl.chunk - 1) / pl.chunk;
    }
    if (s > max_splits) s = max_splits;
    // whole rounds of 16-token tiles for the 8 warps: every warp of the item
    // gets the same number of tiles (8K at 19 splits gave 27 tiles per item,
    // four warps of four and four of three)
    constexpr int kRound = kDecWarps * kDecTile;
    len = ((n + s - 1) / s + kRound - 1) / kRound * kRound;
    sb = (n + len - 1) / len;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared memory (from a 1024-byte aligned base): per-warp rings
// [warp][S][K tile | V tile], each tile D/64 halves of 16 rows x 128 B with the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)) -- the
// layout TMA writes and the cp.async path reproduces; consumer scratch;
// per-warp stage validity masks and mbarriers; the plan's prefix array.
template <int D, int S, int NH, bool F8 = false>
struct DecSmem {
    static constexpr int kHalf = kDecTile * 128;                         // 16 rows x 128 B
    static constexpr int kTile16 = (D / 64) * kHalf;                     // one K or V tile of 16-bit values
    static constexpr int kTile = F8 ? kDecTile * D : kTile16;            // one K or V tile as loaded
    static constexpr int kStage = 2 * kTile;
    static constexpr int kStaging = F8 ? kTile16 : 0;                    // fp8: the V tile widened to f16
    static constexpr int kRing = S * kStage + kStaging;                  // per warp
    static constexpr int kScratchOff = kDecWarps * kRing;
    // half the warps' O states [4][G][D + 4] fp32 at a time, later the split merge
    // [sb][G][2] + [sb][G] + [G]
    static constexpr int kCombineStride = D + 4;   // padded row: the four t4 lanes of a store hit distinct banks
    static constexpr int kCombine = (kDecWarps / 2) * 8 * NH * kCombineStride * 4;
    static constexpr int kMerge = (3 * kDecMaxSplits * 8 * NH + 16 * NH) * 4;
    static constexpr int kScratch = kCombine > kMerge ? kCombine : kMerge;
    static constexpr int kMaskOff = kScratchOff + kScratch;
    static constexpr int kBarOff = kMaskOff + kDecWarps * S * 4;
    // q rows of the current item [8 NH][D / 2 + 4] words (bf16 pairs; rows
    // padded so the fragment reads, 8 rows x 4 words, hit distinct banks)
    static constexpr int kQStride = D / 2 + 4;
    static constexpr int kQOff = kBarOff + kDecWarps * S * 8;
    static constexpr int kPrefOff = kQOff + 8 * NH * kQStride * 4;
    // after the prefix array [batch + 1]: each request's (clamped length, table row), int2 [batch]
    __host__ __device__ static constexpr size_t req_off(int batch) { return (size_t)kPrefOff + (size_t)(batch + 2) / 2 * 8; }
    static constexpr size_t bytes(int batch) { return 1024 + req_off(batch) + (size_t)batch * 8; }
    // byte offset of 16-byte chunk c of row r inside a K or V tile
    __device__ static __forceinline__ uint32_t off(int r, int c)
    {
        return (uint32_t)((c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    }
    // fp8 tiles: row r of D bytes, 16-byte chunk c (128-byte rows XOR-swizzled
    // like off; 64-byte rows plain -- both conflict free for the fragment reads)
    __device__ static __forceinline__ uint32_t off8(int r, int c)
    {
        return D == 128 ? (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)) : (uint32_t)(r * D + (c << 4));
    }
};
constexpr size_t kSmemLimit = 232448 - 4096;   // opt-in maximum minus static shared memory (with margin)

// Everything an item needs, derived from the plan (identical in every warp).
struct DecItem {
    int b, s, h, sb, t0, t1, ntiles;
    int row;    // -1 if the request row is invalid
    int wofs;   // tile i of the item is computed by warp (i + wofs) % 8
};

// request of a work item: the largest b with s_pref[b] <= item (shared memory only)
__device__ __forceinline__ int item_request(const int *s_pref, int batch, int item)
{
    int lo = 0, hi = batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] <= item) lo = mid; else hi = mid;
    }
    return lo;
}

// Tokens of request b this launch attends to: [start, start + n).  PREFIX:
// a virtual request (group, chunk) covers its group's shared prefix (none for
// an empty chunk) through the chunk's first member's page-table row.
template <int MODE>
__device__ __forceinline__ void req_span(const DecodeArgs &a, int b, int &start, int &n, int &row)
{
    if (MODE == MODE_PREFIX) {
        const int g = b / a.cpg, c = b - g * a.cpg;
        const int first = __ldg(a.grp_indptr + g) + c * a.C;
        start = 0;
        n = 0;
        row = -1;
        if (first < __ldg(a.grp_indptr + g + 1)) {
            const int m0 = __ldg(a.grp_reqs + first);
            if (m0 >= 0 && m0 < a.B_real) {
                n = clamp_len(__ldg(a.grp_prefix + g), a.max_ctx);
                row = __ldg(a.req_pool_indices + m0);
            }
        }
        return;
    }
    const int full = clamp_len(__ldg(a.seq_lens + b), a.max_ctx);
    start = MODE == MODE_SUFFIX ? min(max(__ldg(a.req_start + b), 0), full) : 0;
    n = full - start;
    row = __ldg(a.req_pool_indices + b);
}

template <int MODE>
__device__ __forceinline__ int req_len(const DecodeArgs &a, int b)
{
    if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8) {
        return clamp_len(__ldg(a.seq_lens + b), a.max_ctx);
    } else {
        int start, n, row;
        req_span<MODE>(a, b, start, n, row);
        return n;
    }
}

// s_req (plain, fused and fp8 modes): each request's clamped length and
// table row, read from global memory once, during the plan.
template <int MODE>
__device__ __forceinline__ DecItem dec_item(const DecodeArgs &a, const int *s_pref, const int2 *s_req,
                                            const DecPlan &chunk, int item, int seg0 = 0)
{
    DecItem I;
    I.wofs = 0;
    if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8) {
        if (chunk.bal) {
            // piece p of this CTA's tile range: segment seg0 + p (s_pref holds
            // each request's first tile within a kv head's run of segments)
            const int seg = seg0 + (item - (int)blockIdx.x) / (int)gridDim.x;
            I.h = seg / a.batch;
            I.b = seg - I.h * a.batch;
            const int2 rq = s_req[I.b];
            int n = rq.x;
            const int tb = seg_tiles(n);
            const int S0 = I.h * s_pref[a.batch] + s_pref[I.b];   // the segment's first tile
            const int x0 = (int)blockIdx.x * chunk.W;
            const int u0 = max(x0, S0), u1 = min(x0 + chunk.W, S0 + tb);
            I.s = (int)blockIdx.x - S0 / chunk.W;
            I.sb = (S0 + tb - 1) / chunk.W - S0 / chunk.W + 1;
            I.row = rq.y;
            if (I.row < 0 || I.row >= a.req_rows) {
                I.row = -1;
                n = 0;
            }
            I.t0 = (u0 - S0) * kDecTile;
            I.t1 = min(n, (u1 - S0) * kDecTile);
            I.ntiles = I.t1 > I.t0 ? (I.t1 - I.t0 + kDecTile - 1) / kDecTile : 0;
            I.wofs = (u0 - x0) & (kDecWarps - 1);
            return I;
        }
    }
    const int lo = item_request(s_pref, a.batch, item);
    I.b = lo;
    const int local = item - s_pref[lo];
    I.s = local / a.Hkv;
    I.h = local - I.s * a.Hkv;
    if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8) {
        const int2 rq = s_req[lo];
        int n = rq.x;
        int len;
        split_of(n, chunk, a.max_splits, I.sb, len);
        I.row = rq.y;
        if (I.row < 0 || I.row >= a.req_rows) {
            I.row = -1;
            n = 0;
        }
        I.t0 = I.s * len;
        I.t1 = min(n, I.t0 + len);
    } else {
        int start, n;
        req_span<MODE>(a, lo, start, n, I.row);
        int len;
        split_of(n, chunk, a.max_splits, I.sb, len);
        if (I.row < 0 || I.row >= a.req_rows) {
            I.row = -1;
            n = 0;
        }
        I.t0 = start + I.s * len;
        I.t1 = start + min(n, I.s * len + len);
    }
    I.ntiles = I.t1 > I.t0 ? (I.t1 - I.t0 + kDecTile - 1) / kDecTile : 0;
    return I;
}

// BAL: the instance for large batches (merges deferred), which takes the
// balanced plan when it fits; the other instances carry none of its code.
template <int D, int S, int NH, int MODE, bool BAL = false>
__global__ void __launch_bounds__(kDecThreads, 1) paged_decode_kernel(const __grid_constant__ DecodeArgs a)
{
    using L = DecSmem<D, S, NH, MODE == MODE_FP8>;
    constexpr bool FUSED = MODE == MODE_FUSED;
    constexpr bool F8 = MODE == MODE_FP8;
    // the suffix launch plans from req_start, which the prefix launch writes:
    // it never plans before its wait
    const bool early = a.early_meta && MODE != MODE_SUFFIX;
    const bool early_kv = early && a.early_kv && (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8);
    constexpr int KSTEPS = D / 16;
    constexpr int DM = D / 16;         // 16-row d tiles of O^T
    constexpr int CPR = D / 8;         // 16-byte chunks per row
    constexpr int TPI = 32 / CPR;      // rows per warp-wide copy instruction

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));
    float *scratch = reinterpret_cast<float *>(smem + L::kScratchOff);
    uint32_t *s_vmask = reinterpret_cast<uint32_t *>(smem + L::kMaskOff);
    int32_t *s_pref = reinterpret_cast<int32_t *>(smem + L::kPrefOff);
    int2 *s_req = reinterpret_cast<int2 *>(smem + L::req_off(a.batch));
    __shared__ float s_m[kDecWarps][16], s_l[kDecWarps][16];
    __shared__ int s_red[kDecWarps], s_red2[kDecWarps], s_red3[kDecWarps];
    __shared__ int s_flag, s_pend[3];
    __shared__ int s_abort_storage;
    __shared__ int32_t s_pos[FUSED ? kDecThreads : 1];   // fused step: positions[b] of this CTA's first items
    volatile int *s_abort = &s_abort_storage;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int B = a.batch, Hkv = a.Hkv, G = a.G;
    const uint32_t bars = smem_u32(smem + L::kBarOff) + warp * S * 8;   // this warp's stage barriers
    if (lane == 0) {
        // 32 lanes' cp.async completions + lane 0's arrival carrying the TMA bytes
        for (int i = 0; i < S; ++i) mbar_init(bars + i * 8, 33);
        fence_mbar_init();
    }
    if (tid == 0) *s_abort = 0;
    if (!early) pdl_wait();

    // ---------------------------------------------------------- planning
    // the balanced plan: large batches of the plain, fused and fp8 modes,
    // whose merges the second kernel does
    constexpr bool kBal = BAL && (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8);
    int my_tot = 0, my_tiles = 0, my_tbmax = 0;
    for (int b = tid; b < B; b += kDecThreads) {
        const int n = req_len<MODE>(a, b);
        my_tot += n;
        if constexpr (kBal) {
            my_tiles += seg_tiles(n);
            my_tbmax = max(my_tbmax, seg_tiles(n));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        my_tot += __shfl_xor_sync(0xffffffffu, my_tot, o);
        if constexpr (kBal) {
            my_tiles += __shfl_xor_sync(0xffffffffu, my_tiles, o);
            my_tbmax = max(my_tbmax, __shfl_xor_sync(0xffffffffu, my_tbmax, o));
        }
    }
    if (lane == 0) {
        s_red[warp] = my_tot;
        s_red2[warp] = my_tiles;
        s_red3[warp] = my_tbmax;
    }
    __syncthreads();
    long long tot = 0, tiles = 0;
    int tb_max = 0;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
        tot += s_red[w];
        if constexpr (kBal) {
            tiles += s_red2[w];
            tb_max = max(tb_max, s_red3[w]);
        }
    }
    const DecPlan chunk = make_plan(tot, B, Hkv, (int)gridDim.x, tiles, tb_max, a.max_splits, kBal && a.defer_merge);
    {
        const int per = (B + kDecThreads - 1) / kDecThreads;
        const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
        // items (split x kv head) per request, or (balanced) its tiles
        auto units = [&](int n) -> int {
            if (chunk.bal) return seg_tiles(n);   // per kv head
            int sb, len;
            split_of(n, chunk, a.max_splits, sb, len);
            return sb * Hkv;
        };
        int run = 0;
        for (int b = b_lo; b < b_hi; ++b) run += units(req_len<MODE>(a, b));
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
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
            const int n = req_len<MODE>(a, b);
            excl += units(n);
            if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8)
                s_req[b] = make_int2(n, __ldg(a.req_pool_indices + b));
        }
        if (tid == kDecThreads - 1) s_pref[B] = base + incl;
    }
    __syncthreads();
    const int total_items = s_pref[B];
    // this CTA's items are blockIdx.x, + gridDim.x, ... below item_end; in the
    // balanced plan, piece p of its tile range (segments seg0, seg0 + 1, ...)
    int item_end = total_items, seg0 = 0;
    if (chunk.bal) {
        // total_items: the tiles of one kv head's segments
        const int x0 = (int)blockIdx.x * chunk.W, T = Hkv * total_items;
        item_end = 0;
        if (x0 < T) {
            const int xl = min(x0 + chunk.W, T) - 1;
            const int h0 = x0 / total_items, hl = xl / total_items;
            seg0 = h0 * B + item_request(s_pref, B, x0 - h0 * total_items);
            const int segl = hl * B + item_request(s_pref, B, xl - hl * total_items);
            item_end = (int)blockIdx.x + (segl - seg0 + 1) * (int)gridDim.x;
        }
    }
    const int64_t slot_stride = (int64_t)Hkv * D;
    const uint32_t ring = smem_u32(smem) + warp * L::kRing;
    bool bad = false;   // a ring wait timed out: skip work, keep the barriers
    int ring_err = 0;   // error bits found while loading tiles, written at the end (some precede the wait)

    // ------------------------------------------- this warp's load cursors
    // a cursor walks (item, tile) pairs in the order the warp computes them:
    // tiles warp, warp+8, ... of the CTA's items blockIdx.x, +gridDim.x, ...
    // `cur` is the next tile to load, `nxt` the one after; both hold their
    // page-table entries (lane t < 16: token t), fetched when the cursor moved
    struct Cursor {
        int item, tile, slot;
        DecItem I;
    };
    auto settle = [&](Cursor &c) {
        while (c.item < item_end && c.tile >= c.I.ntiles) {
            c.item += gridDim.x;
            if (c.item < item_end) c.I = dec_item<MODE>(a, s_pref, s_req, chunk, c.item, seg0);
            c.tile = (warp - c.I.wofs) & (kDecWarps - 1);
        }
        c.slot = -1;
        if (c.item < item_end && lane < kDecTile && c.I.row >= 0) {
            const int tok = c.I.t0 + c.tile * kDecTile + lane;
            if (tok < c.I.t1) c.slot = __ldg(a.req_to_token + (int64_t)c.I.row * a.max_ctx + tok);
        }
    };
    Cursor cur;
    cur.item = blockIdx.x;
    cur.I.ntiles = 0;
    cur.I.row = -1;
    cur.I.t0 = cur.I.t1 = cur.I.h = cur.I.wofs = 0;
    if (cur.item < item_end) cur.I = dec_item<MODE>(a, s_pref, s_req, chunk, cur.item, seg0);
    cur.tile = (warp - cur.I.wofs) & (kDecWarps - 1);
    // the CTA's first item, kept for the item loop: in early-metadata mode it
    // is derived before the wait, so the loop's first iteration re-reads nothing
    const DecItem first_I = cur.I;
    settle(cur);
    Cursor nxt = cur;
    nxt.tile += kDecWarps;
    settle(nxt);
    int n_issued = 0;
    // load the `cur` tile into ring stage n_issued % S, then advance both cursors
    auto issue = [&]() {
        if (cur.item >= item_end) return;
        const int st = n_issued % S;
        const uint32_t kb = ring + st * L::kStage, vb = kb + L::kTile, fb = bars + st * 8;
        const int tok0 = cur.I.t0 + cur.tile * kDecTile;
        int sl = cur.slot;
        const bool in_range = lane < kDecTile && tok0 + lane < cur.I.t1;
        if (in_range && (sl < 0 || sl >= a.size)) ring_err |= PA_DEVERR_SLOT;
        const bool ok = in_range && sl >= 0 && sl < a.size;
        if (!ok) sl = -1;
        const unsigned vmask = __ballot_sync(0xffffffffu, ok);
        if constexpr (F8) {
            // 16 tokens on one page: a TMA box of 16 D-byte rows per K / V
            // tile; otherwise D-byte rows by cp.async, D/16 lanes per row,
            // masked rows zero-filled, not read
            constexpr int CPR8 = D / 16, TPI8 = 32 / CPR8;
            const int s0 = __shfl_sync(0xffffffffu, sl, 0);
            const bool page = (__ballot_sync(0xffffffffu, ok && sl == s0 + lane) & 0xFFFFu) == 0xFFFFu;
            if (lane == 0) {
                s_vmask[warp * S + st] = vmask;
                mbar_arrive_expect_tx(fb, page ? 2u * L::kTile : 0u);
            }
            __syncwarp();
            if (page) {
                if (lane == 0) {
                    tma_load_2d(kb, &a.tm_k, cur.I.h * D, a.layer_row0 + s0, fb);
                    tma_load_2d(vb, &a.tm_v, cur.I.h * D, a.layer_row0 + s0, fb);
                }
            } else {
                const uint8_t *kh = a.k8_layer + (int64_t)cur.I.h * D;
                const uint8_t *vh = a.v8_layer + (int64_t)cur.I.h * D;
#pragma unroll
                for (int j = 0; j < kDecTile / TPI8; ++j) {
                    const int r = j * TPI8 + lane / CPR8;
                    const int ch = lane % CPR8;
                    const int rs = __shfl_sync(0xffffffffu, sl, r);
                    const int64_t off = rs >= 0 ? (int64_t)rs * slot_stride + ch * 16 : 0;
                    const int nb = rs >= 0 ? 16 : 0;
                    cp_async_16(kb + L::off8(r, ch), kh + off, nb);
                    cp_async_16(vb + L::off8(r, ch), vh + off, nb);
                }
            }
        } else {
            // 16 tokens on 16 consecutive slots (one page): four TMA boxes
            const int s0 = __shfl_sync(0xffffffffu, sl, 0);
            const bool page = (__ballot_sync(0xffffffffu, ok && sl == s0 + lane) & 0xFFFFu) == 0xFFFFu;
            if (lane == 0) {
                s_vmask[warp * S + st] = vmask;
                mbar_arrive_expect_tx(fb, page ? 2u * L::kTile : 0u);
            }
            __syncwarp();
            const int h = cur.I.h;
            if (page) {
                if (lane == 0) {
#pragma unroll
                    for (int hh = 0; hh < D / 64; ++hh) {
                        tma_load_2d(kb + hh * L::kHalf, &a.tm_k, h * D + hh * 64, a.layer_row0 + s0, fb);
                        tma_load_2d(vb + hh * L::kHalf, &a.tm_v, h * D + hh * 64, a.layer_row0 + s0, fb);
                    }
                }
            } else {
                const __nv_bfloat16 *kh = a.k_layer + (int64_t)h * D;
                const __nv_bfloat16 *vh = a.v_layer + (int64_t)h * D;
#pragma unroll
                for (int j = 0; j < kDecTile / TPI; ++j) {
                    const int r = j * TPI + lane / CPR;
                    const int ch = lane % CPR;
                    const int rs = __shfl_sync(0xffffffffu, sl, r);
                    const int64_t off = rs >= 0 ? (int64_t)rs * slot_stride + ch * 8 : 0;
                    const int nb = rs >= 0 ? 16 : 0;      // masked rows: zero fill, no read
                    const uint32_t o = L::off(r, ch);
                    cp_async_16(kb + o, kh + off, nb);
                    cp_async_16(vb + o, vh + off, nb);
                }
            }
        }
        cp_async_arrive_noinc(fb);
        ++n_issued;
        cur = nxt;
        nxt.tile += kDecWarps;
        settle(nxt);
    };

    // the plan and the first page-table entries only read index arrays; K/V,
    // q, the workspace and out wait for the preceding kernel
    // early K/V: a warp's first tiles are copied before the wait, stopping at
    // the first tile that holds a request's newest token (the last tile of
    // its last split), which the preceding kernel may write.  The fused step
    // does not stop there: it replaces that row in shared memory (below).
    int pre = 0;
    if (early_kv) {
        while (pre < S - 1 && cur.item < item_end &&
               (FUSED || !(cur.I.s == cur.I.sb - 1 && cur.tile == cur.I.ntiles - 1))) {
            issue();
            ++pre;
        }
    }
    if (FUSED) {
        // positions[b] of this CTA's first items (an index array: ahead of the
        // wait in early-metadata mode), so the q rotation needs no global load
        const int item = blockIdx.x + tid * (int)gridDim.x;
        if (item < item_end)
            s_pos[tid] = __ldg(a.positions + (chunk.bal ? (seg0 + tid) % B : item_request(s_pref, a.batch, item)));
        __syncthreads();
    }
    if (early) pdl_wait();
    pdl_launch_dependents();
    if (MODE == MODE_PREFIX && blockIdx.x == 0) {
        // the suffix launch's per-request start token and prefix row
        for (int b = tid; b < a.B_real; b += kDecThreads) {
            a.req_start[b] = 0;
            a.req_pre[b] = -1;
        }
        __syncthreads();
        const int n_mem = __ldg(a.grp_indptr + a.n_groups);
        for (int e = tid; e < n_mem; e += kDecThreads) {
            int lo = 0, hi = a.n_groups;   // group of entry e: largest g with grp_indptr[g] <= e
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(a.grp_indptr + mid) <= e) lo = mid; else hi = mid;
            }
            const int i = e - __ldg(a.grp_indptr + lo);
            const int b = __ldg(a.grp_reqs + e);
            if (b >= 0 && b < a.B_real && i < a.cpg * a.C) {
                a.req_start[b] = max(__ldg(a.grp_prefix + lo), 0);
                a.req_pre[b] = (lo * a.cpg + i / a.C) * 16 + i % a.C;
            }
        }
    }
    for (; pre < S - 1; ++pre) issue();

    // ------------------------------------------------------ split merge
    // The CTA whose ticket completes (b, h) merges all its splits in split
    // order, writes bf16 and re-arms the ticket.  Whole-CTA; uses the scratch.
    // The first 20 splits (8 when G > 8) of this thread's output elements are
    // requested before the (m, l) pairs, so both travel in one round trip; the split
    // weights are computed warp-parallel (a warp per q head, lanes over
    // splits, shuffle max and sum).
    int pend_prev = -1;                        // thread 0: pending ticket result
    // Final output of element (request b, q head hq, dim d) from the merged
    // unnormalised acc, sum l and max mx (log2 units).  PREFIX writes the
    // normalised fp32 row and its log-sum-exp; SUFFIX combines with the
    // request's prefix row, if it has one, by log-sum-exp.
    auto emit = [&](int b, int hq, int d, float acc, float l, float mx, int pre) {
        const float o = l > 0.f ? acc / l : 0.f;
        if (MODE == MODE_PREFIX) {
            a.pre_o[((int64_t)b * a.Hq + hq) * D + d] = o;
            if (d == 0) a.pre_lse[(int64_t)b * a.Hq + hq] = l > 0.f ? mx + __log2f(l) : -INFINITY;
            return;
        }
        if (MODE == MODE_SUFFIX && pre >= 0) {
            const int h = hq / G, j = hq - h * G;
            const int64_t prow = ((int64_t)(pre >> 4) * Hkv + h) * (a.C * G) + (pre & 15) * G + j;
            const float lse_p = __ldcg(a.pre_lse + prow), o_p = __ldcg(a.pre_o + prow * D + d);
            const float lse_s = l > 0.f ? mx + __log2f(l) : -INFINITY;
            const float M = fmaxf(lse_s, lse_p);
            float val = 0.f;
            if (M != -INFINITY) {
                const float ws = ex2(lse_s - M), wp = ex2(lse_p - M);
                val = (ws * o + wp * o_p) / (ws + wp);
            }
            a.out[((int64_t)b * a.Hq + hq) * D + d] = __float2bfloat16_rn(val);
            return;
        }
        a.out[((int64_t)b * a.Hq + hq) * D + d] = __float2bfloat16_rn(o);
    };
    auto merge_splits = [&](int b, int h, int sb) {
        const int hq0 = h * G;
        float *s_w = scratch;              // [sb][G] split weights
        float *s_lt = s_w + sb * G;        // [G] weighted sums of l
        float *s_M = s_lt + G;             // [G] the maxima they are relative to
        const int pre = MODE == MODE_SUFFIX ? __ldcg(a.req_pre + b) : -1;
        constexpr int EPT = (8 * NH * D + kDecThreads - 1) / kDecThreads;
        constexpr int SPL = kDecMaxSplits / 32;   // splits per lane
        const int64_t split_stride = (int64_t)a.cap_batch * a.Hq * D;
        const float *obase = a.o_part + ((int64_t)b * a.Hq + hq0) * D;
        // splits per element per round trip: 20 covers the one-wave plans'
        // 19 splits per head in one trip (registers EPT * SB)
        constexpr int SB = EPT <= 4 ? 20 : 8;
        float v[EPT][SB];
        auto load_batch = [&](int ss) {
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const int e = tid + k * kDecThreads;
#pragma unroll
                for (int j = 0; j < SB; ++j)
                    v[k][j] = ld_cg_ordered_if(e < G * D && ss + j < sb, obase + e + (ss + j) * split_stride);
            }
        };
        // this warp's first head's (m, l) pairs, then the first batch of
        // partials: all requested before any value is used (one round trip)
        const int64_t ml_stride = (int64_t)a.cap_batch * a.Hq * 2;   // floats per split
        float mv[SPL], lv[SPL];
        auto load_ml = [&](int gg) {
            const float *ml = a.ml_part + ((int64_t)b * a.Hq + hq0 + gg) * 2;
#pragma unroll
            for (int r = 0; r < SPL; ++r) {
                const int ss = lane + 32 * r;
                mv[r] = ss < sb ? __ldcg(ml + ss * ml_stride) : -INFINITY;
                lv[r] = ss < sb ? __ldcg(ml + ss * ml_stride + 1) : 0.f;
            }
        };
        if (warp < G) load_ml(warp);
        load_batch(0);
        for (int gg = warp; gg < G; gg += kDecWarps) {
            if (gg != warp) load_ml(gg);
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < SPL; ++r) M = fmaxf(M, mv[r]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float Mr = M == -INFINITY ? 0.f : M;
            float lt = 0.f;
#pragma unroll
            for (int r = 0; r < SPL; ++r) {
                const int ss = lane + 32 * r;
                if (ss < sb) {
                    const float wt = ex2(mv[r] - Mr);
                    s_w[ss * G + gg] = wt;
                    lt += wt * lv[r];
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
            if (lane == 0) {
                s_lt[gg] = lt;
                if constexpr (MODE == MODE_PREFIX || MODE == MODE_SUFFIX) s_M[gg] = Mr;
            }
        }
        __syncthreads();
        float acc[EPT];
#pragma unroll
        for (int k = 0; k < EPT; ++k) acc[k] = 0.f;
        for (int ss = 0; ss < sb; ss += SB) {   // each element summed in split order
            if (ss > 0) load_batch(ss);
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const int e = tid + k * kDecThreads;
                if (e >= G * D) continue;
                const int gg = e / D;
#pragma unroll
                for (int j = 0; j < SB; ++j)
                    if (ss + j < sb) acc[k] += s_w[(ss + j) * G + gg] * v[k][j];
            }
        }
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int e = tid + k * kDecThreads;
            if (e >= G * D) continue;
            if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8) {
                const float lt = s_lt[e / D];
                a.out[((int64_t)b * a.Hq + hq0) * D + e] = __float2bfloat16_rn(lt > 0.f ? acc[k] / lt : 0.f);
            } else {
                emit(b, hq0 + e / D, e % D, acc[k], s_lt[e / D], s_M[e / D], pre);
            }
        }
        if (tid == 0) a.counters[b * Hkv + h] = 0;
        __syncthreads();
    };
    // examine the pending ticket (whole CTA): merge if this CTA was last
    auto resolve_ticket = [&]() {
        if (tid == 0) {
            // the ticket's acquire made the other CTAs' partials visible
            s_flag = pend_prev >= 0 && pend_prev == s_pend[2] - 1;
            pend_prev = -1;
        }
        __syncthreads();
        if (s_flag) merge_splits(s_pend[0], s_pend[1], s_pend[2]);
    };

    int n_done = 0;   // tiles computed (or, after a timed-out wait, skipped) by this warp
    int n_landed = 0; // tiles whose ring wait succeeded: those after it may still be in flight
    bool ticket_pending = false;   // CTA-uniform: the previous item took a merge ticket
    for (int item = blockIdx.x; item < item_end; item += gridDim.x) {
        const DecItem I = item == (int)blockIdx.x ? first_I : dec_item<MODE>(a, s_pref, s_req, chunk, item, seg0);
        const int hq0 = I.h * G;
        if (a.wait_ns == 0 && !bad) {
            // a wait limit of 0: give up at the first item, as a timed-out ring wait would
            *s_abort = 1;
            set_error(a.err, PA_DEVERR_TIMEOUT);
            bad = true;
        }
        // Fused step: the warp that computes the last tile of a (request, kv
        // head)'s last split -- warp 0 if the item has no tile -- loads that
        // head's new K and V rows together with q (lane c < D/8: K chunk c;
        // lane D/8 + c: V chunk c; K lanes also their cos / sin values).  It
        // writes them at loc[b] (K rotated) and, once the tile has landed,
        // over the newest token's row of the tile, so the rows are never read
        // back from the cache.
        int32_t new_pos = 0, new_slot = -1;
        bool new_own = false, new_tile = false;
        uint4 new_x = make_uint4(0u, 0u, 0u, 0u);
        float4 new_c = make_float4(0.f, 0.f, 0.f, 0.f), new_s = new_c;
        constexpr int NCH = D / 8;   // 16-byte chunks of a K or V row
        if constexpr (FUSED) {
            const int k_item = (item - (int)blockIdx.x) / (int)gridDim.x;
            new_pos = k_item < kDecThreads ? s_pos[k_item] : __ldg(a.positions + I.b);
            new_own = I.s == I.sb - 1 && warp == (I.ntiles > 0 ? (I.ntiles - 1 + I.wofs) % kDecWarps : 0);
            if (new_own) {
                new_slot = __ldg(a.loc + I.b);
                const bool slot_ok = new_slot >= 0 && new_slot < a.size;
                const bool pos_ok = new_pos >= 0 && new_pos < a.max_pos;
                const bool match = I.row >= 0 && I.t1 > 0 &&
                                   __ldg(a.req_to_token + (int64_t)I.row * a.max_ctx + I.t1 - 1) == new_slot;
                new_tile = I.ntiles > 0 && slot_ok && match;
                if (!slot_ok) new_slot = -1;
                const int e = (pos_ok ? 0 : PA_DEVERR_POS) |
                              (!slot_ok || (I.row >= 0 && I.t1 > 0 && !match) ? PA_DEVERR_SLOT : 0);
                if (lane == 0 && e) set_error(a.err, e);
                const bool isv = lane >= NCH;
                const int c = lane - (isv ? NCH : 0);
                if (lane < 2 * NCH) {
                    const int64_t src = ((int64_t)I.b * Hkv + I.h) * D;
                    new_x = __ldg(reinterpret_cast<const uint4 *>((isv ? a.v_new : a.k_new) + src) + c);
                    if (!isv && pos_ok) {
                        new_c = __ldg(reinterpret_cast<const float4 *>(a.cos_tab + (int64_t)new_pos * (D / 2)) + c);
                        new_s = __ldg(reinterpret_cast<const float4 *>(a.sin_tab + (int64_t)new_pos * (D / 2)) + c);
                    }
                }
            }
        }
        // the new rows as stored (K rotated), written at loc[b]; true if the
        // tile may take them too
        auto put_new_rows = [&]() -> uint4 {
            uint4 x = new_x;
            if (lane < NCH && new_pos >= 0 && new_pos < a.max_pos)
                x = make_uint4(rope_pair_bf16(x.x, new_c.x, new_s.x), rope_pair_bf16(x.y, new_c.y, new_s.y),
                               rope_pair_bf16(x.z, new_c.z, new_s.z), rope_pair_bf16(x.w, new_c.w, new_s.w));
            if (lane < 2 * NCH && new_slot >= 0) {
                const bool isv = lane >= NCH;
                __nv_bfloat16 *dst = (isv ? a.v_layer_w : a.k_layer_w) + (int64_t)new_slot * slot_stride + (int64_t)I.h * D;
                reinterpret_cast<uint4 *>(dst)[lane - (isv ? NCH : 0)] = x;
            }
            return x;
        };
        if (FUSED && new_own && I.ntiles == 0) put_new_rows();
        // Q^T as the MMA's B operand: n = head (8 per n-tile), k = d
        uint32_t qb[KSTEPS][NH][2];
        {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(a.q + ((int64_t)I.b * a.Hq + hq0) * D);
            // every load is issued before any use; word i of a head row is
            // RoPE pair i (fused step: rotated by table row positions[b]);
            // prefix launch: row hd of a virtual request is head hd % G of
            // member hd / G of its chunk, G the real GQA group
            if constexpr (MODE != MODE_PREFIX) {
                // the item's G head rows through shared memory: every thread
                // loads whole words of them (consecutive threads, consecutive
                // words), the fused step rotates each pair once per CTA, and
                // every warp then reads its B fragments from the staged rows
                uint32_t *s_q = reinterpret_cast<uint32_t *>(smem + L::kQOff);
                constexpr int QW = D / 2;   // words (RoPE pairs) of a head row
                constexpr int QE = (8 * NH * QW + kDecThreads - 1) / kDecThreads;
                int32_t pc = 0;
                bool rot = false;
                if constexpr (FUSED) {
                    pc = (new_pos >= 0 && new_pos < a.max_pos) ? new_pos : 0;   // out of range: no rotation
                    rot = pc == new_pos;
                }
                uint32_t qw[QE];
                float qc[QE], qs[QE];
#pragma unroll
                for (int k = 0; k < QE; ++k) {
                    const int e = tid + k * kDecThreads, hd = e / QW, i = e - hd * QW;
                    qw[k] = hd < G ? __ldg(q32 + hd * QW + i) : 0u;
                    if constexpr (FUSED) {
                        qc[k] = hd < G ? __ldg(a.cos_tab + (int64_t)pc * QW + i) : 0.f;
                        qs[k] = hd < G ? __ldg(a.sin_tab + (int64_t)pc * QW + i) : 0.f;
                    }
                }
#pragma unroll
                for (int k = 0; k < QE; ++k) {
                    const int e = tid + k * kDecThreads, hd = e / QW, i = e - hd * QW;
                    uint32_t x = (FUSED && rot) ? rope_pair_bf16(qw[k], qc[k], qs[k]) : qw[k];
                    if constexpr (F8) x = bf16x2_to_f16x2_sat(x);   // fp8 cache: q as f16
                    if (hd < 8 * NH) s_q[hd * L::kQStride + i] = x;
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt) {
                        if constexpr (F8) {
                            // the keys' permuted head dimension: k-step kk of
                            // lane t4 covers d = t4 D/4 + 4 kk + {0, 1 | 2, 3}
                            const uint32_t *row = s_q + (nt * 8 + g) * L::kQStride + t4 * (D / 8) + 2 * kk;
                            qb[kk][nt][0] = row[0];
                            qb[kk][nt][1] = row[1];
                        } else {
                            const uint32_t *row = s_q + (nt * 8 + g) * L::kQStride + kk * 8 + t4;
                            qb[kk][nt][0] = row[0];
                            qb[kk][nt][1] = row[4];
                        }
                    }
            } else {
            const uint32_t *qrow[NH];
            bool qok[NH];
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                const int hd = nt * 8 + g;
                qok[nt] = hd < G;
                qrow[nt] = q32 + hd * (D / 2);
                {
                    const int gr = I.b / a.cpg, c = I.b - gr * a.cpg;
                    const int m = hd / a.G_real, j = hd - m * a.G_real;
                    const int e = __ldg(a.grp_indptr + gr) + c * a.C + m;
                    qok[nt] = qok[nt] && m < a.C && e < __ldg(a.grp_indptr + gr + 1);
                    const int bm = qok[nt] ? __ldg(a.grp_reqs + e) : 0;
                    qok[nt] = qok[nt] && bm >= 0 && bm < a.B_real;
                    qrow[nt] = reinterpret_cast<const uint32_t *>(
                        a.q + ((int64_t)(qok[nt] ? bm : 0) * a.Hq_real + I.h * a.G_real + j) * D);
                }
            }
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                for (int nt = 0; nt < NH; ++nt) {
                    qb[kk][nt][0] = qok[nt] ? __ldg(qrow[nt] + kk * 8 + t4) : 0u;
                    qb[kk][nt][1] = qok[nt] ? __ldg(qrow[nt] + kk * 8 + 4 + t4) : 0u;
                }
            }
        }
        float o[DM][NH][4];
#pragma unroll
        for (int i = 0; i < DM; ++i)
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) o[i][nt][0] = o[i][nt][1] = o[i][nt][2] = o[i][nt][3] = 0.f;
        float m[NH][2], l[NH][2];
#pragma unroll
        for (int nt = 0; nt < NH; ++nt) m[nt][0] = m[nt][1] = -INFINITY, l[nt][0] = l[nt][1] = 0.f;

        float sl2_f8 = 0.f;   // fp8: softmax scale (log2 units) times the head's K scale
        if constexpr (F8) sl2_f8 = a.scale_log2 * __ldg(a.k_scale + I.h);
        for (int i = (warp - I.wofs) & (kDecWarps - 1); i < I.ntiles; i += kDecWarps) {
            if (!bad) issue();
            const int st = n_done % S;
            if (!bad && !mbar_wait(bars + st * 8, (n_done / S) & 1, s_abort, a.err, PA_DEVERR_TIMEOUT, a.wait_ns))
                bad = true;
            if (!bad) ++n_landed;
            ++n_done;
            if (FUSED && new_own && i == I.ntiles - 1) {
                const uint4 x = put_new_rows();
                if (!bad && new_tile) {
                    // the newest token's row of the landed tile: generic writes,
                    // ordered before the ring's next async-proxy (TMA) refill
                    const int r = I.t1 - 1 - (I.t0 + i * kDecTile);
                    if (lane < 2 * NCH) {
                        const bool isv = lane >= NCH;
                        const uint32_t tb = ring + st * L::kStage + (isv ? L::kTile : 0);
                        st_shared_v4(tb + L::off(r, lane - (isv ? NCH : 0)), x.x, x.y, x.z, x.w);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
            }
            if (bad) continue;
            const uint32_t kb = ring + st * L::kStage, vb = kb + L::kTile;
            const uint32_t vmask = s_vmask[warp * S + st];
            // S^T = K Q^T (16 tokens x 8 heads per n-tile)
            float sc[NH][4], sc2[NH][4];   // two independent accumulation chains (even / odd k)
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                sc2[nt][0] = sc2[nt][1] = sc2[nt][2] = sc2[nt][3] = 0.f;
            }
            if constexpr (F8) {
                // A fragments straight from the e4m3 rows g and g + 8: lane t4
                // holds bytes [t4 D/4, (t4+1) D/4) of each, four per k-step
                constexpr int F8CH = D / 64;
                uint32_t kw[2][KSTEPS];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int j = 0; j < F8CH; ++j) {
                        const uint4 v = ld_shared_v4(kb + L::off8(g + 8 * rr, t4 * F8CH + j));
                        kw[rr][4 * j] = v.x;
                        kw[rr][4 * j + 1] = v.y;
                        kw[rr][4 * j + 2] = v.z;
                        kw[rr][4 * j + 3] = v.w;
                    }
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    uint32_t af[4];
                    af[0] = e4m3x2_to_f16x2(kw[0][kk]);
                    af[1] = e4m3x2_to_f16x2(kw[1][kk]);
                    af[2] = e4m3x2_to_f16x2(kw[0][kk] >> 16);
                    af[3] = e4m3x2_to_f16x2(kw[1][kk] >> 16);
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt) {
                        if (kk & 1) mma_f16_16816(sc2[nt], af, qb[kk][nt][0], qb[kk][nt][1]);
                        else mma_f16_16816(sc[nt], af, qb[kk][nt][0], qb[kk][nt][1]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NH; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] += sc2[nt][e];
            } else {
                const int r = ((lane >> 3) & 1) * 8 + (lane & 7);
                const int c_hi = lane >> 4;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    uint32_t af[4];
                    ldmatrix_x4(kb + L::off(r, kk * 2 + c_hi), af[0], af[1], af[2], af[3]);
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt) {
                        if (kk & 1) mma_bf16_16816(sc2[nt], af, qb[kk][nt][0], qb[kk][nt][1]);
                        else mma_bf16_16816(sc[nt], af, qb[kk][nt][0], qb[kk][nt][1]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NH; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] += sc2[nt][e];
            }
            // mask, scale; column (head) maxima over the 16 tokens
            const bool ok0 = (vmask >> g) & 1u, ok1 = (vmask >> (g + 8)) & 1u;
            float mr[NH][2], al[NH][2];
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                if constexpr (F8) {
                    sc[nt][0] = ok0 ? sc[nt][0] * sl2_f8 : -INFINITY;
                    sc[nt][1] = ok0 ? sc[nt][1] * sl2_f8 : -INFINITY;
                    sc[nt][2] = ok1 ? sc[nt][2] * sl2_f8 : -INFINITY;
                    sc[nt][3] = ok1 ? sc[nt][3] * sl2_f8 : -INFINITY;
                } else {
                    sc[nt][0] = ok0 ? sc[nt][0] * a.scale_log2 : -INFINITY;
                    sc[nt][1] = ok0 ? sc[nt][1] * a.scale_log2 : -INFINITY;
                    sc[nt][2] = ok1 ? sc[nt][2] * a.scale_log2 : -INFINITY;
                    sc[nt][3] = ok1 ? sc[nt][3] * a.scale_log2 : -INFINITY;
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float v = fmaxf(sc[nt][j], sc[nt][j + 2]);
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                    const float mn = fmaxf(m[nt][j], v);
                    mr[nt][j] = mn == -INFINITY ? 0.f : mn;
                    al[nt][j] = ex2(m[nt][j] - mr[nt][j]);
                    m[nt][j] = mn;
                }
            }
            // P = exp2(s - m), lane-partial column sums, P^T fragments
            uint32_t pb[NH][2];
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                const float p0 = ex2(sc[nt][0] - mr[nt][0]);
                const float p1 = ex2(sc[nt][1] - mr[nt][1]);
                const float p2 = ex2(sc[nt][2] - mr[nt][0]);
                const float p3 = ex2(sc[nt][3] - mr[nt][1]);
                l[nt][0] = l[nt][0] * al[nt][0] + (p0 + p2);
                l[nt][1] = l[nt][1] * al[nt][1] + (p1 + p3);
                if constexpr (F8) {
                    pb[nt][0] = movmatrix_trans(pack_f16x2(p0, p1));
                    pb[nt][1] = movmatrix_trans(pack_f16x2(p2, p3));
                } else {
                    pb[nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));
                    pb[nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));
                }
            }
#pragma unroll
            for (int dm = 0; dm < DM; ++dm)
#pragma unroll
                for (int nt = 0; nt < NH; ++nt) {
                    o[dm][nt][0] *= al[nt][0];
                    o[dm][nt][1] *= al[nt][1];
                    o[dm][nt][2] *= al[nt][0];
                    o[dm][nt][3] *= al[nt][1];
                }
            // O^T += V^T P^T: V^T fragments by transposing ldmatrix of the V rows
            if constexpr (F8) {
                // widen the e4m3 V tile to f16 in the warp's staging tile (bf16
                // tile layout); the staging was last read before the previous
                // tile's closing __syncwarp
                constexpr int CPR8 = D / 16;
                const uint32_t stg = ring + S * L::kStage;
#pragma unroll
                for (int j = 0; j < kDecTile * CPR8 / 32; ++j) {
                    const int qc = j * 32 + lane, r = qc / CPR8, c = qc % CPR8;
                    const uint4 v = ld_shared_v4(vb + L::off8(r, c));
                    st_shared_v4(stg + L::off(r, 2 * c), e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16),
                                 e4m3x2_to_f16x2(v.y), e4m3x2_to_f16x2(v.y >> 16));
                    st_shared_v4(stg + L::off(r, 2 * c + 1), e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16),
                                 e4m3x2_to_f16x2(v.w), e4m3x2_to_f16x2(v.w >> 16));
                }
                __syncwarp();
                const int r = ((lane >> 4) & 1) * 8 + (lane & 7);
                const int c_lo = (lane >> 3) & 1;
#pragma unroll
                for (int dm = 0; dm < DM; ++dm) {
                    uint32_t af[4];
                    ldmatrix_x4_trans(stg + L::off(r, dm * 2 + c_lo), af[0], af[1], af[2], af[3]);
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt) mma_f16_16816(o[dm][nt], af, pb[nt][0], pb[nt][1]);
                }
            } else {
                const int r = ((lane >> 4) & 1) * 8 + (lane & 7);
                const int c_lo = (lane >> 3) & 1;
#pragma unroll
                for (int dm = 0; dm < DM; ++dm) {
                    uint32_t af[4];
                    ldmatrix_x4_trans(vb + L::off(r, dm * 2 + c_lo), af[0], af[1], af[2], af[3]);
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt) mma_bf16_16816(o[dm][nt], af, pb[nt][0], pb[nt][1]);
                }
            }
            __syncwarp();
        }

        if constexpr (F8) {
            const float vsc = __ldg(a.v_scale + I.h);
#pragma unroll
            for (int dm = 0; dm < DM; ++dm)
#pragma unroll
                for (int nt = 0; nt < NH; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[dm][nt][e] *= vsc;
        }
        // ------------------------------------- merge the warps' states
#pragma unroll
        for (int nt = 0; nt < NH; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 4);
                l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 8);
                l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 16);
            }
        // scratch free (the previous item is done with it); all warps stop
        // together if any ring wait timed out
        if (__syncthreads_or(bad)) break;
        if (ticket_pending) resolve_ticket();   // the previous item's split merge, if this CTA completed it
        ticket_pending = false;
        if (g == 0) {
#pragma unroll
            for (int nt = 0; nt < NH; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hd = nt * 8 + 2 * t4 + j;
                    if (hd < G) {
                        s_m[warp][hd] = m[nt][j];
                        s_l[warp][hd] = l[nt][j];
                    }
                }
        }
        // O states go through the scratch in one round when all eight warps'
        // G rows fit (G <= 4 NH), else in two (warps 0-3, then 4-7); either
        // way every element sums warps 0..7 in order with the same weights
        constexpr int EPT = (8 * NH * D + kDecThreads - 1) / kDecThreads;
        const bool one_round = G <= 4 * NH;
        const int wpr = one_round ? kDecWarps : kDecWarps / 2;   // warps per round
        float acc[EPT], lsum[EPT], Mx[EPT];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            if (rr == 1 && one_round) break;
            if (rr == 1) __syncthreads();   // round 0 readers are done with the scratch
            if (one_round || (warp >> 2) == rr) {
                const int wl = one_round ? warp : warp & 3;
#pragma unroll
                for (int dm = 0; dm < DM; ++dm)
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int hd = nt * 8 + 2 * t4 + (e & 1);
                            const int d = dm * 16 + g + 8 * (e >> 1);
                            if (hd < G) scratch[(wl * G + hd) * L::kCombineStride + d] = o[dm][nt][e];
                        }
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < EPT; ++k) {
                const int e = tid + k * kDecThreads;
                if (e >= G * D) continue;
                const int gg = e / D, d = e - gg * D;
                if (rr == 0) {
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w][gg]);
                    Mx[k] = M;
                    acc[k] = 0.f;
                    lsum[k] = 0.f;
                }
                const float Mr = Mx[k] == -INFINITY ? 0.f : Mx[k];
#pragma unroll
                for (int w = 0; w < kDecWarps; ++w) {
                    if (w >= wpr) break;
                    const int wg = rr * (kDecWarps / 2) + w;
                    const float wt = ex2(s_m[wg][gg] - Mr);
                    lsum[k] += wt * s_l[wg][gg];
                    acc[k] += wt * scratch[(w * G + gg) * L::kCombineStride + d];
                }
            }
        }
        const int pre_b = (MODE == MODE_SUFFIX && I.sb == 1) ? __ldcg(a.req_pre + I.b) : -1;
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int e = tid + k * kDecThreads;
            if (e >= G * D) continue;
            const int gg = e / D, d = e - gg * D;
            if (I.sb == 1) {
                if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8)
                    a.out[((int64_t)I.b * a.Hq + hq0 + gg) * D + d] =
                        __float2bfloat16_rn(lsum[k] > 0.f ? acc[k] / lsum[k] : 0.f);
                else
                    emit(I.b, hq0 + gg, d, acc[k], lsum[k], Mx[k], pre_b);
            } else {
                const int64_t pr = ((int64_t)I.s * a.cap_batch + I.b) * a.Hq + hq0 + gg;
                a.o_part[pr * D + d] = acc[k];
                if (d == 0) {
                    a.ml_part[pr * 2] = Mx[k];
                    a.ml_part[pr * 2 + 1] = lsum[k];
                }
            }
        }
        // deferred merge: the first split records the split count in the
        // (otherwise unused) ticket word, which the merge kernel reads and zeroes
        if constexpr (BAL) {
            if (a.defer_merge && I.sb > 1 && I.s == 0 && tid == 0) a.counters[I.b * Hkv + I.h] = I.sb;
        }
        if (I.sb > 1 && !a.defer_merge) {
            // ticket for (b, h): the barrier orders every thread's partial
            // stores before thread 0's acquire-release atomic (release: this
            // CTA's partials; acquire: those of the CTAs that came before, for
            // the one that completes the count); its result is only examined at
            // the next item end (or at exit), so the round trip overlaps the
            // next item's tiles
            __syncthreads();
            ticket_pending = true;
            if (tid == 0) {
                pend_prev = atom_add_acq_rel_gpu(a.counters + I.b * Hkv + I.h, 1);
                s_pend[0] = I.b;
                s_pend[1] = I.h;
                s_pend[2] = I.sb;
            }
        }
    }
    if (!bad && !*s_abort && ticket_pending) resolve_ticket();
    if (bad || *s_abort) {
        // aborted: let this warp's loads already in flight land before the
        // CTA's shared memory goes away (bounded, 10 ms per stage)
        for (int j = n_landed; j < n_issued; ++j) mbar_drain(bars + (j % S) * 8, (j / S) & 1);
    }
    if (ring_err) set_error(a.err, ring_err);
}

// Deferred split merge of a large batch.  The decode kernel wrote every
// split's partials and merged nothing: with many items per CTA, the CTA that
// completed a (request, kv head) last would merge it, and the merges piled up
// on the CTAs that were already behind.  This kernel merges every (request,
// kv head) of more than one split, one per CTA at a time, over the whole GPU,
// after the decode kernel (it waits for it first).  Each (request, kv head)'s
// split count is the one its first split recorded in the ticket word (the
// kernel zeroes the word again), so no plan is recomputed here; the
// arithmetic is the in-kernel merge's: split weights warp-parallel, each
// element summed in split order.
template <int D, int NH>
__global__ void __launch_bounds__(kDecThreads) paged_decode_merge_kernel(const __grid_constant__ DecodeArgs a)
{
    constexpr int GMAX = 8 * NH;
    constexpr int EPT = (GMAX * D + kDecThreads - 1) / kDecThreads;
    constexpr int SPL = kDecMaxSplits / 32;   // splits per lane
    __shared__ float s_w[kDecMaxSplits * GMAX];   // [split][head] weights
    __shared__ float s_lt[GMAX];                  // weighted sums of l
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.batch, Hkv = a.Hkv, G = a.G;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t split_stride = (int64_t)a.cap_batch * a.Hq * D;
    const int64_t ml_stride = (int64_t)a.cap_batch * a.Hq * 2;
    for (int p = blockIdx.x; p < B * Hkv; p += gridDim.x) {
        const int b = p / Hkv, h = p - b * Hkv;
        // the split count the decode kernel's first split recorded (0: one
        // split, written by the decode kernel itself)
        const int sb = __ldcg(a.counters + p);
        if (sb <= 1 || sb > a.max_splits) continue;
        const int hq0 = h * G;
        const float *obase = a.o_part + ((int64_t)b * a.Hq + hq0) * D;
        // the first splits' partials of this thread's elements, requested
        // before the (m, l) pairs (ordered loads: one round trip for both)
        constexpr int SB = 8;
        float v[EPT][SB];
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int e = tid + k * kDecThreads;
#pragma unroll
            for (int j = 0; j < SB; ++j) v[k][j] = ld_cg_ordered_if(e < G * D && j < sb, obase + e + j * split_stride);
        }
        for (int gg = warp; gg < G; gg += kDecWarps) {
            const float *ml = a.ml_part + ((int64_t)b * a.Hq + hq0 + gg) * 2;
            float mv[SPL], lv[SPL];
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < SPL; ++r) {
                const int ss = lane + 32 * r;
                mv[r] = ss < sb ? __ldcg(ml + ss * ml_stride) : -INFINITY;
                lv[r] = ss < sb ? __ldcg(ml + ss * ml_stride + 1) : 0.f;
                M = fmaxf(M, mv[r]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float Mr = M == -INFINITY ? 0.f : M;
            float lt = 0.f;
#pragma unroll
            for (int r = 0; r < SPL; ++r) {
                const int ss = lane + 32 * r;
                if (ss < sb) {
                    const float wt = ex2(mv[r] - Mr);
                    s_w[ss * G + gg] = wt;
                    lt += wt * lv[r];
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
            if (lane == 0) s_lt[gg] = lt;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int e = tid + k * kDecThreads;
            if (e >= G * D) continue;
            const int gg = e / D;
            float acc = 0.f;   // summed in split order
#pragma unroll
            for (int j = 0; j < SB; ++j)
                if (j < sb) acc += s_w[j * G + gg] * v[k][j];
            for (int ss = SB; ss < sb; ++ss) acc += s_w[ss * G + gg] * __ldcg(obase + e + ss * split_stride);
            const float lt = s_lt[gg];
            a.out[((int64_t)b * a.Hq + hq0) * D + e] = __float2bfloat16_rn(lt > 0.f ? acc / lt : 0.f);
        }
        __syncthreads();   // s_w, s_lt reuse; every thread has read the count
        if (tid == 0) a.counters[p] = 0;
    }
}

template <int D, int S, int NH, int MODE, bool BAL = false>
static pa_status launch_decode(const DecodeArgs &a, cudaStream_t st)
{
    auto kern = paged_decode_kernel<D, S, NH, MODE, BAL>;
    const size_t smem = DecSmem<D, S, NH, MODE == MODE_FP8>::bytes(a.batch);
    if (smem > kSmemLimit) return PA_ERR_UNSUPPORTED;
    if (!ensure_dynamic_smem(reinterpret_cast<const void *>(kern), smem)) return PA_ERR_CUDA;
    if (launch_kernel(kern, dim3(num_sms()), dim3(kDecThreads), smem, st, a) != cudaSuccess) return PA_ERR_CUDA;
    if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8) {
        if (a.defer_merge) {
            const int pairs = a.batch * a.Hkv, cap = 8 * num_sms();
            if (launch_kernel(paged_decode_merge_kernel<D, NH>, dim3(pairs < cap ? pairs : cap), dim3(kDecThreads), 0,
                              st, a) != cudaSuccess)
                return PA_ERR_CUDA;
        }
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Deepest ring whose shared memory fits this batch.
template <int D, int NH, int MODE>
static pa_status dispatch_decode(const DecodeArgs &a, cudaStream_t st)
{
    constexpr bool kCanBal = MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8;
    if constexpr (kCanBal) {
        // large batches (merges deferred): the instance with the balanced plan
        if (a.defer_merge) {
            if constexpr (MODE == MODE_FP8) {
                if (DecSmem<D, 5, NH, true>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 5, NH, MODE, true>(a, st);
                if (DecSmem<D, 4, NH, true>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 4, NH, MODE, true>(a, st);
                return launch_decode<D, 2, NH, MODE, true>(a, st);
            } else {
                if (DecSmem<D, 4, NH>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 4, NH, MODE, true>(a, st);
                if (DecSmem<D, 3, NH>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 3, NH, MODE, true>(a, st);
                return launch_decode<D, 2, NH, MODE, true>(a, st);
            }
        }
    }
    if constexpr (MODE == MODE_FP8) {
        // stages of half the bytes: a deeper ring keeps as many bytes in flight
        if (DecSmem<D, 5, NH, true>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 5, NH, MODE>(a, st);
        if (DecSmem<D, 4, NH, true>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 4, NH, MODE>(a, st);
        return launch_decode<D, 2, NH, MODE>(a, st);
    } else {
        if (DecSmem<D, 4, NH>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 4, NH, MODE>(a, st);
        if (DecSmem<D, 3, NH>::bytes(a.batch) <= kSmemLimit) return launch_decode<D, 3, NH, MODE>(a, st);
        return launch_decode<D, 2, NH, MODE>(a, st);
    }
}
static_assert(DecSmem<128, 2, 2>::bytes(kDecMaxBatch) <= kSmemLimit, "decode smem at the largest batch");
static_assert(DecSmem<128, 2, 2, true>::bytes(kDecMaxBatch) <= kSmemLimit, "fp8 decode smem at the largest batch");



// Inputs of the fused step that a plain decode call does not have.
struct StepInputs {
    const void *k_new, *v_new;
    const int32_t *positions, *loc;
    const float *cos_tab, *sin_tab;
    int max_pos;
};

// Validation of the arguments every decode entry point shares (ranges,
// supported shapes, null pointers, alignment); the workspace is checked by
// the caller of this function.  Touches no CUDA state.
static pa_status check_decode_args(const void *q, int batch, int n_q_heads, const void *k_buf, const void *v_buf,
                                   pa_kv_shape s, int layer_id, const int32_t *req_to_token, int req_rows,
                                   int max_ctx, const int32_t *req_pool_indices, const int32_t *seq_lens,
                                   int max_splits, void *out)
{
    if (batch < 0 || batch > kDecMaxBatch || n_q_heads <= 0 || s.n_layers <= 0 || s.size <= 0 ||
        s.n_kv_heads <= 0 || req_rows <= 0 || max_ctx <= 0 || max_splits < 1 || max_splits > kDecMaxSplits)
        return PA_ERR_SHAPE;
    if (layer_id < 0 || layer_id >= s.n_layers) return PA_ERR_SHAPE;
    if (n_q_heads % s.n_kv_heads != 0) return PA_ERR_SHAPE;
    const int G = n_q_heads / s.n_kv_heads;
    if (G > 16 || (s.head_dim != 64 && s.head_dim != 128)) return PA_ERR_UNSUPPORTED;
    if ((int64_t)s.n_layers * s.size >= (int64_t)INT32_MAX - 16) return PA_ERR_SHAPE;
    if (batch == 0) return PA_OK;
    if (!q || !k_buf || !v_buf || !req_to_token || !req_pool_indices || !seq_lens || !out) return PA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_buf) || !aligned16(v_buf) || !aligned16(out) || !aligned4(req_to_token) ||
        !aligned4(req_pool_indices) || !aligned4(seq_lens))
        return PA_ERR_ALIGN;
    return PA_OK;
}

// Validation shared by the workspace entry points: the arguments, then the
// workspace pointer.
static pa_status check_decode(const void *q, int batch, int n_q_heads, const void *k_buf, const void *v_buf,
                              pa_kv_shape s, int layer_id, const int32_t *req_to_token, int req_rows, int max_ctx,
                              const int32_t *req_pool_indices, const int32_t *seq_lens, void *workspace,
                              int max_splits, void *out)
{
    // the workspace checks come first for an empty batch, as before
    const pa_status rc = check_decode_args(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows,
                                           max_ctx, req_pool_indices, seq_lens, max_splits, out);
    if (rc != PA_OK && rc != PA_ERR_NULL && rc != PA_ERR_ALIGN) return rc;
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    return rc;
}

// Launch arguments for `batch` requests of `n_q_heads` heads whose split
// partials live in the decode layout `ws` at `wbase`; errors go to `err`.
static bool fill_decode_args(DecodeArgs &a, const void *q, int batch, int n_q_heads, const void *k_buf,
                             const void *v_buf, pa_kv_shape s, int layer_id, const int32_t *req_to_token,
                             int req_rows, int max_ctx, const int32_t *req_pool_indices, const int32_t *seq_lens,
                             float scale, int max_splits, void *out, int32_t *err, const DecodeWsLayout &ws,
                             unsigned char *wbase, bool bf16_cache = true)
{
    memset(&a, 0, sizeof a);
    const cuuint64_t dims[2] = {(cuuint64_t)s.n_kv_heads * s.head_dim, (cuuint64_t)s.n_layers * s.size};
    const cuuint64_t strides[1] = {(cuuint64_t)s.n_kv_heads * s.head_dim * 2};
    const cuuint32_t box[2] = {64, kDecTile};
    if (bf16_cache && (!encode_tmap_bf16(&a.tm_k, k_buf, 2, dims, strides, box) ||
                       !encode_tmap_bf16(&a.tm_v, v_buf, 2, dims, strides, box)))
        return false;
    a.layer_row0 = layer_id * s.size;
    const int64_t layer_off = (int64_t)layer_id * s.size * s.n_kv_heads * s.head_dim;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k_layer = static_cast<const __nv_bfloat16 *>(k_buf) + layer_off;
    a.v_layer = static_cast<const __nv_bfloat16 *>(v_buf) + layer_off;
    a.req_to_token = req_to_token;
    a.req_pool_indices = req_pool_indices;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    a.counters = reinterpret_cast<int32_t *>(wbase + ws.counters_off);
    a.ml_part = reinterpret_cast<float *>(wbase + ws.ml_off);
    a.o_part = reinterpret_cast<float *>(wbase + ws.o_off);
    a.batch = batch;
    a.Hq = n_q_heads;
    a.Hkv = s.n_kv_heads;
    a.G = n_q_heads / s.n_kv_heads;
    a.size = s.size;
    a.req_rows = req_rows;
    a.max_ctx = max_ctx;
    a.cap_batch = ws.cap_batch;
    a.max_splits = max_splits;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    a.early_meta = early_metadata();
    a.early_kv = launch_overlap() == PA_OVERLAP_EARLY_KV;
    a.wait_ns = wait_limit_ns();
    return true;
}

template <int MODE>
static pa_status dispatch_mode(const DecodeArgs &a0, int head_dim, cudaStream_t st)
{
    DecodeArgs a = a0;
    if constexpr (MODE == MODE_PLAIN || MODE == MODE_FUSED || MODE == MODE_FP8) {
        // more (request, kv head) pairs than half the CTAs: many items per CTA,
        // merged by the second kernel
        a.defer_merge = 2 * a.batch * a.Hkv > num_sms();
    }
    if (head_dim == 128) return a.G > 8 ? dispatch_decode<128, 2, MODE>(a, st) : dispatch_decode<128, 1, MODE>(a, st);
    return a.G > 8 ? dispatch_decode<64, 2, MODE>(a, st) : dispatch_decode<64, 1, MODE>(a, st);
}

template <int MODE>
static pa_status decode_call(const void *q, int batch, int n_q_heads, const void *k_buf, const void *v_buf,
                             pa_kv_shape s, int layer_id, const int32_t *req_to_token, int req_rows, int max_ctx,
                             const int32_t *req_pool_indices, const int32_t *seq_lens, float scale, void *workspace,
                             size_t workspace_bytes, int max_splits, void *out, const StepInputs *step,
                             cudaStream_t st)
{
    pa_status rc = check_decode(q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                                req_pool_indices, seq_lens, workspace, max_splits, out);
    if (rc != PA_OK) return rc;
    if (step && step->max_pos <= 0) return PA_ERR_SHAPE;
    const DecodeWsLayout ws = decode_ws_layout(workspace_bytes, n_q_heads, s.n_kv_heads, s.head_dim, max_splits);
    if (ws.cap_batch < batch || ws.total > workspace_bytes) return PA_ERR_WORKSPACE;
    if (batch == 0) return PA_OK;
    if (step) {
        if (!step->k_new || !step->v_new || !step->positions || !step->loc || !step->cos_tab || !step->sin_tab)
            return PA_ERR_NULL;
        if (!aligned16(step->k_new) || !aligned16(step->v_new) || !aligned4(step->positions) ||
            !aligned4(step->loc) || !aligned16(step->cos_tab) || !aligned16(step->sin_tab))
            return PA_ERR_ALIGN;
    }
    unsigned char *w = static_cast<unsigned char *>(workspace);
    DecodeArgs a;
    if (!fill_decode_args(a, q, batch, n_q_heads, k_buf, v_buf, s, layer_id, req_to_token, req_rows, max_ctx,
                          req_pool_indices, seq_lens, scale, max_splits, out, reinterpret_cast<int32_t *>(w), ws, w))
        return PA_ERR_CUDA;
    if (step) {
        const int64_t layer_off = (int64_t)layer_id * s.size * s.n_kv_heads * s.head_dim;
        a.k_new = static_cast<const __nv_bfloat16 *>(step->k_new);
        a.v_new = static_cast<const __nv_bfloat16 *>(step->v_new);
        a.positions = step->positions;
        a.loc = step->loc;
        a.cos_tab = step->cos_tab;
        a.sin_tab = step->sin_tab;
        a.max_pos = step->max_pos;
        a.k_layer_w = static_cast<__nv_bfloat16 *>(const_cast<void *>(k_buf)) + layer_off;
        a.v_layer_w = static_cast<__nv_bfloat16 *>(const_cast<void *>(v_buf)) + layer_off;
    }
    return dispatch_mode<MODE>(a, s.head_dim, st);
}

}  // namespace pa

/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * The calls follow the hot path described on the AstrAI commit pages:
 *   - commit 398e8a3 (tests/inference/test_cache.py): inference on packed 3-D
 *     [tokens, heads, head_dim] tensors; rotary embedding on packed inputs;
 *     int32 page-table, request-row and cache-location indices; K/V stored at
 *     buffer[layer_id, loc] of per-layer [n_layers, size, n_kv_heads, head_dim]
 *     buffers; split-KV decode into workspace-owned partials (decode_o_part,
 *     decode_ml_part) pre-allocated once, zero allocation in the decode loop, so
 *     every address is stable under CUDA-graph capture;
 *   - commit e58a728 (docs/developer/architecture.md): rotary from a real cos/sin
 *     table; prompts packed into one forward and addressed by cumulative query
 *     lengths (qo_indptr); paged prefill (attn_paged_prefill); decode reading
 *     K/V through req_to_token.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     row-major, with 16-byte aligned base addresses.  bf16 data travel as
 *     IEEE bfloat16 (2 bytes), indices as int32, tables and workspaces as fp32;
 *     the fp8 entry points' caches as one e4m3 byte per element with fp32
 *     per-(layer, kv head) scales.
 *   - The library allocates nothing, keeps no per-call state and never
 *     synchronises the stream (pa_get_error excepted).  Work is enqueued on the
 *     given stream; every call except pa_get_error can be captured in a CUDA
 *     graph, since grid shapes depend only on call arguments and workspace
 *     capacity, never on device-resident lengths.
 *   - Validation first: every host-side check runs before any launch, and a
 *     call that returns an error has enqueued nothing and written nothing.
 *   - Device-side index errors (a cache slot, request row or position out of
 *     range) never trap: the offending element is skipped (treated as masked,
 *     or left unwritten) and a sticky bit is OR-ed into a device error word,
 *     read outside the hot loop with pa_get_error.
 *   - Return values are pa_status codes; PA_ERR_CUDA means a launch failed
 *     (cudaGetLastError after the launch).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = 1,         /* a required pointer is NULL */
    PA_ERR_SHAPE = 2,        /* a size, count or index argument is out of range */
    PA_ERR_ALIGN = 3,        /* a pointer is not 16-byte (workspace: 256-byte) aligned */
    PA_ERR_UNSUPPORTED = 4,  /* head_dim / GQA group not supported by the kernels */
    PA_ERR_WORKSPACE = 5,    /* workspace too small for this call */
    PA_ERR_CUDA = 6,         /* a CUDA runtime / driver call failed */
    PA_ERR_DEVICE_INDEX = 7  /* (pa_get_error only) the device error word is non-zero */
} pa_status;

/* Bits of the device error word. */
#define PA_DEVERR_SLOT 0x1      /* a cache slot (loc or req_to_token entry) outside [0, size) */
#define PA_DEVERR_ROW 0x2       /* a req_pool_indices entry outside [0, req_rows) */
#define PA_DEVERR_LEN 0x4       /* a seq_len / indptr length outside [0, max_ctx] or n_r > L_r */
#define PA_DEVERR_POS 0x8       /* a rotary position outside [0, max_pos) */
#define PA_DEVERR_TIMEOUT 0x10  /* a bounded pipeline wait gave up (internal error); the call aborted */

/* Shape of one of the two KV buffers, bf16 [n_layers, size, n_kv_heads, head_dim];
 * slot `loc` of layer `l` starts at element ((l * size + loc) * n_kv_heads) * head_dim. */
typedef struct {
    int n_layers;
    int size;        /* slots per layer */
    int n_kv_heads;
    int head_dim;
} pa_kv_shape;

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status s);

/* ------------------------------------------------------- launch overlap
 * Programmatic dependent launch lets a call's kernel start while the kernel
 * before it on the stream finishes: its CTAs take SMs as the earlier kernel's
 * CTAs leave, set up shared memory and barriers, and then wait for the earlier
 * kernel's writes before touching anything it may have written.  Each kernel
 * lets its successor start only after its own wait, so the overlap never
 * reaches back further than one kernel.  Process-wide setting, read at each
 * call (and frozen into a graph at capture):
 *   PA_OVERLAP_OFF  (default) plain launches.
 *   PA_OVERLAP_SAFE  overlap; a kernel reads no global memory before its wait.
 *     Correct in any stream.
 *   PA_OVERLAP_EARLY_METADATA  overlap, and the index inputs -- seq_lens,
 *     req_pool_indices, req_to_token, qo_indptr, kv_indptr, positions, loc --
 *     are read before the wait (the decode and prefill work plans and the
 *     first page-table entries are ready when the earlier kernel ends).  The
 *     caller guarantees that the kernel launched immediately before a call on
 *     its stream does not write those index arrays.  Data (q, k, v, caches,
 *     tables, workspace, out) are always read after the wait.
 *   PA_OVERLAP_EARLY_KV  early metadata, and decode attention (plain, fused
 *     step, fp8) also starts copying K/V cache rows before the wait: every
 *     row except each request's newest one (position seq_lens[b] - 1), which
 *     is read after the wait (the fused step takes it from k_new / v_new).  The caller guarantees that the kernel launched
 *     immediately before a decode call writes no cache row of that call's
 *     layer other than the requests' newest rows (true in a decode step,
 *     where that kernel is the new token's projection, RoPE or KV store, or
 *     another layer's attention).  Other calls behave as in early-metadata
 *     mode. */
#define PA_OVERLAP_OFF 0
#define PA_OVERLAP_SAFE 1
#define PA_OVERLAP_EARLY_METADATA 2
#define PA_OVERLAP_EARLY_KV 3
/* PA_ERR_SHAPE for an unknown mode. */
pa_status pa_set_launch_overlap(int mode);
int pa_get_launch_overlap(void);

/* ------------------------------------------------------ wait time limit
 * Every pipeline wait inside the kernels (a warp waiting for copies or
 * tensor-core work of its own CTA) gives up after a time limit: the CTA then
 * sets PA_DEVERR_TIMEOUT, lets the copies and MMAs it has issued finish,
 * frees its tensor memory and exits, so a stuck pipeline ends the call with
 * an error instead of a hang.  The limit is process-wide, read at each call
 * (and frozen into a graph at capture); the default is 2 s.  Setting 0 makes
 * each decode or prefill CTA give up at its first work item, exactly as if a
 * wait had timed out there: a test hook that drives the abort path without
 * any fault.  Restore the default (2000000000) afterwards. */
void pa_set_wait_timeout_ns(uint64_t ns);
uint64_t pa_get_wait_timeout_ns(void);

/* ----------------------------------------------------------- workspaces
 * A workspace is one caller-allocated device buffer, 256-byte aligned.  Its
 * first 4 bytes are the device error word.  Initialise it once with
 * pa_workspace_init before first use (it zeroes the error word and the decode
 * merge counters, which the decode kernels afterwards return to zero
 * themselves: the merge tickets, or for large batches the split counts that
 * the merge kernel reads).
 *
 * Decode layout, derived only from (workspace_bytes, n_q_heads, n_kv_heads,
 * head_dim, max_splits), so changing the batch between calls moves nothing:
 *   [0, 256)   error word + padding
 *   counters   int32 [cap_batch * n_kv_heads]  (one per request x kv head)
 *   ml_part    fp32  [max_splits, cap_batch, n_q_heads, 2]   (running max in
 *              log2 units, running sum) -- the pages' decode_ml_part
 *   o_part     fp32  [max_splits, cap_batch, n_q_heads, head_dim]  unnormalised
 *              partial outputs -- the pages' decode_o_part
 * where cap_batch is the largest batch the bytes hold. */
size_t pa_decode_workspace_bytes(int max_batch, int n_q_heads, int n_kv_heads, int head_dim,
                                 int max_splits);

/* Prefill workspace: the error word plus the prefill work queue, two int32
 * words inside the 256-byte header (the next work item to claim and the number
 * of CTAs that have finished; the kernel returns both to zero before it ends).
 * A decode workspace also serves prefill.  A workspace serves one call at a
 * time: calls that share one must be ordered on a stream. */
size_t pa_prefill_workspace_bytes(void);

/* Zero the whole workspace on `st` (cudaMemsetAsync).  Call once after
 * allocation, outside any graph capture that replays it while work is in flight. */
pa_status pa_workspace_init(void *workspace, size_t workspace_bytes, cudaStream_t st);

/* Copy the workspace's device error word to *device_error.  Synchronises `st`
 * (keep it out of the hot loop and out of graph capture).  Returns
 * PA_ERR_DEVICE_INDEX if the word is non-zero, PA_OK otherwise.  The word is
 * sticky: pa_workspace_init clears it.  After PA_DEVERR_TIMEOUT the aborted
 * call may have left decode merge counters non-zero: call pa_workspace_init
 * before the workspace is used again (index-error bits alone leave the
 * counters intact). */
pa_status pa_get_error(const void *workspace, int32_t *device_error, cudaStream_t st);

/* Same, for a bare int32 error word passed to pa_kv_store / pa_rope_packed. */
pa_status pa_get_error_word(const int32_t *error_word, int32_t *device_error, cudaStream_t st);

/* --------------------------------------------------------------- KV store
 * Commit 398e8a3: new tokens' K/V written at buffer[layer_id, loc] with int32
 * cache locations.  For every token t < n_tokens and kv head h:
 *     k_buf[layer_id, loc[t], h, :] = k_new[t, h, :]
 *     v_buf[layer_id, loc[t], h, :] = v_new[t, h, :]
 * A bit-exact copy.  k_new / v_new: bf16 [n_tokens, n_kv_heads, head_dim];
 * loc: int32 [n_tokens].  head_dim must be a multiple of 8.  Locations must be
 * distinct within one call (duplicates race).  A location outside [0, size)
 * is skipped and sets PA_DEVERR_SLOT in *error_word (if error_word != NULL).
 * n_tokens == 0 is a no-op. */
pa_status pa_kv_store(void *k_buf, void *v_buf, pa_kv_shape s, int layer_id, const void *k_new,
                      const void *v_new, const int32_t *loc, int n_tokens, int32_t *error_word,
                      cudaStream_t st);

/* ----------------------------------------------------------------- RoPE
 * Commit 398e8a3 (rotary extended to packed 3-D inputs) and commit e58a728
 * (cos/sin table, not a complex buffer).  In place on q bf16
 * [n_tokens, n_q_heads, head_dim] and k bf16 [n_tokens, n_kv_heads, head_dim]
 * (k may be NULL when n_kv_heads == 0).  For token t with p = positions[t]
 * and pair i < head_dim/2 (interleaved pairs (2i, 2i+1)):
 *     x[2i]   <- x[2i] * cos_tab[p, i] - x[2i+1] * sin_tab[p, i]
 *     x[2i+1] <- x[2i] * sin_tab[p, i] + x[2i+1] * cos_tab[p, i]
 * in fp32, rounded to bf16 (nearest even).  cos_tab / sin_tab: fp32
 * [max_pos, head_dim/2].  head_dim must be a multiple of 8.  A position outside
 * [0, max_pos) leaves that token unchanged and sets PA_DEVERR_POS. */
pa_status pa_rope_packed(void *q, int n_q_heads, void *k, int n_kv_heads, int head_dim,
                         const int32_t *positions, int n_tokens, const float *cos_tab,
                         const float *sin_tab, int max_pos, int32_t *error_word, cudaStream_t st);

/* ------------------------------------------------------------ decode attn
 * Commit 398e8a3: packed decode over the paged cache with int32 indices and
 * split-KV partials in a caller workspace; commit e58a728: K/V read through
 * req_to_token.  For request b < batch with n = seq_lens[b] and
 * row = req_pool_indices[b], and query head hq with kv head h = hq / G
 * (G = n_q_heads / n_kv_heads):
 *     s_j   = scale * <q[b, hq, :], K[layer_id, req_to_token[row, j], h, :]>, j < n
 *     out[b, hq, :] = sum_j softmax(s)_j * V[layer_id, req_to_token[row, j], h, :]
 * q, out: bf16 [batch, n_q_heads, head_dim]; req_to_token: int32
 * [req_rows, max_ctx]; req_pool_indices, seq_lens: int32 [batch] (device).
 * seq_lens counts the current token, whose K/V must already be stored.
 * n == 0 writes zeros.  Entries req_to_token[row, j >= n] are never read.
 * Computed as split-KV flash-decoding: each (request, kv head) range is cut
 * into at most max_splits pieces, chosen on the device from seq_lens and the
 * SM count, whose fp32 partials (o_part, ml_part) are merged by log-sum-exp in
 * a fixed order (run-to-run bit-identical).  With at most half as many
 * (request, kv head) pairs as SMs, the merge runs inside the one decode
 * kernel (the CTA that completes a pair merges it).  A larger batch is two
 * kernels on `st`: decode, which writes every split's partials, then a merge
 * kernel spread over the whole GPU (it writes only out).  For such a batch
 * every CTA takes an equal range of 16-token tiles over the (kv head,
 * request) pairs, a pair's pieces being its splits (a pair that would need
 * more than max_splits pieces falls back to splits of a common length).  This
 * also holds for pa_decode_step and pa_paged_decode_attn_fp8.
 * Supported: head_dim in {64, 128}; 1 <= G <= 16; 1 <= max_splits <= 128;
 * batch <= 4096 and <= the workspace's cap_batch for these head counts and
 * max_splits.  A 16-token tile whose positions sit on one page moves as TMA
 * boxes, any other tile as 16-byte cp.async rows: k_buf and v_buf must be
 * 16-byte aligned, which with head_dim 64/128 makes every row 16-byte
 * aligned. */
pa_status pa_paged_decode_attn(const void *q, int batch, int n_q_heads, const void *k_buf,
                               const void *v_buf, pa_kv_shape s, int layer_id,
                               const int32_t *req_to_token, int req_rows, int max_ctx,
                               const int32_t *req_pool_indices, const int32_t *seq_lens,
                               float scale, void *workspace, size_t workspace_bytes,
                               int max_splits, void *out, cudaStream_t st);

/* ------------------------------------------- decode attn, no allocation
 * No counterpart on the pages: an addition for callers that cannot hand the
 * library a workspace.  Some callers have no way to allocate device memory
 * at the point where decode runs -- a plugin inside a host program that owns
 * every device allocation, or a serving loop that forbids cudaMalloc because
 * it synchronises the device and stalls every stream -- and this entry point
 * serves them.  It computes exactly what pa_paged_decode_attn computes (same
 * arguments, same results bit for bit for the same max_splits), but its
 * scratch (split partials, merge tickets, error word) is a fixed 16 MiB array
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing itself and calls no allocating routine.
 *   - Size limit: the partials of `batch` requests must fit the 16 MiB:
 *     16 MiB >= 1024 + batch * (n_kv_heads*4 + max_splits*n_q_heads*(head_dim+2)*4)
 *     (e.g. 15 requests at Hq=32, head_dim 128, max_splits 64); larger calls
 *     return PA_ERR_WORKSPACE.
 *   - Every argument check (those of pa_paged_decode_attn, the size limit,
 *     error_word's alignment) runs before the first CUDA call: a call that
 *     returns an error has enqueued nothing and written nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call clears the error word and the merge tickets on `st` before
 *     its kernel, so a call never sees the previous call's state; the array
 *     otherwise keeps the last call's contents.  All calls on all streams of a
 *     device share the one array: calls that may overlap on the GPU race and
 *     must be serialised by the caller (e.g. one stream).
 *   - error_word (device pointer, may be NULL) receives a copy of the call's
 *     device error word (PA_DEVERR_* bits) on `st`. */
pa_status pa_paged_decode_attn_noalloc(const void *q, int batch, int n_q_heads, const void *k_buf,
                                       const void *v_buf, pa_kv_shape s, int layer_id,
                                       const int32_t *req_to_token, int req_rows, int max_ctx,
                                       const int32_t *req_pool_indices, const int32_t *seq_lens,
                                       float scale, int max_splits, void *out, int32_t *error_word,
                                       cudaStream_t st);

/* ------------------------------------------------------- fp8 (e4m3) cache
 * Commit e58a728 (docs/developer/architecture.md) names an fp8 test among the
 * CUDA kernel sources and says nothing else about fp8; the scheme is this
 * library's reading.  An fp8 cache holds each K/V element as one OCP E4M3
 * byte (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest finite
 * 448; S.1111.111 is NaN) in uint8 buffers [n_layers, size, n_kv_heads,
 * head_dim].  k_scale and v_scale are fp32 [n_layers, n_kv_heads] device
 * arrays owned by the caller (static, per-head calibration is the caller's
 * business); element x of kv head h in layer l is stored as
 *     byte = e4m3( fp32(x) / scale[l, h] )   (IEEE fp32 division; round to
 *            nearest, ties to even; finite overflow saturates to +-448)
 * and read back as e4m3_value(byte) * scale[l, h].
 *
 * pa_kv_store_fp8: as pa_kv_store, quantising.  k_new / v_new bf16
 * [n_tokens, n_kv_heads, head_dim]; head_dim a multiple of 16; buffers 16-byte
 * aligned.  Same location checks and error word as pa_kv_store. */
pa_status pa_kv_store_fp8(void *k_buf, void *v_buf, pa_kv_shape s, int layer_id, const void *k_new,
                          const void *v_new, const int32_t *loc, int n_tokens, const float *k_scale,
                          const float *v_scale, int32_t *error_word, cudaStream_t st);

/* pa_paged_decode_attn_fp8: pa_paged_decode_attn over an fp8 cache -- the
 * same arguments, workspace, split plan, limits and error reporting, plus the
 * two scale arrays; k_buf / v_buf are the uint8 buffers.  Key j of kv head h
 * is e4m3_value(K[layer_id, slot_j, h, :]) * k_scale[layer_id, h], value rows
 * likewise with v_scale.  Rows move as 16-byte cp.async copies.  The dot
 * products run on f16 tensor-core MMAs with fp32 accumulation: q is rounded
 * to f16 (exact for bf16 values of magnitude 2^-14 .. 65504; larger ones are
 * clamped to +-65504), keys and values are exact in f16, the softmax weights
 * are rounded to f16. */
pa_status pa_paged_decode_attn_fp8(const void *q, int batch, int n_q_heads, const void *k_buf,
                                   const void *v_buf, pa_kv_shape s, int layer_id,
                                   const int32_t *req_to_token, int req_rows, int max_ctx,
                                   const int32_t *req_pool_indices, const int32_t *seq_lens,
                                   float scale, const float *k_scale, const float *v_scale,
                                   void *workspace, size_t workspace_bytes, int max_splits, void *out,
                                   cudaStream_t st);

/* pa_paged_prefill_attn_fp8: pa_paged_prefill_attn over an fp8 cache -- the
 * same arguments, workspace, limits (head_dim 64 or 128, G in {1, 2, 4, 8,
 * 16}) and error reporting, plus the two scale arrays; k_buf / v_buf are the
 * uint8 buffers.  Key j of kv head h is e4m3_value(K[layer_id, slot_j, h, :])
 * * k_scale[layer_id, h], value rows likewise with v_scale.  The e4m3 tiles
 * are widened to bf16 in shared memory (exact) before the tcgen05 MMAs, so q
 * stays bf16 and the arithmetic is that of pa_paged_prefill_attn: the K scale
 * joins the softmax scale and the V scale multiplies each output row. */
pa_status pa_paged_prefill_attn_fp8(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                    const void *v_buf, pa_kv_shape s, int layer_id, const int32_t *qo_indptr,
                                    const int32_t *kv_indptr, int n_reqs, const int32_t *req_to_token, int req_rows,
                                    int max_ctx, const int32_t *req_pool_indices, float scale, const float *k_scale,
                                    const float *v_scale, void *workspace, size_t workspace_bytes, void *out,
                                    cudaStream_t st);

/* ------------------------------------------------------ fused decode step
 * One layer's decode step in one launch (commit 398e8a3: the CUDA-graph
 * decode step over packed inputs, rotary embedding on packed 3-D inputs, K/V
 * stored at buffer[layer_id, loc]).  Same results, bit for bit, as
 *     pa_rope_packed(q', k', positions, cos_tab, sin_tab)   on copies q', k'
 *     pa_kv_store(k_buf, v_buf, layer_id, k', v_new, loc)
 *     pa_paged_decode_attn(q', ...)
 * with one new token per request:
 *   q: bf16 [batch, n_q_heads, head_dim]; k_new, v_new: bf16 [batch,
 *   n_kv_heads, head_dim]; q and k_new are only read (the rotated q stays in
 *   registers, the rotated k goes to the cache).
 *   positions: int32 [batch], the new token's rotary position; cos_tab,
 *   sin_tab: fp32 [max_pos, head_dim / 2].
 *   loc: int32 [batch], the new token's slot.  It must be the request's last
 *   position, loc[b] == req_to_token[req_pool_indices[b], seq_lens[b] - 1]:
 *   attention takes that row from k_new / v_new (rotated), not from the
 *   cache, and no other request may list the slot.  A mismatch sets
 *   PA_DEVERR_SLOT (the row is still written at loc[b]; attention then reads
 *   the table's slot from the cache).
 *   k_buf, v_buf: written at [layer_id, loc[b]]; the other rows are read.
 * Everything else, the workspace and the limits are those of
 * pa_paged_decode_attn.  A position outside [0, max_pos) sets PA_DEVERR_POS
 * and leaves that token's q and k unrotated, as pa_rope_packed does. */
pa_status pa_decode_step(const void *q, const void *k_new, const void *v_new, int batch, int n_q_heads,
                         const int32_t *positions, const float *cos_tab, const float *sin_tab, int max_pos,
                         void *k_buf, void *v_buf, pa_kv_shape s, int layer_id, const int32_t *loc,
                         const int32_t *req_to_token, int req_rows, int max_ctx,
                         const int32_t *req_pool_indices, const int32_t *seq_lens, float scale,
                         void *workspace, size_t workspace_bytes, int max_splits, void *out, cudaStream_t st);

/* ------------------------------------------------------- cascade decode
 * Shared-prefix decode (commit 398e8a3 / e58a728: requests whose page-table
 * rows point at the same cached prefix pages, radix reuse).  The members of
 * group g are the requests group_reqs[group_indptr[g] .. group_indptr[g+1]),
 * and the first group_prefix[g] tokens of every member sit on the same slots
 * (the caller's contract; each member is in at most one group and
 * group_prefix[g] < its seq_len).  Same result as pa_paged_decode_attn, within
 * the attention tolerance (the split structure differs): the prefix is read
 * once per chunk of 16 / G members, its rows merged with each member's own
 * tokens by log-sum-exp.  Two kernel launches.
 *   group_indptr int32 [n_groups + 1], group_reqs int32 [group_indptr[n_groups]],
 *   group_prefix int32 [n_groups] (device); members past max_group_size in a
 *   group are treated as ungrouped.
 * The workspace layout is fixed by `caps`, which must be the same for every
 * call on one workspace (sized by pa_cascade_workspace_bytes, initialised by
 * pa_workspace_init); batch <= caps.max_batch, n_groups <= caps.max_groups,
 * caps.max_groups * ceil(max_group_size / (16 / G)) <= 4096.  Other limits as
 * pa_paged_decode_attn.  Under PA_OVERLAP_EARLY_METADATA the group arrays
 * count as index inputs. */
typedef struct {
    int max_batch, max_groups, max_group_size, max_splits;
} pa_cascade_caps;
size_t pa_cascade_workspace_bytes(pa_cascade_caps caps, int n_q_heads, int n_kv_heads, int head_dim);
pa_status pa_paged_decode_attn_cascade(const void *q, int batch, int n_q_heads, const void *k_buf,
                                       const void *v_buf, pa_kv_shape s, int layer_id,
                                       const int32_t *req_to_token, int req_rows, int max_ctx,
                                       const int32_t *req_pool_indices, const int32_t *seq_lens,
                                       const int32_t *group_indptr, const int32_t *group_reqs,
                                       const int32_t *group_prefix, int n_groups, pa_cascade_caps caps,
                                       float scale, void *workspace, size_t workspace_bytes, void *out,
                                       cudaStream_t st);

/* ----------------------------------------------------------- prefill attn
 * Commit e58a728: packed prompts with a shared prefix start in one forward,
 * paged prefill (attn_paged_prefill), rows located by cumulative query lengths;
 * commit 398e8a3: request mappings for cached prefix pages.  Request r owns
 * packed query rows qo_indptr[r] .. qo_indptr[r+1]-1 (n_r rows) and has
 * L_r = kv_indptr[r+1] - kv_indptr[r] cached tokens (prefix p_r = L_r - n_r,
 * then the n_r new tokens, whose K/V must already be stored).  Query i of
 * request r (position p_r + i) attends to positions 0 .. p_r + i through
 * req_to_token[req_pool_indices[r], position]:
 *     out[t, hq, :] = sum_j softmax(scale * <q[t, hq], K_j>)_j V_j
 * q, out: bf16 [n_tokens, n_q_heads, head_dim]; qo_indptr, kv_indptr: int32
 * [n_reqs + 1] (device), qo_indptr[n_reqs] == n_tokens.  QK^T and PV run on
 * tcgen05 tensor cores (bf16 operands, fp32 accumulation in tensor memory, P
 * rounded to bf16).  Supported: head_dim 64 or 128; G in {1, 2, 4, 8, 16}.
 * n_r > L_r or L_r > max_ctx sets PA_DEVERR_LEN and skips that request. */
pa_status pa_paged_prefill_attn(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                const void *v_buf, pa_kv_shape s, int layer_id,
                                const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                const int32_t *req_to_token, int req_rows, int max_ctx,
                                const int32_t *req_pool_indices, float scale, void *workspace,
                                size_t workspace_bytes, void *out, cudaStream_t st);

/* As pa_paged_prefill_attn, and the same epilogue also writes each request's
 * last row, out[qo_indptr[r+1] - 1], to last_out[r]: bf16 [n_reqs, n_q_heads,
 * head_dim] (commit e58a728: select per-request final logits from cumulative
 * query lengths).  A request with no rows leaves last_out[r] unwritten.
 * last_out must be non-NULL and 16-byte aligned. */
pa_status pa_paged_prefill_attn_last(const void *q, int n_tokens, int n_q_heads, const void *k_buf,
                                     const void *v_buf, pa_kv_shape s, int layer_id,
                                     const int32_t *qo_indptr, const int32_t *kv_indptr, int n_reqs,
                                     const int32_t *req_to_token, int req_rows, int max_ctx,
                                     const int32_t *req_pool_indices, float scale, void *workspace,
                                     size_t workspace_bytes, void *out, void *last_out, cudaStream_t st);

/* Dense prefill: prompts with no cached prefix, K/V read straight from the
 * packed new tokens instead of through a page table (commit e58a728: prompts
 * packed into one forward, rows addressed by cumulative query lengths).
 * q, out: bf16 [n_tokens, n_q_heads, head_dim]; k, v: bf16 [n_tokens,
 * n_kv_heads, head_dim], the new tokens' (rotated) K and V, packed by the same
 * qo_indptr; query i of request r attends to tokens 0..i of request r.
 * Gives the same bits as pa_paged_prefill_attn over a cache holding exactly
 * these rows with no prefix.  last_out as in pa_paged_prefill_attn_last, or
 * NULL.  Supported: head_dim 64 or 128, G in {1, 2, 4, 8, 16}, n_reqs <= 2048. */
pa_status pa_dense_prefill_attn(const void *q, int n_tokens, int n_q_heads, const void *k, const void *v,
                                int n_kv_heads, int head_dim, const int32_t *qo_indptr, int n_reqs, float scale,
                                void *workspace, size_t workspace_bytes, void *out, void *last_out,
                                cudaStream_t st);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */

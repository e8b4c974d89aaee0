// pa_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

constexpr int kWorkspaceHeader = 256;   // error word + padding at the start of a workspace
// prefill work queue, int32 words inside the header (separate 64-byte sectors):
// the next item to claim and the number of CTAs that have finished
constexpr int kPrefillQueueWord = 16;
constexpr int kPrefillDoneWord = 32;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// SM count of the current device (cached per device; a property, not call state).
int num_sms();

// Raise the dynamic shared-memory limit of kernel `kern` on the current device
// to at least `bytes`.  The attribute is per device, so the largest value set
// is remembered per (kernel, device), under a lock.  false if the runtime
// refused.
bool ensure_dynamic_smem(const void *kern, size_t bytes);

// Current launch-overlap mode (PA_OVERLAP_*).
int launch_overlap();

// Time limit of the kernels' bounded pipeline waits (pa_set_wait_timeout_ns).
uint64_t wait_limit_ns();

// Index arrays may be read before the wait for the preceding kernel
// (PA_OVERLAP_EARLY_METADATA, and PA_OVERLAP_EARLY_KV which includes it).
bool early_metadata();

// Launch `kern` on `st`, as a programmatic dependent of the preceding kernel
// when launch overlap is on.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_overlap() != PA_OVERLAP_OFF ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Encode a TMA tensor map over a bf16 tensor of `rank` (<= 3) dimensions
// (dims innermost first, strides in bytes for dims 1..rank-1) with the given
// box, 128-byte swizzle, zero fill out of range.  The driver entry point is
// resolved once through the runtime (no libcuda link).  false on failure.
bool encode_tmap_bf16(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                      const cuuint32_t *box);

// The same over a byte tensor (e4m3 cache rows): without swizzle a box lands
// in shared memory as plain rows; with swizzle128 (128-byte inner box) it
// lands in the 128-byte XOR-swizzled layout.
bool encode_tmap_u8(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box, bool swizzle128 = false);

// Decode workspace geometry, a pure function of its arguments.
struct DecodeWsLayout {
    int cap_batch;
    size_t counters_off, ml_off, o_off, total;
};
DecodeWsLayout decode_ws_layout(size_t workspace_bytes, int n_q_heads, int n_kv_heads, int head_dim,
                                int max_splits);

}  // namespace pa

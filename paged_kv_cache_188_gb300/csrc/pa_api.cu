// pa_api.cu -- host side of the C ABI: status names, workspace geometry and
// initialisation, device error word readback.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {

static volatile int g_overlap = PA_OVERLAP_OFF;

int launch_overlap() { return g_overlap; }

static volatile uint64_t g_wait_ns = 2000000000ull;

uint64_t wait_limit_ns() { return g_wait_ns; }

bool early_metadata() { return g_overlap == PA_OVERLAP_EARLY_METADATA || g_overlap == PA_OVERLAP_EARLY_KV; }

int num_sms()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

bool ensure_dynamic_smem(const void *kern, size_t bytes)
{
    struct Rec {
        const void *kern;
        int dev;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Rec> recs;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (Rec &r : recs) {
        if (r.kern != kern || r.dev != dev) continue;
        if (r.bytes >= bytes) return true;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
            return false;
        r.bytes = bytes;
        return true;
    }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return false;
    recs.push_back(Rec{kern, dev, bytes});
    return true;
}

static size_t per_request_bytes(int n_q_heads, int n_kv_heads, int head_dim, int max_splits)
{
    return (size_t)n_kv_heads * 4 + (size_t)max_splits * n_q_heads * 2 * 4 +
           (size_t)max_splits * n_q_heads * head_dim * 4;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

static bool encode_tmap(CUtensorMap *m, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle, const void *ptr,
                        int rank, const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dtype, rank, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_bf16(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                      const cuuint32_t *box)
{
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, ptr, rank, dims, strides, box);
}

bool encode_tmap_u8(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box, bool swizzle128)
{
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                       swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, ptr, rank, dims, strides,
                       box);
}

DecodeWsLayout decode_ws_layout(size_t workspace_bytes, int n_q_heads, int n_kv_heads, int head_dim,
                                int max_splits)
{
    DecodeWsLayout L{};
    const size_t slack = 4 * 256;
    const size_t per_b = per_request_bytes(n_q_heads, n_kv_heads, head_dim, max_splits);
    if (per_b == 0 || workspace_bytes < slack) return L;
    size_t cap = (workspace_bytes - slack) / per_b;
    if (cap > (1u << 30)) cap = 1u << 30;
    L.cap_batch = (int)cap;
    L.counters_off = kWorkspaceHeader;
    L.ml_off = align_up(L.counters_off + cap * n_kv_heads * 4, 256);
    L.o_off = align_up(L.ml_off + (size_t)max_splits * cap * n_q_heads * 2 * 4, 256);
    L.total = L.o_off + (size_t)max_splits * cap * n_q_heads * head_dim * 4;
    return L;
}

}  // namespace pa

using namespace pa;

extern "C" const char *pa_status_string(pa_status s)
{
    switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: a size or index argument is out of range";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: a pointer is not 16-byte (workspace 256-byte) aligned";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head_dim or GQA group not supported";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA call failed";
    case PA_ERR_DEVICE_INDEX: return "PA_ERR_DEVICE_INDEX: the device error word is set";
    }
    return "unknown pa_status";
}

extern "C" size_t pa_decode_workspace_bytes(int max_batch, int n_q_heads, int n_kv_heads, int head_dim,
                                            int max_splits)
{
    if (max_batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_splits <= 0) return 0;
    return 4 * 256 + (size_t)max_batch * per_request_bytes(n_q_heads, n_kv_heads, head_dim, max_splits);
}

extern "C" size_t pa_prefill_workspace_bytes(void) { return 4096; }

extern "C" pa_status pa_workspace_init(void *workspace, size_t workspace_bytes, cudaStream_t st)
{
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    if (workspace_bytes < (size_t)kWorkspaceHeader) return PA_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_get_error_word(const int32_t *error_word, int32_t *device_error, cudaStream_t st)
{
    if (!error_word || !device_error) return PA_ERR_NULL;
    if (!aligned4(error_word)) return PA_ERR_ALIGN;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, error_word, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    *device_error = v;
    return v ? PA_ERR_DEVICE_INDEX : PA_OK;
}

extern "C" pa_status pa_get_error(const void *workspace, int32_t *device_error, cudaStream_t st)
{
    if (!workspace) return PA_ERR_NULL;
    if (!aligned256(workspace)) return PA_ERR_ALIGN;
    return pa_get_error_word(static_cast<const int32_t *>(workspace), device_error, st);
}

extern "C" pa_status pa_set_launch_overlap(int mode)
{
    if (mode != PA_OVERLAP_OFF && mode != PA_OVERLAP_SAFE && mode != PA_OVERLAP_EARLY_METADATA &&
        mode != PA_OVERLAP_EARLY_KV)
        return PA_ERR_SHAPE;
    pa::g_overlap = mode;
    return PA_OK;
}

extern "C" int pa_get_launch_overlap(void) { return pa::g_overlap; }

extern "C" void pa_set_wait_timeout_ns(uint64_t ns) { pa::g_wait_ns = ns; }

extern "C" uint64_t pa_get_wait_timeout_ns(void) { return pa::g_wait_ns; }

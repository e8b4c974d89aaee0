// pa_common.cuh -- device helpers shared by the paged-KV attention kernels
// (sm_103a).  Inline PTX for cp.async, ldmatrix and the warp-level bf16 MMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

__device__ __forceinline__ void set_error(int32_t *err, int bits)
{
    if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes == 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
// Wait until every cp.async this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Read-only load of *p if `pred` (else -1), kept in program order with the
// other memory operations (volatile, memory clobber): issued where it is
// written, not moved down to the first use of its value.
__device__ __forceinline__ int32_t ld_nc_ordered_s32_if(bool pred, const int32_t *p)
{
    int32_t v = -1;
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q ld.global.nc.s32 %0, [%1];\n}\n"
                 : "+r"(v)
                 : "l"(p), "r"((int)pred)
                 : "memory");
    return v;
}

// L2 load of *p if `pred` (else 0), kept in program order with the other
// memory operations (volatile, memory clobber): a batch of these is issued
// where it is written, not moved down to the first use of its values.
__device__ __forceinline__ float ld_cg_ordered_if(bool pred, const float *p)
{
    float v = 0.f;
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q ld.global.cg.f32 %0, [%1];\n}\n"
                 : "+f"(v)
                 : "l"(p), "r"((int)pred)
                 : "memory");
    return v;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D[16x8] += A[16x16] * B[16x8], bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D[16x8] += A[16x16] * B[16x8], f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// transpose an 8x8 b16 matrix held one 32-bit pair per thread (mma fragment layout)
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// barrier over the first `nthreads` threads that use id `id` (warp multiples)
// Programmatic dependent launch.  pdl_wait: block until the kernel this grid
// was launched behind has finished and its writes are visible (returns at once
// for a plain launch).  pdl_launch_dependents: let the next kernel on the
// stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// two fp32 -> packed bf16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// two fp32 -> packed f16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two e4m3 bytes (the low one first) -> f16x2 (the low byte's value in the low
// half).  Exact: every e4m3 value is an f16 number.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Two e4m3 bytes (the low one first) -> bf16x2.  Exact: every e4m3 value is
// a bf16 number (3 significant bits, exponents -9 .. 8).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    __half_raw lo, hi;
    lo.x = h.x;
    hi.x = h.y;
    return pack_bf16x2(__half2float(__half(lo)), __half2float(__half(hi)));
}

// bf16x2 word -> f16x2 word, each value clamped to the f16 range first (f16
// holds bf16's 8 significant bits; magnitudes below 2^-14 lose low bits).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_sat(uint32_t w)
{
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    return pack_f16x2(fminf(fmaxf(lo, -65504.f), 65504.f), fminf(fmaxf(hi, -65504.f), 65504.f));
}

// Sixteen fp32 values x[i] / scale (IEEE division) -> e4m3 bytes, round to
// nearest even, finite overflow saturating to +-448; x[0] in the low byte.
__device__ __forceinline__ uint4 quant_e4m3x16(const float (&x)[16], float scale)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t a = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * i], scale), __fdiv_rn(x[4 * i + 1], scale)), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * i + 2], scale), __fdiv_rn(x[4 * i + 3], scale)), __NV_SATFINITE, __NV_E4M3);
        w[i] = (uint32_t)a | ((uint32_t)b << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rotate one interleaved bf16 pair (x0, x1) stored as a 32-bit word by the
// angle with cosine c and sine s: (x0*c - x1*s, x0*s + x1*c), rounded to bf16
// (nearest even).  The products x1*s and x1*c are split exactly into p + e
// (FMA remainder), so a cancelling sum keeps its low bits.  Shared by the RoPE
// kernel and the fused decode step so both give the same bits.
__device__ __forceinline__ uint32_t rope_pair_bf16(uint32_t w, float c, float s)
{
    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    const float x0 = __low2float(pr), x1 = __high2float(pr);
    const float p0 = x1 * s, e0 = fmaf(x1, s, -p0);
    const float p1 = x1 * c, e1 = fmaf(x1, c, -p1);
    const float y0 = fmaf(x0, c, -p0) - e0;
    const float y1 = fmaf(x0, s, p1) + e1;
    return pack_bf16x2(y0, y1);
}

// Packed pairs of fp32 values (low, high) for the sm_100-family two-float
// arithmetic; each lane of fma_f32x2 / add_f32x2 is one IEEE round-to-nearest
// operation, the same value as the scalar fmaf / add.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi)
{
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float f32x2_lo(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float f32x2_hi(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float fast_exp2(float x)
{
    return exp2f(x);
}

}  // namespace pa

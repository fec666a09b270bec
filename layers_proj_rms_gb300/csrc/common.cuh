// Shared device helpers for the mHC kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// Device-side fault word: a kernel that gives up a bounded wait writes a
// nonzero code through this pointer and returns; the host reads the word
// with mhc_device_error().  The first fault code is kept.
__device__ __forceinline__ void report_fault(int *fault, int code)
{
    if (fault) atomicCAS(fault, 0, code);
}

// ---- bf16 <-> fp32, 8 values per 16-byte vector ---------------------------

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        f[2 * q] = __uint_as_float(w[q] << 16);
        f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    uint4 v;
    v.x = pack2(f[0], f[1]);
    v.y = pack2(f[2], f[3]);
    v.z = pack2(f[4], f[5]);
    v.w = pack2(f[6], f[7]);
    return v;
}

// The three bf16 terms of one fp32 weight: hi = bf16(w), lo = bf16(w - hi),
// lo2 = bf16(w - hi - lo).  Both differences are exact in fp32 (each is a
// rounding error of a value that fits in 24 bits), so hi + lo + lo2 equals w
// to within 2^-24 relative.
__device__ __forceinline__ void w_terms(float w, float &hi, float &lo, float &lo2)
{
    hi = __bfloat162float(__float2bfloat16_rn(w));
    const float r1 = w - hi;
    lo = __bfloat162float(__float2bfloat16_rn(r1));
    lo2 = __bfloat162float(__float2bfloat16_rn(r1 - lo));
}

// The hardware's approximate reciprocal (rcp.approx: at most 1 ulp from
// 1/x, denormal inputs flushed): one instruction where 1.0f / x is a
// correctly rounded inline sequence with a slow-path branch.
__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- packed fp32 pairs: f32x2 arithmetic, two IEEE fp32 operations (each
// rounded as its scalar form) per instruction --------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// 8 bf16 -> 4 pairs (elements 2q, 2q+1) and back (round to nearest even)
__device__ __forceinline__ void unpack8x2(const uint4 v, f32x2 (&p)[4])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        p[q] = f2_make(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
}
__device__ __forceinline__ uint4 pack8x2(const f32x2 (&p)[4])
{
    float f[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) f2_split(p[q], f[2 * q], f[2 * q + 1]);
    return pack8(f);
}

// Streaming 16-byte loads: read-only path, no L1 allocation for data that is
// touched once.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// 8-byte load from shared memory by 32-bit shared address
__device__ __forceinline__ uint2 lds64(uint32_t saddr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr));
    return v;
}

// 16-byte load from shared memory by 32-bit shared address (an explicit
// ld.shared; a generic pointer derived by integer arithmetic would go
// through the generic path).
__device__ __forceinline__ uint4 lds128(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr));
    return v;
}

// Programmatic dependent launch: every kernel of the library is launched
// with programmatic stream serialization (launch_k in launch.h), so its grid
// may be set up while the previous kernel on the stream drains; pdl_wait()
// at the top of each kernel then blocks until that kernel has completed and
// its memory is visible.  Without the launch attribute it returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float lds32f(uint32_t saddr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// Segment of controller logit o: 0 pre, 1 post, 2 res.
__device__ __forceinline__ int seg_of(int o, int n) { return o < n ? 0 : (o < 2 * n ? 1 : 2); }

}  // namespace mhc

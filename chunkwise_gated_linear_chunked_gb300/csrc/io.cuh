// Element I/O helpers: 4-wide loads/stores of fp32 or bf16 rows, widened to / narrowed from fp32 (RN).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gla {

template <typename T>
struct IO;

template <>
struct IO<float> {
    static __device__ __forceinline__ float load1(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float4 load4(const float *p)
    {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ void store4(float *p, float4 v)
    {
        *reinterpret_cast<float4 *>(p) = v;
    }
};

template <>
struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ float load1(const __nv_bfloat16 *p)
    {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ float4 load4(const __nv_bfloat16 *p)
    {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v)
    {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<const unsigned *>(&a);
        u.y = *reinterpret_cast<const unsigned *>(&b);
        *reinterpret_cast<uint2 *>(p) = u;
    }
};

template <>
struct IO<__half> {
    static __device__ __forceinline__ float load1(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ float4 load4(const __half *p)
    {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
};

__device__ __forceinline__ float at(const float4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

}  // namespace gla

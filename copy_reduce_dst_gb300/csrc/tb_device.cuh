// Device-side helpers shared by the kernels of libtb: vector global memory
// access without L1 allocation, the elementwise float add, and the global
// nanosecond timer used to bound every wait.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tb {
namespace dev {

// ---------------------------------------------------------------------------
// Vector memory access.  VB = bytes per access: 4 (scalar), 16 or 32 (the
// 256-bit global access of sm_100-class GPUs).  Values travel as raw 32-bit
// words, so a copy never passes through a float operation.
// ---------------------------------------------------------------------------
template <int VB>
struct Vec {
    uint32_t w[VB / 4];
};

template <int VB>
__device__ __forceinline__ void vload(Vec<VB> &v, const void *p);

template <>
__device__ __forceinline__ void vload<4>(Vec<4> &v, const void *p)
{
    asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
}

template <>
__device__ __forceinline__ void vload<16>(Vec<16> &v, const void *p)
{
    asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
        : "l"(p));
}

template <>
__device__ __forceinline__ void vload<32>(Vec<32> &v, const void *p)
{
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
          "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
        : "l"(p));
}

template <int VB>
__device__ __forceinline__ void vstore(void *p, const Vec<VB> &v);

template <>
__device__ __forceinline__ void vstore<4>(void *p, const Vec<4> &v)
{
    asm volatile("st.global.L1::no_allocate.b32 [%0], %1;" ::"l"(p), "r"(v.w[0]));
}

template <>
__device__ __forceinline__ void vstore<16>(void *p, const Vec<16> &v)
{
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]));
}

template <>
__device__ __forceinline__ void vstore<32>(void *p, const Vec<32> &v)
{
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
                 "r"(v.w[6]), "r"(v.w[7]));
}

// acc += x elementwise: one IEEE binary32 add, round to nearest even, per
// element (__fadd_rn is never contracted into an FMA).
template <int VB>
__device__ __forceinline__ void vadd(Vec<VB> &acc, const Vec<VB> &x)
{
#pragma unroll
    for (int e = 0; e < VB / 4; ++e)
        acc.w[e] = __float_as_uint(__fadd_rn(__uint_as_float(acc.w[e]), __uint_as_float(x.w[e])));
}


__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace dev
}  // namespace tb

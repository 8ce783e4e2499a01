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

// Stores of the vector form, streaming (.cs: evict-first in the caches), as
// the destination is written once per launch and read by nobody in it.
// Measured on GB300 against L1::no_allocate stores: 4 MiB transfer with
// rotation, 10 graphed iterations 2.43-2.44 against 2.52-2.53 us per
// iteration (mean of 25 runs); 64 iterations, 8 MiB and 3 x 256 MiB the
// same within 1%.
template <int VB>
__device__ __forceinline__ void vstore(void *p, const Vec<VB> &v);

template <>
__device__ __forceinline__ void vstore<4>(void *p, const Vec<4> &v)
{
    asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(p), "r"(v.w[0]));
}

template <>
__device__ __forceinline__ void vstore<16>(void *p, const Vec<16> &v)
{
    asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]));
}

template <>
__device__ __forceinline__ void vstore<32>(void *p, const Vec<32> &v)
{
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
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


// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream be scheduled once every CTA of this one has issued it;
// wait_prerequisite returns once the kernel this one was launched behind
// has completed and its memory operations are visible.  Both do nothing
// for a launch without the programmatic attribute.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_prerequisite()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// Bulk (TMA) copies between global and shared memory: cp.async.bulk
// global -> shared completes on an mbarrier; shared -> global is tracked by
// bulk groups.  No tensor map, no cluster multicast.  Every wait is bounded.
// ---------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the phase of the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of the given parity, for at most limit_ns; a limit of
// 0 does not wait at all (one non-blocking probe).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (limit_ns == 0)
        return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns)
            return false;
    return true;
}

// Announces `bytes` of bulk-copy traffic on an mbarrier (this thread's
// arrival); the copies that complete it are issued with bulk_copy_in.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_copy_in(uint32_t smem, uint64_t gsrc, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem),
        "l"(gsrc), "r"(bytes), "r"(bar)
        : "memory");
}

// One bulk copy global -> shared that alone completes the mbarrier's phase.
__device__ __forceinline__ void bulk_load(uint32_t smem, uint64_t gsrc, uint32_t bytes, uint32_t bar)
{
    mbar_expect_tx(bar, bytes);
    bulk_copy_in(smem, gsrc, bytes, bar);
}

__device__ __forceinline__ void bulk_store(uint64_t gdst, uint32_t smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Newest group may still be reading shared memory; all older ones are done.
__device__ __forceinline__ void bulk_wait_read_all_but_newest()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Makes this thread's ordinary shared-memory writes visible to later bulk
// copies (the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace dev
}  // namespace tb

// Kernels of libtb for sm_103a (GB300): the reduce-copy, the batched copy,
// the source-pattern fills and the timing gate.
//
// Everything here is HBM-bound streaming: no kernel is a contraction, so none
// touches the tensor cores.  Loads use the non-coherent path without L1
// allocation (each byte is read once per launch) and stores skip L1.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "tb_internal.h"

namespace tb {
namespace {

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

// ---------------------------------------------------------------------------
// K1: reduce-copy.  N = number of sources (0 = memset, 1 = bit copy).
// Each thread keeps U vectors of every source in flight: all N*U loads are
// issued before the first add, then the sums run left to right per element
// and U vector stores follow.
// ---------------------------------------------------------------------------
struct ReduceArgs {
    const float *src[TB_MAX_SRCS];
    float *dst;
    uint64_t n;
    uint64_t head;
    uint64_t nvec;
    uint32_t nsub;         // sub-executors; never more than the grid's CTAs
    uint32_t memset_word;
};

// The CTAs of a launch are dealt to the sub-executors as evenly as integers
// allow (sub-executor s gets CTAs [s*G/S, (s+1)*G/S)), and each sub-executor
// owns a contiguous range of body vectors in proportion to its CTAs, so every
// CTA streams the same share whether or not S divides the grid G.
struct SubRange {
    uint32_t part, nparts;   // this CTA's rank within its sub-executor, and their count
    uint64_t vbeg, vend;     // the sub-executor's body vectors
};

__device__ __forceinline__ SubRange sub_range(uint64_t nvec, uint32_t S)
{
    const uint32_t G = gridDim.x, b = blockIdx.x;
    const uint32_t sub = (uint32_t)(((uint64_t)(b + 1) * S - 1) / G);
    const uint32_t c0 = (uint32_t)((uint64_t)sub * G / S);
    const uint32_t c1 = (uint32_t)((uint64_t)(sub + 1) * G / S);
    const uint64_t q = nvec / G, r = nvec % G;
    SubRange sr;
    sr.part = b - c0;
    sr.nparts = c1 - c0;
    sr.vbeg = q * c0 + (r * c0) / G;
    sr.vend = q * c1 + (r * c1) / G;
    return sr;
}

// Scalar element i, used for the head and the tail of a launch.
template <int N>
__device__ __forceinline__ void reduce_one(const ReduceArgs &a, uint64_t i)
{
    if constexpr (N == 0) {
        reinterpret_cast<uint32_t *>(a.dst)[i] = a.memset_word;
    } else {
        uint32_t acc = reinterpret_cast<const uint32_t *>(a.src[0])[i];
#pragma unroll
        for (int k = 1; k < N; ++k)
            acc = __float_as_uint(__fadd_rn(__uint_as_float(acc), a.src[k][i]));
        reinterpret_cast<uint32_t *>(a.dst)[i] = acc;
    }
}

template <int N, int VB, int U>
__device__ __forceinline__ void reduce_vectors(const ReduceArgs &a, const char *const *s, char *d,
                                               uint64_t v0, uint64_t stride, uint64_t vend,
                                               bool full)
{
    Vec<VB> acc[U];
    if constexpr (N == 0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < VB / 4; ++e)
                acc[u].w[e] = a.memset_word;
    } else {
        Vec<VB> x[N > 1 ? N - 1 : 1][U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (full || v0 + u * stride < vend)
                vload<VB>(acc[u], s[0] + (v0 + u * stride) * VB);
#pragma unroll
        for (int k = 1; k < N; ++k)
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (full || v0 + u * stride < vend)
                    vload<VB>(x[k - 1][u], s[k] + (v0 + u * stride) * VB);
#pragma unroll
        for (int k = 1; k < N; ++k)
#pragma unroll
            for (int u = 0; u < U; ++u)
                vadd<VB>(acc[u], x[k - 1][u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (full || v0 + u * stride < vend)
            vstore<VB>(d + (v0 + u * stride) * VB, acc[u]);
}

template <int N, int VB, int U>
__global__ void __launch_bounds__(512) k_reduce(const ReduceArgs a)
{
    const uint32_t tid = threadIdx.x;
    const uint32_t bd = blockDim.x;
    const SubRange sr = sub_range(a.nvec, a.nsub);

    const char *s[N > 0 ? N : 1];
#pragma unroll
    for (int k = 0; k < N; ++k)
        s[k] = reinterpret_cast<const char *>(a.src[k] + a.head);
    char *d = reinterpret_cast<char *>(a.dst + a.head);

    const uint64_t vend = sr.vend;
    const uint64_t tile = (uint64_t)bd * U;
    const uint64_t step = (uint64_t)sr.nparts * tile;
    for (uint64_t t = sr.vbeg + sr.part * tile; t < vend; t += step) {
        if (t + tile <= vend)
            reduce_vectors<N, VB, U>(a, s, d, t + tid, bd, vend, true);
        else
            reduce_vectors<N, VB, U>(a, s, d, t + tid, bd, vend, false);
    }

    if (blockIdx.x == 0 && tid < a.head)
        reduce_one<N>(a, tid);
    const uint64_t tail0 = a.head + a.nvec * (VB / 4);
    if (blockIdx.x == gridDim.x - 1 && tail0 + tid < a.n)
        reduce_one<N>(a, tail0 + tid);
}

// More than 8 sources: the source loop runs at run time, each thread holding
// two vectors of one source at a time.
template <int VB>
__global__ void __launch_bounds__(512) k_reduce_many(const ReduceArgs a, int n_src)
{
    const uint32_t tid = threadIdx.x;
    const uint32_t bd = blockDim.x;
    const SubRange sr = sub_range(a.nvec, a.nsub);
    const uint64_t vend = sr.vend;
    const uint64_t tile = (uint64_t)bd * 2;
    const uint64_t step = (uint64_t)sr.nparts * tile;
    const uint64_t W = VB / 4;
    for (uint64_t t = sr.vbeg + sr.part * tile; t < vend; t += step) {
        const uint64_t v0 = t + tid, v1 = t + bd + tid;
        if (v0 >= vend)
            break;
        const bool ok1 = v1 < vend;
        Vec<VB> acc0, acc1, x0, x1;
        vload<VB>(acc0, a.src[0] + a.head + v0 * W);
        if (ok1)
            vload<VB>(acc1, a.src[0] + a.head + v1 * W);
        for (int k = 1; k < n_src; ++k) {
            vload<VB>(x0, a.src[k] + a.head + v0 * W);
            if (ok1)
                vload<VB>(x1, a.src[k] + a.head + v1 * W);
            vadd<VB>(acc0, x0);
            if (ok1)
                vadd<VB>(acc1, x1);
        }
        vstore<VB>(a.dst + a.head + v0 * W, acc0);
        if (ok1)
            vstore<VB>(a.dst + a.head + v1 * W, acc1);
    }
    const uint64_t tail0 = a.head + a.nvec * W;
    auto one = [&](uint64_t i) {
        uint32_t acc = reinterpret_cast<const uint32_t *>(a.src[0])[i];
        for (int k = 1; k < n_src; ++k)
            acc = __float_as_uint(__fadd_rn(__uint_as_float(acc), a.src[k][i]));
        reinterpret_cast<uint32_t *>(a.dst)[i] = acc;
    };
    if (blockIdx.x == 0 && tid < a.head)
        one(tid);
    if (blockIdx.x == gridDim.x - 1 && tail0 + tid < a.n)
        one(tail0 + tid);
}

using ReduceKernel = void (*)(const ReduceArgs);

template <int N, int VB>
ReduceKernel pick_unroll(int u)
{
    switch (u) {
    case 1: return k_reduce<N, VB, 1>;
    case 2: return k_reduce<N, VB, 2>;
    default: return k_reduce<N, VB, 4>;
    }
}

template <int N>
ReduceKernel pick_vec(int vb, int u)
{
    switch (vb) {
    case 32: return pick_unroll<N, 32>(u);
    case 16: return pick_unroll<N, 16>(u);
    default: return k_reduce<N, 4, 4>;
    }
}

ReduceKernel pick_reduce(int n_src, int vb, int u)
{
    switch (n_src) {
    case 0: return pick_vec<0>(vb, u);
    case 1: return pick_vec<1>(vb, u);
    case 2: return pick_vec<2>(vb, u);
    case 3: return pick_vec<3>(vb, u);
    case 4: return pick_vec<4>(vb, u);
    case 5: return pick_vec<5>(vb, u);
    case 6: return pick_vec<6>(vb, u);
    case 7: return pick_vec<7>(vb, u);
    case 8: return pick_vec<8>(vb, u);
    default: return nullptr;
    }
}

// Largest unroll whose in-flight words (sources x unroll x words per vector)
// stay in registers without spilling at 512 threads per CTA.
int max_unroll(int n_src, int vb)
{
    const int words = std::max(1, n_src) * (vb / 4);
    const int budget = vb == 32 ? 48 : 64;
    for (int u = 4; u > 1; u /= 2)
        if (words * u <= budget)
            return u;
    return 1;
}

// Default: the largest unroll that still fits 64 registers, i.e. two
// 512-thread CTAs per SM.
int default_unroll(int n_src, int vb)
{
    const int words = std::max(1, n_src) * (vb / 4);
    for (int u = 4; u > 1; u /= 2)
        if (words * u <= 32)
            return u;
    return 1;
}

// ---------------------------------------------------------------------------
// Source patterns ("TransferBench data validation", "Expected source pattern")
// ---------------------------------------------------------------------------

// Default pattern: PrepSrcValue(bufferIdx, i) as float32.
__global__ void k_fill_default(float *dst, uint64_t n, uint32_t mult)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t r = (uint32_t)(i % 383u);
        const uint32_t v = ((r * 517u) % 383u + 31u) * mult;
        dst[i] = (float)v;
    }
}

// SplitMix64 finaliser (Steele, Lea & Flood, OOPSLA 2014).
__device__ __forceinline__ uint64_t sm64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

struct CompressArgs {
    float *dst;
    uint64_t n;
    uint64_t seed;     // seed + bufferIdx
    uint32_t cum[5];   // running sums of the mode percentages
};

// fillCompress: thread per 64-byte line.  Output number j of a SplitMix64
// stream seeded with s is mix(s + (j + 1) * gamma), so line L starts its 17
// draws at counter 17 * L without walking the stream.
__global__ void k_fill_compress(const CompressArgs a)
{
    constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
    const uint64_t lines = (a.n + 15) / 16;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t L = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; L < lines; L += stride) {
        const uint64_t base = a.seed + 17u * L * kGamma;
        const uint32_t r = (uint32_t)(sm64_mix(base + kGamma) % 100u);
        int mode = 0;
        while (mode < 4 && r >= a.cum[mode])
            ++mode;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint64_t d = sm64_mix(base + (uint64_t)(j + 2) * kGamma);
            const int32_t m = (int32_t)(d >> 40) - (1 << 23);
            w[j] = __float_as_uint((float)m * 0x1p-23f);
        }
        // Zeroing masks on little-endian 32-bit words.
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (mode == 1)
                w[j] &= 0x00FF00FFu;  // bytes 1 and 3 of each word
            else if (mode == 2)
                w[j] &= 0x0000FFFFu;  // bytes 2-3 of each word
            else if (mode == 3 && (j & 1))
                w[j] = 0u;            // every odd word
            else if (mode == 4 && j >= 8)
                w[j] = 0u;            // upper 32 bytes
        }
        uint32_t *out = reinterpret_cast<uint32_t *>(a.dst) + L * 16;
        const uint64_t left = a.n - L * 16;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if ((uint64_t)j < left)
                out[j] = w[j];
    }
}

struct RepeatArgs {
    float *dst;
    uint64_t n;
    uint32_t len;
    float pat[4096];
};

__global__ void k_fill_repeat(const __grid_constant__ RepeatArgs a)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n; i += stride)
        a.dst[i] = a.pat[i % a.len];
}

// ---------------------------------------------------------------------------
// Gate: one thread polls a host-mapped flag until it is set or the deadline
// passes; either way it records the outcome and returns, so a lost release
// costs at most timeout_ns and never hangs the GPU.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__global__ void k_gate(const volatile uint32_t *flag, volatile uint32_t *status, uint64_t timeout_ns)
{
    const uint64_t t0 = global_ns();
    for (;;) {
        if (*flag != 0u) {
            *status = 1u;
            break;
        }
        if (global_ns() - t0 > timeout_ns) {
            *status = 2u;
            break;
        }
        __nanosleep(1000);
    }
    __threadfence_system();
}

// ---------------------------------------------------------------------------
// K2: batched copy.  copy_range copies len bytes with `size` cooperating
// threads (a warp or a CTA), any alignment:
//   - head bytes until dst is 16-byte aligned, one byte per thread;
//   - body in 16-byte vectors: direct when src is then 16-byte aligned too,
//     otherwise every output vector is funnel-shifted out of the two aligned
//     source vectors that hold its bytes (both contain bytes of the range,
//     so no load leaves the source's aligned 16-byte words);
//   - tail bytes, one byte per thread.
// ---------------------------------------------------------------------------
constexpr int kCopyUnroll = 4;

__device__ __forceinline__ uint4 ld16(const uint4 *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st16(uint4 *p, const uint4 &v)
{
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w));
}

// Bytes sh .. sh+15 of the 32-byte concatenation lo|hi (little-endian).
__device__ __forceinline__ uint4 shift_pair(const uint4 &lo, const uint4 &hi, uint32_t q, uint32_t rbits)
{
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t o[5];
#pragma unroll
    for (int j = 0; j < 5; ++j)
        o[j] = q == 0 ? w[j] : (q == 1 ? w[j + 1] : (q == 2 ? w[j + 2] : w[j + 3]));
    uint4 r;
    r.x = __funnelshift_r(o[0], o[1], rbits);
    r.y = __funnelshift_r(o[1], o[2], rbits);
    r.z = __funnelshift_r(o[2], o[3], rbits);
    r.w = __funnelshift_r(o[3], o[4], rbits);
    return r;
}

__device__ __forceinline__ void copy_range(uint8_t *dst, const uint8_t *src, uint64_t len,
                                           uint32_t rank, uint32_t size)
{
    uint64_t h = (16u - ((uintptr_t)dst & 15u)) & 15u;
    if (h > len)
        h = len;
    if (rank < h)
        dst[rank] = src[rank];
    dst += h;
    src += h;
    len -= h;

    const uint64_t nv = len >> 4;
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    const uint32_t sh = (uint32_t)((uintptr_t)src & 15u);
    uint64_t v = rank;
    if (sh == 0) {
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        for (; v + (kCopyUnroll - 1) * (uint64_t)size < nv; v += kCopyUnroll * (uint64_t)size) {
            uint4 r[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u)
                r[u] = ld16(s + v + u * size);
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u)
                st16(d + v + u * size, r[u]);
        }
        for (; v < nv; v += size)
            st16(d + v, ld16(s + v));
    } else {
        const uint4 *s = reinterpret_cast<const uint4 *>(src - sh);
        const uint32_t q = sh >> 2, rbits = (sh & 3u) * 8u;
        for (; v + (kCopyUnroll - 1) * (uint64_t)size < nv; v += kCopyUnroll * (uint64_t)size) {
            uint4 lo[kCopyUnroll], hi[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                lo[u] = ld16(s + v + u * size);
                hi[u] = ld16(s + v + u * size + 1);
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u)
                st16(d + v + u * size, shift_pair(lo[u], hi[u], q, rbits));
        }
        for (; v < nv; v += size)
            st16(d + v, shift_pair(ld16(s + v), ld16(s + v + 1), q, rbits));
    }

    const uint64_t done = nv << 4;
    if (rank < len - done)
        dst[done + rank] = src[done + rank];
}

__device__ __forceinline__ WorkItem load_item(const WorkItem *p)
{
    WorkItem w;
    w.src = __ldg(&p->src);
    w.dst = __ldg(&p->dst);
    w.len = __ldg(&p->len);
    return w;
}

struct BatchArgs {
    const WorkItem *shorts;      // n_short copies, longest first
    const WorkItem *longs;       // n_long copies
    const uint64_t *prefix;      // stream offset of each long copy
    const uint32_t *chunk_desc;  // long copy holding each chunk's first byte
    uint32_t *status;            // nullable: set to 1 if a bounded wait expired
    uint64_t long_bytes;
    uint32_t n_short;
    uint32_t chunks;
};

// ---------------------------------------------------------------------------
// Bulk (TMA) copies through shared memory: cp.async.bulk global -> shared
// completes on an mbarrier; cp.async.bulk shared -> global is tracked by
// bulk groups.  No tensor map, no cluster multicast.
// ---------------------------------------------------------------------------
constexpr int kStages = 3;
constexpr uint32_t kBlock = 16384;                 // bytes per bulk copy
constexpr size_t kBarBytes = 128;                  // mbarriers, then stages
constexpr size_t kBatchSmem = kBarBytes + (size_t)kStages * kBlock;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait

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

// Waits for the phase of the given parity, for at most kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    return true;
}

__device__ __forceinline__ void bulk_load(uint32_t smem, uint64_t gsrc, uint32_t bytes, uint32_t bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem),
        "l"(gsrc), "r"(bytes), "r"(bar)
        : "memory");
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

// Walks this CTA's chunks of the long-copy stream (chunks b, b + G, ...),
// one piece (a contiguous part of one long copy) at a time.
struct PieceWalker {
    const BatchArgs &a;
    uint32_t c;
    uint64_t pos, end;
    uint32_t d;

    __device__ explicit PieceWalker(const BatchArgs &args) : a(args), c(blockIdx.x), pos(0), end(0), d(0)
    {
        open();
    }
    __device__ void open()
    {
        if (c < a.chunks) {
            pos = chunk_start(a.long_bytes, a.chunks, c);
            end = chunk_start(a.long_bytes, a.chunks, c + 1);
            d = __ldg(a.chunk_desc + c);
        }
    }
    __device__ bool next(uint64_t &src, uint64_t &dst, uint64_t &len)
    {
        while (c < a.chunks) {
            if (pos < end) {
                const WorkItem w = load_item(a.longs + d);
                const uint64_t off = pos - __ldg(a.prefix + d);
                const uint64_t take = min(w.len - off, end - pos);
                src = w.src + off;
                dst = w.dst + off;
                len = take;
                pos += take;
                if (off + take == w.len)
                    ++d;
                return true;
            }
            c += gridDim.x;
            open();
        }
        return false;
    }
};

// A piece is copied by bulk copies when src and dst share their address
// modulo 16: a byte head brings both to 16 bytes, the body moves in bulk,
// a byte tail (< 16 bytes) ends it.  Other pieces are copied by threads.
__device__ __forceinline__ bool bulk_split(uint64_t src, uint64_t dst, uint64_t len, uint64_t &head,
                                           uint64_t &body)
{
    if (((src ^ dst) & 15u) != 0)
        return false;
    head = min((16u - (dst & 15u)) & 15u, len);
    body = (len - head) & ~(uint64_t)15;
    return true;
}

// Thread 0's bulk pipeline over the bodies of this CTA's pieces: kStages
// blocks of up to kBlock bytes in flight; block k uses stage k % kStages.
// Returns false if a wait expired (status recorded, copies drained).
__device__ bool bulk_pipeline(const BatchArgs &a, uint32_t bars, uint32_t stages)
{
    PieceWalker walk(a);
    uint64_t bsrc = 0, bdst = 0, bleft = 0;
    auto next_block = [&](uint64_t &gs, uint64_t &gd, uint32_t &nb) -> bool {
        while (bleft == 0) {
            uint64_t s, d, l, h, body;
            if (!walk.next(s, d, l))
                return false;
            if (bulk_split(s, d, l, h, body) && body > 0) {
                bsrc = s + h;
                bdst = d + h;
                bleft = body;
            }
        }
        nb = (uint32_t)(bleft < kBlock ? bleft : kBlock);
        gs = bsrc;
        gd = bdst;
        bsrc += nb;
        bdst += nb;
        bleft -= nb;
        return true;
    };

    uint64_t gdst[kStages];
    uint32_t nbytes[kStages];
    uint32_t uses = 0;  // bit s: parity of stage s's next phase
    uint32_t issued = 0;
    for (int s = 0; s < kStages; ++s) {
        uint64_t gs;
        if (!next_block(gs, gdst[s], nbytes[s]))
            break;
        bulk_load(stages + s * kBlock, gs, nbytes[s], bars + 8 * s);
        ++issued;
    }
    bool ok = true;
    for (uint32_t i = 0; i < issued; ++i) {
        const uint32_t s = i % kStages;
        if (!mbar_wait_bounded(bars + 8 * s, (uses >> s) & 1u)) {
            ok = false;
            break;
        }
        uses ^= 1u << s;
        bulk_store(gdst[s], stages + s * kBlock, nbytes[s]);
        if (i >= 1) {
            const uint32_t sp = (i - 1) % kStages;
            uint64_t gs;
            if (next_block(gs, gdst[sp], nbytes[sp])) {
                bulk_wait_read_all_but_newest();
                bulk_load(stages + sp * kBlock, gs, nbytes[sp], bars + 8 * sp);
                ++issued;
            }
        }
    }
    if (!ok) {
        if (a.status)
            *reinterpret_cast<volatile uint32_t *>(a.status) = 1u;
        // Let the loads still in flight land (each wait bounded again).
        for (uint32_t k = 0; k < kStages; ++k)
            mbar_wait_bounded(bars + 8 * k, (uses >> k) & 1u);
    }
    bulk_wait_all();
    return ok;
}

// Threads other than warp 0: the bytes of this CTA's pieces that the bulk
// pipeline does not move (heads, tails, pieces whose src and dst differ
// modulo 16).
__device__ void long_edges(const BatchArgs &a, uint32_t rank, uint32_t size)
{
    PieceWalker walk(a);
    uint64_t s, d, l, h, body;
    while (walk.next(s, d, l)) {
        if (bulk_split(s, d, l, h, body)) {
            if (rank < h)
                reinterpret_cast<uint8_t *>(d)[rank] = reinterpret_cast<const uint8_t *>(s)[rank];
            const uint64_t t = h + body;
            if (rank < l - t)
                reinterpret_cast<uint8_t *>(d)[t + rank] = reinterpret_cast<const uint8_t *>(s)[t + rank];
        } else {
            copy_range(reinterpret_cast<uint8_t *>(d), reinterpret_cast<const uint8_t *>(s), l, rank,
                       size);
        }
    }
}

// Persistent grid of one wave.
//   Long copies: their bytes form one stream of `chunks` equal chunks; CTA b
//   owns chunks b, b + G, ... (the same number for every CTA, the grid
//   sweeping the stream front to back).  Thread 0 moves the 16-byte-aligned
//   bodies with a bulk-copy pipeline through shared memory; warps 1.. copy
//   the leftover edges.
//   Short copies (longest first in memory) go to warps 1.. (all warps when
//   there are no long copies), dealt in boustrophedon order: round r goes up
//   the warp list when r is even and down when it is odd, which keeps every
//   warp's byte total close to the mean.  Odd warps walk their rounds from
//   the smallest item up, so small latency-bound copies overlap large ones.
//   Each warp fetches its next item before copying the current one.
__global__ void __launch_bounds__(kBatchThreads, 4) k_batch(const BatchArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const bool has_long = a.chunks > 0;
    if (has_long) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < kStages; ++s)
                mbar_init(smem_u32(smem) + 8 * s);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (warp == 0) {
            if (lane == 0)
                bulk_pipeline(a, smem_u32(smem), smem_u32(smem + kBarBytes));
            return;
        }
        long_edges(a, threadIdx.x - 32, blockDim.x - 32);
    }

    const uint32_t w0 = has_long ? 1u : 0u;
    const uint32_t warps_per_cta = (blockDim.x >> 5) - w0;
    const uint64_t W = (uint64_t)gridDim.x * warps_per_cta;
    const uint64_t wid = (uint64_t)blockIdx.x * warps_per_cta + (warp - w0);
    const uint64_t n_short = a.n_short;
    const uint64_t R = (n_short + W - 1) / W;
    const bool reverse = wid & 1u;
    // The k-th item this warp copies (k in [0, R)), or n_short if none.
    auto item_at = [&](uint64_t k) {
        const uint64_t r = reverse ? (R - 1 - k) : k;
        return r * W + ((r & 1) ? (W - 1 - wid) : wid);
    };
    uint64_t k = 0;
    while (k < R && item_at(k) >= n_short)
        ++k;
    if (k >= R)
        return;
    WorkItem cur = load_item(a.shorts + item_at(k));
    for (;;) {
        uint64_t kn = k + 1;
        while (kn < R && item_at(kn) >= n_short)
            ++kn;
        const bool more = kn < R;
        WorkItem nxt = cur;
        if (more)
            nxt = load_item(a.shorts + item_at(kn));
        copy_range(reinterpret_cast<uint8_t *>(cur.dst), reinterpret_cast<const uint8_t *>(cur.src),
                   cur.len, lane, 32u);
        if (!more)
            break;
        cur = nxt;
        k = kn;
    }
}

int g_batch_ctas_per_sm = 0;

}  // namespace

// ---------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------

int reduce_ctas_per_sm(int n_src, int vec_bytes, int block_threads, int unroll)
{
    void *fn = n_src <= 8 ? (void *)pick_reduce(n_src, vec_bytes, unroll)
                          : (vec_bytes == 16 ? (void *)k_reduce_many<16> : (void *)k_reduce_many<4>);
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, block_threads, 0) != cudaSuccess ||
        blocks < 1)
        blocks = 1;
    return blocks;
}

int plan_reduce(ReducePlan *p, const void *const *srcs, int n_src, void *dst, uint64_t num_bytes,
                int num_subexec, int ctas_per_subexec, int block_threads, int vec_bytes, int unroll,
                uint32_t memset_byte, int num_sms)
{
    if (!p || !dst || n_src < 0 || n_src > TB_MAX_SRCS || num_bytes % 4 != 0 || num_subexec < 0 ||
        ctas_per_subexec < 0 || block_threads < 0 || block_threads > 512 || block_threads % 32 != 0 ||
        unroll < 0 || unroll > 4 || unroll == 3 || num_sms < 1 ||
        (vec_bytes != 0 && vec_bytes != 4 && vec_bytes != 16 && vec_bytes != 32))
        return TB_EINVAL;
    if (n_src > 0 && !srcs)
        return TB_EINVAL;
    uintptr_t any = (uintptr_t)dst;
    for (int k = 0; k < n_src; ++k) {
        if (!srcs[k])
            return TB_EINVAL;
        any |= (uintptr_t)srcs[k];
    }
    if (any & 3u)
        return TB_EINVAL;

    *p = ReducePlan{};
    p->n_src = n_src;
    for (int k = 0; k < n_src; ++k)
        p->src[k] = static_cast<const float *>(srcs[k]);
    p->dst = static_cast<float *>(dst);
    p->n = num_bytes / 4;
    const uint32_t b = memset_byte & 0xFFu;
    p->memset_word = b | (b << 8) | (b << 16) | (b << 24);

    // Widest vector whose alignment every pointer shares: then one head
    // brings them all to a vector boundary together.
    auto common = [&](uintptr_t mask) {
        const uintptr_t m = (uintptr_t)dst & mask;
        for (int k = 0; k < n_src; ++k)
            if (((uintptr_t)srcs[k] & mask) != m)
                return false;
        return true;
    };
    int vb = common(31) ? 32 : (common(15) ? 16 : 4);
    if (vec_bytes != 0) {
        if (vec_bytes > vb)
            return TB_ENOTSUP;
        vb = vec_bytes;
    }
    if (n_src > 8) {  // the run-time source loop has 4- and 16-byte forms only
        if (vec_bytes == 32)
            return TB_ENOTSUP;
        if (vb == 32)
            vb = 16;
    }
    p->vec_bytes = vb;

    if (vb > 4) {
        const uintptr_t mis = (uintptr_t)dst & (uintptr_t)(vb - 1);
        const uint64_t head = mis ? ((uint64_t)vb - mis) / 4 : 0;
        p->head = std::min<uint64_t>(head, p->n);
    }
    p->nvec = (p->n - p->head) / ((uint64_t)vb / 4);
    p->block_threads = block_threads ? block_threads : 512;
    p->unroll = vb == 4 ? 4 : std::min(unroll ? unroll : default_unroll(n_src, vb), max_unroll(n_src, vb));

    // One full wave of resident CTAs, or S * ctas_per_subexec when the caller
    // fixes the CTAs of each sub-executor (1 = TransferBench's one block per
    // sub-executor); never fewer CTAs than sub-executors.
    const int per_sm = reduce_ctas_per_sm(n_src, vb, p->block_threads, p->unroll);
    const int64_t full = (int64_t)num_sms * per_sm;
    const int64_t S = num_subexec > 0 ? num_subexec : full;
    const int64_t G = ctas_per_subexec > 0 ? S * ctas_per_subexec : std::max<int64_t>(S, full);
    if (G > (int64_t)INT32_MAX)
        return TB_EINVAL;
    p->num_subexec = (int)S;
    p->grid = (int)G;
    return TB_OK;
}

cudaError_t launch_reduce(const ReducePlan &p, cudaStream_t stream)
{
    ReduceArgs a{};
    for (int k = 0; k < p.n_src; ++k)
        a.src[k] = p.src[k];
    a.dst = p.dst;
    a.n = p.n;
    a.head = p.head;
    a.nvec = p.nvec;
    a.nsub = (uint32_t)p.num_subexec;
    a.memset_word = p.memset_word;
    const unsigned grid = (unsigned)p.grid;
    if (p.n == 0)
        return cudaSuccess;
    if (p.n_src > 8) {
        if (p.vec_bytes == 16)
            k_reduce_many<16><<<grid, p.block_threads, 0, stream>>>(a, p.n_src);
        else
            k_reduce_many<4><<<grid, p.block_threads, 0, stream>>>(a, p.n_src);
    } else {
        ReduceKernel k = pick_reduce(p.n_src, p.vec_bytes, p.unroll);
        k<<<grid, p.block_threads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_fill_source(float *dst, uint64_t n, const tb_pattern &pat, int buffer_idx,
                               int num_sms, cudaStream_t stream)
{
    if (n == 0)
        return cudaSuccess;
    const int threads = 256;
    const uint64_t want = (n + threads - 1) / threads;
    const unsigned grid = (unsigned)std::min<uint64_t>(want, (uint64_t)num_sms * 8);
    switch (pat.kind) {
    case TB_PATTERN_DEFAULT:
        k_fill_default<<<grid, threads, 0, stream>>>(dst, n, (uint32_t)buffer_idx + 1u);
        break;
    case TB_PATTERN_COMPRESS: {
        CompressArgs a{};
        a.dst = dst;
        a.n = n;
        a.seed = pat.seed + (uint64_t)buffer_idx;
        uint32_t run = 0;
        for (int m = 0; m < 5; ++m) {
            run += pat.compress_pct[m];
            a.cum[m] = run;
        }
        const uint64_t lines = (n + 15) / 16;
        const unsigned g = (unsigned)std::min<uint64_t>((lines + threads - 1) / threads,
                                                        (uint64_t)num_sms * 8);
        k_fill_compress<<<g, threads, 0, stream>>>(a);
        break;
    }
    case TB_PATTERN_REPEAT: {
        RepeatArgs a;
        a.dst = dst;
        a.n = n;
        a.len = pat.repeat_len;
        for (uint32_t i = 0; i < pat.repeat_len; ++i)
            a.pat[i] = pat.repeat[i];
        k_fill_repeat<<<grid, threads, 0, stream>>>(a);
        break;
    }
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_gate(const volatile uint32_t *flag, uint32_t *status, uint64_t timeout_ns,
                        cudaStream_t stream)
{
    k_gate<<<1, 1, 0, stream>>>(flag, status, timeout_ns);
    return cudaGetLastError();
}

// The batch kernel needs more than the default 48 KiB of dynamic shared memory.
static bool batch_kernel_setup()
{
    static bool done = false;
    if (!done)
        done = cudaFuncSetAttribute(k_batch, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kBatchSmem) == cudaSuccess;
    return done;
}

int batch_ctas_per_sm()
{
    if (g_batch_ctas_per_sm == 0) {
        int blocks = 0;
        if (!batch_kernel_setup() ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_batch, kBatchThreads,
                                                          kBatchSmem) != cudaSuccess ||
            blocks < 1)
            blocks = 1;
        g_batch_ctas_per_sm = blocks;
    }
    return g_batch_ctas_per_sm;
}

cudaError_t launch_batch(const void *dev, const BatchPlan &plan, cudaStream_t stream,
                         uint32_t *status)
{
    if (plan.n_short == 0 && plan.n_long == 0)
        return cudaSuccess;
    if (!batch_kernel_setup())
        return cudaErrorInvalidValue;
    const char *base = static_cast<const char *>(dev);
    BatchArgs a;
    a.shorts = reinterpret_cast<const WorkItem *>(base);
    a.longs = a.shorts + plan.n_short;
    a.prefix = reinterpret_cast<const uint64_t *>(base + plan.prefix_offset);
    a.chunk_desc = reinterpret_cast<const uint32_t *>(base + plan.chunk_offset);
    a.status = status;
    a.long_bytes = plan.long_bytes;
    a.n_short = plan.n_short;
    a.chunks = plan.chunks;
    // Short copies only: no shared memory needed.
    const size_t smem = plan.chunks ? kBatchSmem : 0;
    k_batch<<<plan.grid, kBatchThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace tb

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

// Persistent grid of one wave.  Phase 1: CTA b copies the long-copy pieces
// [first[b], first[b+1]) - equal byte shares, so all CTAs finish it
// together.  Phase 2: short copies, longest first, dealt to warps in
// boustrophedon order (round r goes up the warp list when r is even and down
// when it is odd) so each warp's byte total stays close to the mean; each
// warp fetches its next item before copying the current one.
__global__ void __launch_bounds__(kBatchThreads) k_batch(const WorkItem *__restrict__ items,
                                                         const uint32_t *__restrict__ first,
                                                         uint32_t n_short)
{
    const uint32_t i1 = __ldg(first + blockIdx.x + 1);
    for (uint32_t i = __ldg(first + blockIdx.x); i < i1; ++i) {
        const WorkItem w = load_item(items + i);
        copy_range(reinterpret_cast<uint8_t *>(w.dst), reinterpret_cast<const uint8_t *>(w.src),
                   w.len, threadIdx.x, blockDim.x);
    }

    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t warps_per_cta = blockDim.x >> 5;
    const uint64_t W = (uint64_t)gridDim.x * warps_per_cta;
    const uint64_t wid = (uint64_t)blockIdx.x * warps_per_cta + (threadIdx.x >> 5);
    const WorkItem *shorts = items + __ldg(first + gridDim.x);
    auto index = [&](uint64_t r) { return r * W + ((r & 1) ? (W - 1 - wid) : wid); };
    uint64_t r = 0;
    while (r * W < n_short && index(r) >= n_short)
        ++r;
    if (r * W >= n_short)
        return;
    WorkItem cur = load_item(shorts + index(r));
    for (;;) {
        uint64_t rn = r + 1;
        while (rn * W < n_short && index(rn) >= n_short)
            ++rn;
        const bool more = rn * W < n_short;
        WorkItem nxt = cur;
        if (more)
            nxt = load_item(shorts + index(rn));
        copy_range(reinterpret_cast<uint8_t *>(cur.dst), reinterpret_cast<const uint8_t *>(cur.src),
                   cur.len, lane, 32u);
        if (!more)
            break;
        cur = nxt;
        r = rn;
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

int batch_ctas_per_sm()
{
    if (g_batch_ctas_per_sm == 0) {
        int blocks = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_batch, kBatchThreads, 0) !=
                cudaSuccess ||
            blocks < 1)
            blocks = 1;
        g_batch_ctas_per_sm = blocks;
    }
    return g_batch_ctas_per_sm;
}

cudaError_t launch_batch(const void *dev, const BatchPlan &plan, cudaStream_t stream)
{
    if (plan.n_long_items == 0 && plan.n_short == 0)
        return cudaSuccess;
    const WorkItem *items = static_cast<const WorkItem *>(dev);
    const uint32_t *first =
        reinterpret_cast<const uint32_t *>(static_cast<const char *>(dev) + plan.table_offset);
    k_batch<<<plan.grid, kBatchThreads, 0, stream>>>(items, first, plan.n_short);
    return cudaGetLastError();
}

}  // namespace tb

// Small kernels of libtb: the source-pattern fills ("TransferBench data
// validation", "Expected source pattern"), the device-side compare of
// validation (its validateDirect option), and the timing gate.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "tb_device.cuh"
#include "tb_internal.h"

namespace tb {
namespace {

using namespace dev;

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


// Device-side compare: the smallest byte index where a and b differ goes to
// *first (which starts at UINT64_MAX).  16-byte vectors when both pointers
// share their address modulo 16 (after a byte head), bytes otherwise.  A CTA
// stops early once a smaller index than its next position is known.
__device__ __forceinline__ uint32_t first_diff_byte(uint4 x, uint4 y)
{
    const uint32_t w[4] = {x.x ^ y.x, x.y ^ y.y, x.z ^ y.z, x.w ^ y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (w[i])
            return 4 * i + (__ffs(w[i]) - 1) / 8;
    return 16;
}

constexpr uint32_t kCompareUnroll = 4;

__global__ void k_compare(const uint8_t *a, const uint8_t *b, uint64_t n,
                          unsigned long long *first)
{
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t head = (16u - ((uintptr_t)a & 15u)) & 15u;
    if (head > n)
        head = n;
    const bool vec = (((uintptr_t)a ^ (uintptr_t)b) & 15u) == 0;
    if (!vec)
        head = n;
    for (uint64_t i = tid; i < head; i += stride)
        if (a[i] != b[i])
            atomicMin(first, (unsigned long long)i);
    if (!vec)
        return;
    const uint4 *va = reinterpret_cast<const uint4 *>(a + head);
    const uint4 *vb = reinterpret_cast<const uint4 *>(b + head);
    const uint64_t nv = (n - head) / 16;
    // kCompareUnroll vector pairs per thread and step, all loads issued
    // before the first compare.
    for (uint64_t v = tid, it = 0; v < nv; v += kCompareUnroll * stride, ++it) {
        // Every 64 vectors: stop once a difference before this position is known.
        if ((it & (64u / kCompareUnroll - 1u)) == 0 &&
            *reinterpret_cast<volatile unsigned long long *>(first) < head + v * 16)
            break;
        uint4 x[kCompareUnroll], y[kCompareUnroll];
#pragma unroll
        for (int u = 0; u < kCompareUnroll; ++u)
            if (v + u * stride < nv) {
                x[u] = __ldcs(va + v + u * stride);
                y[u] = __ldcs(vb + v + u * stride);
            }
#pragma unroll
        for (int u = 0; u < kCompareUnroll; ++u)
            if (v + u * stride < nv) {
                const uint32_t d = first_diff_byte(x[u], y[u]);
                if (d < 16)
                    atomicMin(first, (unsigned long long)(head + (v + u * stride) * 16 + d));
            }
    }
    const uint64_t t0 = head + nv * 16;
    for (uint64_t i = t0 + tid; i < n; i += stride)
        if (a[i] != b[i])
            atomicMin(first, (unsigned long long)i);
}

}  // namespace

cudaError_t launch_compare(const void *a, const void *b, uint64_t n, unsigned long long *first,
                           int num_sms, cudaStream_t stream)
{
    if (cudaMemsetAsync(first, 0xFF, sizeof(*first), stream) != cudaSuccess)
        return cudaGetLastError();
    if (n == 0)
        return cudaSuccess;
    const int threads = 512;
    const uint64_t want = (n / 16 + threads - 1) / threads + 1;
    const unsigned grid = (unsigned)std::min<uint64_t>(want, (uint64_t)num_sms * 4);
    k_compare<<<grid, threads, 0, stream>>>(static_cast<const uint8_t *>(a),
                                             static_cast<const uint8_t *>(b), n, first);
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
}  // namespace tb

// K1, the reduce-copy kernel of libtb (sm_103a), and its launch planning:
// dst[i] = src0[i] + ... + srcN-1[i] in float32, left to right ("TransferBench
// data validation", table "Number of sources / Expected value").
//
// HBM-bound streaming; no contraction, so no tensor cores.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "tb_device.cuh"
#include "tb_internal.h"

namespace tb {
namespace {

using namespace dev;

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
    uint32_t *status;      // nullable: set to 1 if a bounded wait expired
    uint32_t stages;       // bulk form: pipeline stages (2 .. kRMaxStages)
    uint64_t wait_ns;      // bulk form: limit of each wait for a tile's loads
    uint32_t early;        // 1: read sources before the launch ahead has finished
};

// Tiles of its own that a CTA of the vector form prefetches into L2 before
// waiting for the launch ahead.
constexpr uint32_t kEarlyTiles = 1;

// Prefetches a CTA's first kEarlyTiles tiles of every source into L2 (bulk
// prefetches; thread j * N + k takes tile j of source k).  Used before
// waiting for the launch ahead, whose writes never touch the sources.
template <int N, int VB>
__device__ __forceinline__ void prefetch_tiles(const ReduceArgs &a, uint64_t t0, uint64_t tile,
                                               uint64_t step, uint64_t vend)
{
    const uint32_t k = threadIdx.x % N, j = threadIdx.x / N;
    if (j >= kEarlyTiles)
        return;
    const uint64_t t = t0 + j * step;
    if (t >= vend)
        return;
    const uint64_t nv = min(tile, vend - t);
    const uint64_t p = reinterpret_cast<uint64_t>(a.src[k]) + (a.head + t * (VB / 4)) * 4;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)(nv * VB))
                 : "memory");
}

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

template <int N, int VB, int U, int MAXT = 512>
__global__ void __launch_bounds__(MAXT) k_reduce(const ReduceArgs a)
{
    const uint32_t tid = threadIdx.x;
    const uint32_t bd = blockDim.x;
    const SubRange sr = sub_range(a.nvec, a.nsub);
    pdl_launch_dependents();
    if constexpr (N > 0 && VB >= 16) {
        // Early launch: this CTA's first tiles of every source go to L2
        // while the launch ahead finishes.
        if (a.early)
            prefetch_tiles<N, VB>(a, sr.vbeg + (uint64_t)sr.part * bd * U, (uint64_t)bd * U,
                                  (uint64_t)sr.nparts * bd * U, sr.vend);
    }
    pdl_wait_prerequisite();

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
    pdl_launch_dependents();
    pdl_wait_prerequisite();
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

// ---------------------------------------------------------------------------
// K1, bulk form (1 to 16 sources, every pointer sharing its address modulo
// 16).  The body is cut into tiles of kTile bytes per source (bulk_tile).
// Thread 0 streams each tile's N source pieces into one of the launch's
// shared-memory stages with bulk copies (one mbarrier per stage); all threads add the
// pieces in place, left to right with __fadd_rn, into the stage's first
// buffer; after a proxy fence and a barrier, thread 0 writes that buffer out
// with a bulk copy and refills the previous stage.  With one source the
// tiles go straight from the load to the store (a bit copy).
// ---------------------------------------------------------------------------
constexpr uint32_t kRStages = 3;      // stages of a CTA that shares its SM
constexpr uint32_t kRMaxStages = 16;  // mbarriers in the 128-byte header
constexpr size_t kSmemOptIn = 232448;  // shared memory one CTA may opt into (227 KiB)
constexpr int kBulkThreads = 256;
// Auto engine: bulk_auto(N, bytes per source) picks the bulk form.
// Measured on GB300 (20 graphed iterations, rotation on, us per iteration,
// vector / bulk with the kSharedTile tiles; median of 5, two rounds):
//   1 source   8 MiB 3.26 / 3.31-3.41, 12 MiB 4.54 / 4.03, 16 MiB
//              5.05-5.10 / 4.69, 24 MiB 8.79 / 6.53 (32 KiB tiles);
//   2 sources  8 MiB 4.44 / 5.17-5.20, 12 MiB 6.95-7.05 / 5.56-5.61, 64 MiB
//              28.7 / 28.5, 256 MiB 121.0 / 111.4;
//   3 sources  4 MiB 3.52 / 5.00-5.05, 6 MiB 5.27-5.31 / 5.31, 8 MiB
//              5.77-5.81 / 5.56-5.61, 64 MiB 40.0 / 38.1, 256 MiB 151.5 / 145.2;
//   4 sources  4 MiB 4.18 / 5.11-5.20, 6 MiB 7.15-7.25 / 5.51, 32 MiB
//              26.1-26.2 / 25.4, 256 MiB 192.4 / 183.6;
//   5 sources  3 MiB 4.08 / 4.59-4.64, 4 MiB 7.20 / 4.90, 256 MiB 252.3 / 218.5;
//   6 sources  2 MiB 3.92-3.93 / 4.08, 3 MiB 4.79-4.80 / 4.49-4.54, 256 MiB
//              299.3 / 256.6;
//   7 sources  2 MiB 3.77-3.82 / 4.03, 3 MiB 8.17 / 4.90, 256 MiB 432.4 / 302.0;
//   8 sources  2 MiB 4.08-4.13 / 4.34-4.39, 3 MiB 7.36-7.37 / 5.36-5.41,
//              256 MiB 370.1 / 347.8;
// the bulk form ahead at every larger size measured (up to 256 MiB);
//   9 sources  1 MiB 5.8 / 3.4, 8 MiB 17.1 / 12.8, 256 MiB 376.6 / 365.1;
//   12 sources 2 MiB 9.0 / 5.5, 32 MiB 67.5 / 62.8, 256 MiB 490.6 / 478.4;
//   13 sources 1 MiB 7.5-7.6 / 4.1, 64 MiB 137.8-138.0 / 136.1-136.2, 256 MiB
//              532.3 / 522.2 (1 KiB tiles from 13 sources: 2 KiB stages fit
//              two CTAs per SM, not three, and ran 256 MiB in 562.0-562.7);
//   14 sources 1 MiB 8.1-8.2 / 4.2, 256 MiB 571.5-571.7 / 556.4;
//   15 sources 1 MiB 8.7 / 4.4, 64 MiB 157.4-157.6 / 161.5, 256 MiB
//              610.8-610.9 / 620.7-620.8;
//   16 sources 1 MiB 9.3-9.4 / 4.5-4.6, 32 MiB 87.6 / 84.6, 64 MiB 167.3 /
//              168.9-169.0, 256 MiB 650.0-650.2 / 647.5-647.6.
// So: one or two sources from 12 MiB, three from 8 MiB, four from 6 MiB,
// five from 4 MiB, six to eight from 3 MiB, nine to fourteen from 1 MiB,
// fifteen and sixteen from 1 MiB up to 32 MiB.
constexpr bool bulk_auto(int n_src, uint64_t bytes)
{
    constexpr uint64_t MiB = 1ull << 20;
    switch (n_src) {
    case 1:
    case 2:
        return bytes >= 12 * MiB;
    case 3:
        return bytes >= 8 * MiB;
    case 4:
        return bytes >= 6 * MiB;
    case 5:
        return bytes >= 4 * MiB;
    case 6:
    case 7:
    case 8:
        return bytes >= 3 * MiB;
    case 9:
    case 10:
    case 11:
    case 12:
    case 13:
    case 14:
        return bytes >= 1 * MiB;
    case 15:
    case 16:
        return bytes >= 1 * MiB && bytes < 32 * MiB;
    default:
        return false;
    }
}
// Target tiles per CTA of a bulk launch (while CTAs share SMs).  GB/s at 16
// / 64 / 256 MiB per source with 4 / 8 tiles: 3 sources 7463 / 7496, 7022 /
// 6994, 7401 / 7350; 5 sources 6851 / 6836, 7055 / 7012, 7369 / 7295;
// 7 sources 6218 / 6626, 6824 / 6983, 7171 / 7302; 8 sources 6208 / 6544,
// 6785 / 7032, 7049 / 7334 (2 tiles were slower for every count).
constexpr uint64_t bulk_tiles_per_cta(int n_src)
{
    return n_src >= 6 ? 8 : 4;
}

// Bytes per source of one tile.  With several sources the stages hold N
// pieces each.  While CTAs share SMs, small tiles keep more, shorter
// pipelines per SM than large ones with about the same bytes in flight,
// and the best size depends on N (20 graphed iterations, rotation on, GB/s
// at 16 / 64 / 256 MiB per source, tiles of 4 / 3 / 2 KiB):
//   2 sources 7357 / 7187 / 6398, 7077 / 6915 / 5718, 7206 / 7253 / 5758;
//   3 sources 7376 / 7548 / 7062, 6893 / 7041 / 6733, 7354 / 7401 / 7015;
//   4 sources 6895 / 7042 / 7134, 6815 / 6938 / 7020, 7173 / 7315 / 7331;
//   5 sources 6189 / 6268 / 6884, 6758 / 6764 / 7068, 6864 / 6877 / 7366;
//   6 sources 6106 / 6172 / 6449, 6926 / 6947 / 7082, 7181 / 7244 / 7307;
//   7 sources 5728 / 6130 / 6222, 6280 / 6625 / 6860, 6475 / 6728 / 7192;
//   8 sources 5821 / 6187 / 5833, 6472 / 6856 / 6454, 6649 / 7117 / 6766;
// 8 KiB tiles (three CTAs per SM for 3 sources) ran 3 x 256 MiB at
// 7190-7245 and 16 KiB at 6154-6162; 4-6 stages instead of 3 were slower.
// A CTA alone on its SM (the deep pipeline below) is bound by its
// per-tile barrier and issue instead, so it takes larger tiles (one CTA,
// 64 MiB per source, GB/s for 2 / 3 / 4 sources): 4 KiB 37 / 38 / 42,
// 8 KiB 49 / 59 / 65, 12 KiB 69 / 85 / 96, 16 KiB 86 / 104 / 94.
// One source is a plain relay, which moves more per SM with fewer, larger
// bulk copies: 32 KiB stages, two CTAs per SM (measured 3-4% faster on
// large copies than 8 KiB with eight CTAs per SM), alone or not.
constexpr int kBulkMaxSrcs = 16;
// Tile bytes per source while CTAs share SMs, by source count (index 1 is
// the relay's).
constexpr uint32_t kSharedTile[kBulkMaxSrcs + 1] = {0,    32768, 4096, 3072, 2048, 2048,
                                                    2048, 2048,  3072, 2048, 2048, 2048,
                                                    2048, 1024,  1024, 1024, 1024};
constexpr uint32_t kDeepTile = 16384;
constexpr uint32_t kDeepTileMany = 8192;  // 5 or more sources: two or more stages fit up to 14
constexpr uint32_t kRelayTile = 32768;

constexpr uint32_t bulk_tile(int n_src, bool deep)
{
    return n_src == 1 ? kRelayTile
                      : deep ? (n_src <= 4 ? kDeepTile : kDeepTileMany) : kSharedTile[n_src];
}

constexpr size_t bulk_smem_bytes(int n_src, uint32_t tile, uint32_t stages)
{
    return 128 + (size_t)stages * (size_t)n_src * tile;
}

// Most stages whose shared memory one CTA can hold (a CTA alone on its SM).
constexpr uint32_t bulk_max_stages(int n_src, uint32_t tile)
{
    const size_t fit = (kSmemOptIn - 128) / ((size_t)n_src * tile);
    return (uint32_t)(fit < kRMaxStages ? fit : kRMaxStages);
}

// The pipeline runs a.stages stages (kRStages when CTAs share an SM, up to
// bulk_max_stages when each CTA has an SM to itself, so one CTA keeps more
// bytes in flight).  Stage and phase advance incrementally: tile j uses
// stage j mod stages, on that stage's mbarrier phase floor(j / stages).
template <int N, uint32_t kTile>
__global__ void __launch_bounds__(kBulkThreads) k_reduce_bulk(const ReduceArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr uint32_t kTileVecs = kTile / 16;
    const uint32_t tid = threadIdx.x;
    const uint32_t nst = a.stages;
    const SubRange sr = sub_range(a.nvec, a.nsub);
    const uint64_t span = sr.vend > sr.vbeg ? sr.vend - sr.vbeg : 0;
    const uint64_t ntiles = (span + kTileVecs - 1) / kTileVecs;
    const uint64_t mine = ntiles > sr.part ? (ntiles - sr.part + sr.nparts - 1) / sr.nparts : 0;
    const uint32_t bars = smem_u32(smem);
    const uint32_t stages = smem_u32(smem + 128);
    const uint64_t sbase = (uint64_t)(a.head) * 4;
    pdl_launch_dependents();
    // An early launch issues its first tiles' loads before waiting for the
    // launch ahead (they read only sources); its first store comes after.
    if (!a.early)
        pdl_wait_prerequisite();

    // Tile j of this CTA: first body vector and vector count.
    auto tile = [&](uint64_t j, uint64_t &v0, uint32_t &nv) {
        v0 = sr.vbeg + (sr.part + j * sr.nparts) * kTileVecs;
        const uint64_t left = sr.vend - v0;
        nv = (uint32_t)(left < kTileVecs ? left : kTileVecs);
    };
    auto issue = [&](uint64_t j, uint32_t s) {
        uint64_t v0;
        uint32_t nv;
        tile(j, v0, nv);
        const uint32_t bar = bars + 8 * s;
        mbar_expect_tx(bar, N * nv * 16);
#pragma unroll
        for (int k = 0; k < N; ++k)
            bulk_copy_in(stages + (s * N + k) * kTile,
                         reinterpret_cast<uint64_t>(a.src[k]) + sbase + v0 * 16, nv * 16, bar);
    };

    if (mine > 0) {
        uint64_t issued = 0;  // tiles whose loads thread 0 has issued
        if (tid == 0) {
            for (uint32_t s = 0; s < nst; ++s)
                mbar_init(bars + 8 * s);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            for (; issued < mine && issued < (uint64_t)nst; ++issued)
                issue(issued, (uint32_t)issued);
        }
        if (a.early)
            pdl_wait_prerequisite();
        __syncthreads();
        uint32_t s = 0, parity = 0, prev = nst - 1;
        for (uint64_t j = 0; j < mine; ++j) {
            uint64_t v0;
            uint32_t nv;
            tile(j, v0, nv);
            bool expired = false;
            if (N > 1 || tid == 0) {
                expired = !mbar_wait_bounded(bars + 8 * s, parity, a.wait_ns);
                if (N > 1 && !expired) {
                    const uint32_t out = stages + s * N * kTile;
                    for (uint32_t v = tid; v < nv; v += kBulkThreads) {
                        Vec<16> acc, x;
                        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(acc.w[0]), "=r"(acc.w[1]), "=r"(acc.w[2]), "=r"(acc.w[3])
                                     : "r"(out + v * 16));
#pragma unroll
                        for (int k = 1; k < N; ++k) {
                            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(x.w[0]), "=r"(x.w[1]), "=r"(x.w[2]), "=r"(x.w[3])
                                         : "r"(out + k * kTile + v * 16));
                            vadd<16>(acc, x);
                        }
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(out + v * 16),
                                     "r"(acc.w[0]), "r"(acc.w[1]), "r"(acc.w[2]), "r"(acc.w[3])
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                }
            }
            if (N > 1)
                expired = __syncthreads_or(expired);
            if (expired) {
                if (tid == 0) {
                    if (a.status)
                        *reinterpret_cast<volatile uint32_t *>(a.status) = 1u;
                    // Let the loads already issued land (tiles j .. issued-1,
                    // each wait bounded again).
                    uint32_t ms = s, mp = parity;
                    for (uint64_t m = j; m < issued; ++m) {
                        mbar_wait_bounded(bars + 8 * ms, mp);
                        if (++ms == nst) {
                            ms = 0;
                            mp ^= 1u;
                        }
                    }
                    bulk_wait_all();
                }
                return;
            }
            if (tid == 0) {
                bulk_store(reinterpret_cast<uint64_t>(a.dst) + sbase + v0 * 16,
                           stages + s * N * kTile, nv * 16);
                // Refill the previous tile's stage once its store has read it.
                if (j >= 1 && issued < mine) {
                    bulk_wait_read_all_but_newest();
                    issue(issued, prev);
                    ++issued;
                }
            }
            prev = s;
            if (++s == nst) {
                s = 0;
                parity ^= 1u;
            }
        }
        if (tid == 0)
            bulk_wait_all();
    }

    if (a.early)
        pdl_wait_prerequisite();  // (returns at once if this thread waited already)
    if (blockIdx.x == 0 && tid < a.head)
        reduce_one<N>(a, tid);
    const uint64_t tail0 = a.head + a.nvec * 4;
    if (blockIdx.x == gridDim.x - 1 && tail0 + tid < a.n)
        reduce_one<N>(a, tail0 + tid);
}

using BulkKernel = void (*)(const ReduceArgs);

// The bulk kernel for n_src sources with the shared-SM tile, or the deep
// pipeline's tile when `deep`; *smem = its shared memory at `stages`.
BulkKernel pick_bulk(int n_src, bool deep, uint32_t stages, size_t *smem)
{
    *smem = bulk_smem_bytes(n_src, bulk_tile(n_src, deep), stages);
    switch (n_src) {
    case 1: return k_reduce_bulk<1, kRelayTile>;
    case 2: return deep ? k_reduce_bulk<2, kDeepTile> : k_reduce_bulk<2, kSharedTile[2]>;
    case 3: return deep ? k_reduce_bulk<3, kDeepTile> : k_reduce_bulk<3, kSharedTile[3]>;
    case 4: return deep ? k_reduce_bulk<4, kDeepTile> : k_reduce_bulk<4, kSharedTile[4]>;
    case 5: return deep ? k_reduce_bulk<5, kDeepTileMany> : k_reduce_bulk<5, kSharedTile[5]>;
    case 6: return deep ? k_reduce_bulk<6, kDeepTileMany> : k_reduce_bulk<6, kSharedTile[6]>;
    case 7: return deep ? k_reduce_bulk<7, kDeepTileMany> : k_reduce_bulk<7, kSharedTile[7]>;
    case 8: return deep ? k_reduce_bulk<8, kDeepTileMany> : k_reduce_bulk<8, kSharedTile[8]>;
    case 9: return deep ? k_reduce_bulk<9, kDeepTileMany> : k_reduce_bulk<9, kSharedTile[9]>;
    case 10: return deep ? k_reduce_bulk<10, kDeepTileMany> : k_reduce_bulk<10, kSharedTile[10]>;
    case 11: return deep ? k_reduce_bulk<11, kDeepTileMany> : k_reduce_bulk<11, kSharedTile[11]>;
    case 12: return deep ? k_reduce_bulk<12, kDeepTileMany> : k_reduce_bulk<12, kSharedTile[12]>;
    case 13: return deep ? k_reduce_bulk<13, kDeepTileMany> : k_reduce_bulk<13, kSharedTile[13]>;
    case 14: return deep ? k_reduce_bulk<14, kDeepTileMany> : k_reduce_bulk<14, kSharedTile[14]>;
    case 15: return deep ? k_reduce_bulk<15, kDeepTileMany> : k_reduce_bulk<15, kSharedTile[15]>;
    case 16: return deep ? k_reduce_bulk<16, kDeepTileMany> : k_reduce_bulk<16, kSharedTile[16]>;
    default: *smem = 0; return nullptr;
    }
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

// 1024-thread forms for a CTA alone on its SM: 2 to 4 sources, 32-byte
// vectors, two vectors per source in flight (one for 4 sources).  The
// 3-source, two-vector form spills 80 bytes at 64 registers and still
// measured fastest (131 against 110 GB/s per CTA with one vector).
ReduceKernel pick_wide(int n_src, int u)
{
    switch (n_src) {
    case 2: return u >= 2 ? k_reduce<2, 32, 2, 1024> : k_reduce<2, 32, 1, 1024>;
    case 3: return u >= 2 ? k_reduce<3, 32, 2, 1024> : k_reduce<3, 32, 1, 1024>;
    case 4: return k_reduce<4, 32, 1, 1024>;
    default: return nullptr;
    }
}

constexpr int kWideThreads = 1024;

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


}  // namespace

static int bulk_ctas_per_sm(int n_src)
{
    size_t smem = 0;
    BulkKernel k = pick_bulk(n_src, false, kRStages, &smem);
    return k ? resident_ctas((const void *)k, kBulkThreads, smem) : 0;
}

int reduce_ctas_per_sm(int n_src, int vec_bytes, int block_threads, int unroll)
{
    void *fn = block_threads > 512 ? (void *)pick_wide(n_src, unroll)
               : n_src <= 8 ? (void *)pick_reduce(n_src, vec_bytes, unroll)
                            : (vec_bytes == 16 ? (void *)k_reduce_many<16> : (void *)k_reduce_many<4>);
    return fn ? resident_ctas(fn, block_threads, 0) : 0;
}

int plan_reduce(ReducePlan *p, const void *const *srcs, int n_src, void *dst, uint64_t num_bytes,
                int num_subexec, int ctas_per_subexec, int block_threads, int vec_bytes, int unroll,
                uint32_t memset_byte, int num_sms, int engine)
{
    if (engine < 0 || engine > 2)
        return TB_EINVAL;
    if (!p || !dst || n_src < 0 || n_src > TB_MAX_SRCS || num_bytes % 4 != 0 || num_subexec < 0 ||
        ctas_per_subexec < 0 || block_threads < 0 || block_threads > 512 || block_threads % 32 != 0 ||
        unroll < 0 || unroll > 4 || unroll == 3 || num_sms < 1 ||
        (vec_bytes != 0 && vec_bytes != 4 && vec_bytes != 16 && vec_bytes != 32))
        return TB_EINVAL;
    if (n_src > 0 && !srcs)
        return TB_EINVAL;
    uintptr_t any = (uintptr_t)dst;
    const uintptr_t d0 = (uintptr_t)dst, d1 = d0 + num_bytes;
    if (d1 < d0)
        return TB_EINVAL;
    for (int k = 0; k < n_src; ++k) {
        if (!srcs[k])
            return TB_EINVAL;
        any |= (uintptr_t)srcs[k];
        // dst must not overlap a source: CTAs would read bytes others write.
        const uintptr_t s0 = (uintptr_t)srcs[k], s1 = s0 + num_bytes;
        if (s1 < s0 || (num_bytes > 0 && s0 < d1 && d0 < s1))
            return TB_EINVAL;
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

    // A fixed sub-executor split of at most one CTA per SM (TransferBench's
    // one block per sub-executor): every CTA has an SM to itself.
    const bool alone = ctas_per_subexec > 0 && num_subexec > 0 &&
                       (int64_t)num_subexec * ctas_per_subexec <= (int64_t)num_sms;

    // Engine: the bulk form needs 1..4 sources sharing a 16-byte alignment
    // and works in 16-byte units.  It is the default where bulk_auto says so
    // (large enough transfers), where it keeps more bytes in flight per SM
    // than per-thread
    // vector loads; below that, its per-tile pipeline latency costs more
    // than it saves and the vector form is faster.  A CTA alone on its SM
    // with 2 to 4 sources is limited by the bulk form's per-tile adds and
    // barrier instead; the vector form in a 1024-thread CTA with 32-byte
    // vectors (two per source in flight, one for 4 sources) streams more
    // (per CTA, 64 MiB per source: 126 against 86 GB/s for 2 sources, 142
    // against 104 for 3, 137 against 94 for 4, the bulk form with 16 KiB
    // tiles).  One source stays bulk (a relay: 105 against 88).
    const bool bulk_ok = n_src >= 1 && n_src <= kBulkMaxSrcs && vb >= 16 && vec_bytes != 32;
    if (engine == 2 && !bulk_ok)
        return TB_ENOTSUP;
    const bool vector_alone = alone && vb == 32 && n_src >= 2 && n_src <= 4;
    p->engine = (engine == 2 || (engine == 0 && bulk_ok && vec_bytes == 0 &&
                                 bulk_auto(n_src, num_bytes) && !vector_alone))
                    ? 2
                    : 1;
    if (p->engine == 2) {
        vb = 16;
        p->vec_bytes = 16;
    }

    if (vb > 4) {
        const uintptr_t mis = (uintptr_t)dst & (uintptr_t)(vb - 1);
        const uint64_t head = mis ? ((uint64_t)vb - mis) / 4 : 0;
        p->head = std::min<uint64_t>(head, p->n);
    }
    p->nvec = (p->n - p->head) / ((uint64_t)vb / 4);
    // Unroll: the largest that keeps two 512-thread CTAs per SM, or the
    // largest without spills when each CTA has an SM (and its registers) alone.
    p->unroll = vb == 4 ? 4
                        : std::min(unroll ? unroll : (alone ? max_unroll(n_src, vb)
                                                            : default_unroll(n_src, vb)),
                                   max_unroll(n_src, vb));
    if (n_src > 8)
        p->unroll = 2;  // k_reduce_many keeps two vectors per thread in flight
    // Block size: the caller's, else 512 or 256 threads, whichever keeps
    // more threads resident per SM at this kernel's register use (ties: 512).
    // Many sources need many registers: 4 to 6 sources fit one 512-thread
    // CTA per SM but three 256-thread ones (6 sources, 128 MiB: 6.2 against
    // 4.7-5.1 TB/s).
    p->block_threads = block_threads;
    if (block_threads == 0) {
        const int r512 = reduce_ctas_per_sm(n_src, vb, 512, p->unroll);
        const int r256 = reduce_ctas_per_sm(n_src, vb, 256, p->unroll);
        p->block_threads = 256 * r256 > 512 * r512 ? 256 : 512;
    }
    // A CTA alone on its SM with 2 to 4 sources and 32-byte vectors runs
    // 1024 threads (pick_wide) unless the caller fixed the block size.
    if (alone && p->engine == 1 && vb == 32 && n_src >= 2 && n_src <= 4 && block_threads == 0) {
        p->block_threads = kWideThreads;
        p->unroll = std::min(unroll ? unroll : 2, n_src <= 3 ? 2 : 1);
    }

    // Grid: S * ctas_per_subexec when the caller fixes the CTAs of each
    // sub-executor (1 = TransferBench's one block per sub-executor), else
    // the library's grid below, never fewer CTAs than sub-executors.  The
    // vector form launches at most one wave and no more CTAs than its body
    // has rounds of work (block_threads * unroll vectors each), but at least
    // one per SM: a small transfer is bound by launch and memory latency,
    // and CTAs without a full round add launch work without adding bytes in
    // flight (4 MiB: 152 CTAs 2.5 us against 304 CTAs 2.9 us per iteration).
    if (p->engine == 2)
        p->block_threads = kBulkThreads;
    const int per_sm = p->engine == 2 ? bulk_ctas_per_sm(n_src)
                                      : reduce_ctas_per_sm(n_src, vb, p->block_threads, p->unroll);
    if (per_sm < 1)
        return TB_ECUDA;
    const int64_t full = (int64_t)num_sms * per_sm;
    int64_t wave = full;
    bool whole_rounds = true;  // at least one full round of work per CTA
    if (p->engine == 1) {
        const uint64_t per_cta = (uint64_t)p->block_threads * (uint64_t)p->unroll;
        const uint64_t rounds = (p->nvec + per_cta - 1) / per_cta;
        wave = (int64_t)std::min<uint64_t>((uint64_t)full, std::max<uint64_t>((uint64_t)num_sms, rounds));
        whole_rounds = rounds >= (uint64_t)wave;
    } else {
        // Bulk form: many short-lived CTAs of about bulk_tiles_per_cta tiles
        // each rather than one resident wave with equal shares.  The CTA
        // scheduler then hands the next CTA to whichever SM finishes first,
        // so no SM ends the launch late (1 source, 2 GiB: 7.1 TB/s against
        // 6.6 with one wave; 3 sources, 3 x 256 MiB: 7.18 against 7.11).
        // Whole waves only: a partial last wave leaves SMs idle at the end
        // (1 source, 64 MiB: 1.7 waves 6.7 TB/s, one wave 7.2).
        const uint64_t tile_vecs = bulk_tile(n_src, false) / 16;
        const uint64_t tiles = (p->nvec + tile_vecs - 1) / tile_vecs;
        const uint64_t per_cta = bulk_tiles_per_cta(n_src);
        const uint64_t want = (tiles + per_cta - 1) / per_cta;
        const uint64_t waves = std::max<uint64_t>(1, std::min<uint64_t>(want / (uint64_t)full, 4096));
        wave = (int64_t)(waves * (uint64_t)full);
    }
    // numSubExec = 0 on the library's grid: one range over the whole grid,
    // its tiles dealt round robin, so each wave of CTAs sweeps neighbouring
    // tiles (bulk, 3 sources, 3 x 256 MiB: 7.22 against 6.98 TB/s with a
    // range per CTA; vector, 128 MiB: 2-11% faster for 1 to 12 sources) -
    // as long as every CTA gets a whole round: a smaller vector transfer
    // gives each CTA its own part of a round instead, so that all of them
    // load (4 MiB: 152 CTAs busy, not 64).  With the CTAs per sub-executor
    // fixed: one range per CTA.
    const int64_t S = num_subexec > 0 ? num_subexec
                      : (ctas_per_subexec == 0 && whole_rounds) ? 1 : wave;
    const int64_t G = ctas_per_subexec > 0 ? S * ctas_per_subexec : std::max<int64_t>(S, wave);
    if (G > (int64_t)INT32_MAX)
        return TB_EINVAL;
    p->num_subexec = (int)S;
    p->grid = (int)G;
    // Bulk form: three stages while CTAs share SMs; a grid of at most one CTA
    // per SM gives every CTA all the stages one CTA's shared memory holds, so
    // a lone CTA keeps several times more bytes in flight.
    if (p->engine == 2) {
        p->stages = kRStages;
        p->bulk_deep = 0;
        if (G <= (int64_t)num_sms) {
            const uint32_t deep = bulk_max_stages(n_src, bulk_tile(n_src, true));
            size_t smem = 0;
            BulkKernel k = pick_bulk(n_src, true, deep, &smem);
            if (k && deep >= 2 && resident_ctas((const void *)k, kBulkThreads, smem) >= 1) {
                p->stages = (int)deep;
                p->bulk_deep = 1;
            }
        }
        pick_bulk(n_src, p->bulk_deep != 0, (uint32_t)p->stages, &p->smem_bytes);
    }
    return TB_OK;
}

uint32_t plan_tile_bytes(const ReducePlan &p)
{
    return p.engine == 2 ? bulk_tile(p.n_src, p.bulk_deep != 0) : 0u;
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
    a.status = p.status;
    a.stages = (uint32_t)(p.stages > 0 ? p.stages : (int)kRStages);
    a.wait_ns = p.wait_ns;
    a.early = p.early ? 1u : 0u;
    if (p.n == 0)
        return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.block_threads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    if (p.engine == 2) {
        size_t smem = 0;
        BulkKernel k = pick_bulk(p.n_src, p.bulk_deep != 0, a.stages, &smem);
        if (!k || a.stages < 2 || a.stages > kRMaxStages ||
            resident_ctas((const void *)k, kBulkThreads, smem) < 1)
            return cudaErrorInvalidValue;
        cfg.blockDim = dim3(kBulkThreads);
        cfg.dynamicSmemBytes = smem;
        return cudaLaunchKernelEx(&cfg, k, a);
    }
    if (p.n_src > 8)
        return cudaLaunchKernelEx(&cfg, p.vec_bytes == 16 ? k_reduce_many<16> : k_reduce_many<4>, a,
                                  p.n_src);
    ReduceKernel k = p.block_threads > 512 ? pick_wide(p.n_src, p.unroll)
                                           : pick_reduce(p.n_src, p.vec_bytes, p.unroll);
    if (!k || (p.block_threads > 512 && resident_ctas((const void *)k, p.block_threads, 0) < 1))
        return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace tb

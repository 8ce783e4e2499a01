// K2, the batched descriptor copy of libtb (sm_103a): one launch over a
// packed (src, dst, len) work list (Mooncake RFC #5041, "Design of #5040").
// Long copies stream through a bulk (TMA) pipeline in shared memory; short
// copies go to warps.

#include <cuda_runtime.h>
#include <stdint.h>

#include "tb_device.cuh"
#include "tb_internal.h"

namespace tb {
namespace {

using namespace dev;

// ---------------------------------------------------------------------------
// K2: batched copy.  copy_range copies len bytes with `size` cooperating
// threads (a warp or a CTA), any alignment:
//   - head bytes until dst is 16-byte aligned, a byte per thread;
//   - body in 16-byte vectors: direct when src is then 16-byte aligned too,
//     otherwise every output vector is funnel-shifted out of the two aligned
//     source vectors that hold its bytes (both contain bytes of the range,
//     so no load leaves the source's aligned 16-byte words);
//   - tail bytes, a byte per thread.
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
    for (uint64_t b = rank; b < h; b += size)
        dst[b] = src[b];
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
    for (uint64_t b = done + rank; b < len; b += size)
        dst[b] = src[b];
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
    uint32_t *claim;             // work counter of the short copies (starts at 0)
    const WorkItem *shorts;      // n_short copies
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

// Short copies claimed per atomic: a warp takes kClaim items at a time and
// copies them side by side, 32 / kClaim lanes each, so their loads are in
// flight together.
constexpr uint32_t kClaim = 2;
constexpr uint32_t kLanesPerItem = 32 / kClaim;

// Persistent grid of one wave.
//   Long copies: their bytes form one stream of `chunks` equal chunks; CTA b
//   owns chunks b, b + G, ... (the same number for every CTA, the grid
//   sweeping the stream front to back).  Thread 0 moves the 16-byte-aligned
//   bodies with a bulk-copy pipeline through shared memory; warps 1.. copy
//   the leftover edges.
//   Short copies: every warp (warp 0 once its pipeline has drained) claims
//   kClaim items at a time from a counter in global memory and copies them
//   side by side, 32 / kClaim lanes each; it claims the next ones before
//   copying, so the claim's latency overlaps the copy.  Whichever warp is
//   free takes the next items, which balances the work without any ordering
//   on the host.
__global__ void __launch_bounds__(kBatchThreads, 4) k_batch(const BatchArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (a.chunks > 0) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < kStages; ++s)
                mbar_init(smem_u32(smem) + 8 * s);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        if (warp == 0) {
            if (lane == 0)
                bulk_pipeline(a, smem_u32(smem), smem_u32(smem + kBarBytes));
            __syncwarp();
        } else {
            long_edges(a, threadIdx.x - 32, blockDim.x - 32);
        }
    }

    const uint32_t n_short = a.n_short;
    uint32_t base = 0;
    if (lane == 0)
        base = atomicAdd(a.claim, kClaim);
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t group = lane / kLanesPerItem, rank = lane % kLanesPerItem;
    while (base < n_short) {
        uint32_t next = 0;
        if (lane == 0)
            next = atomicAdd(a.claim, kClaim);
        const uint32_t i = base + group;
        if (i < n_short) {
            const WorkItem w = load_item(a.shorts + i);
            copy_range(reinterpret_cast<uint8_t *>(w.dst), reinterpret_cast<const uint8_t *>(w.src),
                       w.len, rank, kLanesPerItem);
        }
        base = __shfl_sync(0xffffffffu, next, 0);
    }
}

}  // namespace

int batch_ctas_per_sm()
{
    return resident_ctas((const void *)k_batch, kBatchThreads, kBatchSmem);
}

cudaError_t launch_batch(const void *dev, const BatchPlan &plan, cudaStream_t stream,
                         uint32_t *status)
{
    if (plan.n_short == 0 && plan.n_long == 0)
        return cudaSuccess;
    if (batch_ctas_per_sm() < 1)
        return cudaErrorInvalidValue;
    char *base = static_cast<char *>(const_cast<void *>(dev));
    BatchArgs a;
    a.claim = reinterpret_cast<uint32_t *>(base);
    a.shorts = reinterpret_cast<const WorkItem *>(base + kBatchHeader);
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

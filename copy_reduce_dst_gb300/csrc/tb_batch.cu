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
// threads (a warp or part of one, or a CTA), any alignment:
//   - src and dst equal modulo 32: head bytes until dst is 32-byte aligned,
//     then 32-byte vectors (the 256-bit global access of sm_100-class GPUs);
//   - else: head bytes until dst is 16-byte aligned, then 16-byte vectors,
//     direct when src is then 16-byte aligned too, otherwise every output
//     vector is funnel-shifted out of the two aligned source vectors that
//     hold its bytes (both contain bytes of the range, so no load leaves the
//     source's aligned 16-byte words);
//   - tail bytes; head and tail go a byte per thread.
// The body goes in rounds: each thread issues all its loads of a round,
// predicated on the range, before its stores, so a range of up to
// size * 32 * kWideUnroll bytes (32-byte path) costs one memory round trip.
// The unrolls are the largest that compile without spilling at the kernel's
// 64 registers (four 256-thread CTAs per SM); spilling variants (4 or 8
// wide vectors) measured 1.3-1.7x slower on the short copies.
// ---------------------------------------------------------------------------
constexpr int kWideUnroll = 2;    // 32-byte vectors per thread and round
constexpr int kNarrowUnroll = 2;  // 16-byte vectors per thread and round
constexpr int kShiftUnroll = 1;   // funnel-shifted 16-byte vectors per thread and round

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

__device__ __forceinline__ void st32(void *p, const Vec<32> &v)
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
                 "r"(v.w[7]));
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

__device__ __forceinline__ void copy_bytes(uint8_t *dst, const uint8_t *src, uint64_t len,
                                           uint32_t rank, uint32_t size)
{
    for (uint64_t b = rank; b < len; b += size)
        dst[b] = src[b];
}

__device__ __forceinline__ void copy_range(uint8_t *dst, const uint8_t *src, uint64_t len,
                                           uint32_t rank, uint32_t size)
{
    const uint32_t align = ((((uintptr_t)src ^ (uintptr_t)dst) & 31u) == 0) ? 32u : 16u;
    uint64_t h = (align - ((uintptr_t)dst & (align - 1))) & (align - 1);
    if (h > len)
        h = len;
    copy_bytes(dst, src, h, rank, size);
    dst += h;
    src += h;
    len -= h;

    uint64_t done;
    if (align == 32) {
        const uint64_t nv = len >> 5;
        for (uint64_t v = rank; v < nv; v += kWideUnroll * (uint64_t)size) {
            Vec<32> r[kWideUnroll];
#pragma unroll
            for (int u = 0; u < kWideUnroll; ++u)
                if (v + u * (uint64_t)size < nv)
                    vload<32>(r[u], src + (v + u * (uint64_t)size) * 32);
#pragma unroll
            for (int u = 0; u < kWideUnroll; ++u)
                if (v + u * (uint64_t)size < nv)
                    st32(dst + (v + u * (uint64_t)size) * 32, r[u]);
        }
        done = nv << 5;
    } else {
        const uint64_t nv = len >> 4;
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        const uint32_t sh = (uint32_t)((uintptr_t)src & 15u);
        if (sh == 0) {
            const uint4 *s = reinterpret_cast<const uint4 *>(src);
            for (uint64_t v = rank; v < nv; v += kNarrowUnroll * (uint64_t)size) {
                uint4 r[kNarrowUnroll];
#pragma unroll
                for (int u = 0; u < kNarrowUnroll; ++u)
                    if (v + u * (uint64_t)size < nv)
                        r[u] = ld16(s + v + u * size);
#pragma unroll
                for (int u = 0; u < kNarrowUnroll; ++u)
                    if (v + u * (uint64_t)size < nv)
                        st16(d + v + u * size, r[u]);
            }
        } else {
            const uint4 *s = reinterpret_cast<const uint4 *>(src - sh);
            const uint32_t q = sh >> 2, rbits = (sh & 3u) * 8u;
            for (uint64_t v = rank; v < nv; v += kShiftUnroll * (uint64_t)size) {
                uint4 lo[kShiftUnroll], hi[kShiftUnroll];
#pragma unroll
                for (int u = 0; u < kShiftUnroll; ++u)
                    if (v + u * (uint64_t)size < nv) {
                        lo[u] = ld16(s + v + u * size);
                        hi[u] = ld16(s + v + u * size + 1);
                    }
#pragma unroll
                for (int u = 0; u < kShiftUnroll; ++u)
                    if (v + u * (uint64_t)size < nv)
                        st16(d + v + u * size, shift_pair(lo[u], hi[u], q, rbits));
            }
        }
        done = nv << 4;
    }
    copy_bytes(dst + done, src + done, len - done, rank, size);
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
    uint32_t claim_items;        // short copies a warp takes at a time: 1 or 2
    uint64_t wait_ns;            // limit of each wait for a block's load
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
    uint32_t i = 0;
    for (; i < issued; ++i) {
        const uint32_t s = i % kStages;
        if (!mbar_wait_bounded(bars + 8 * s, (uses >> s) & 1u, a.wait_ns)) {
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
        // Let the loads still in flight land: blocks i .. issued-1, at most
        // one per stage, each on its stage's pending phase (waits bounded).
        for (uint32_t m = i; m < issued; ++m) {
            const uint32_t k = m % kStages;
            mbar_wait_bounded(bars + 8 * k, (uses >> k) & 1u);
        }
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

// Short copies.  A warp takes C items at a time (C = 1 or 2) and copies them
// side by side, 32 / C lanes each, so their loads are in flight together.
// Its first C items are fixed by its index among the warps that start on
// short copies (no atomic); the items past those first rounds are claimed
// from the counter, each warp claiming its next items before copying the
// current ones so that the claim's latency overlaps the copy.
template <uint32_t C>
__device__ __forceinline__ void short_copies(const BatchArgs &a, uint32_t first, uint32_t dyn_base,
                                             bool dynamic, uint32_t lane)
{
    constexpr uint32_t kLanes = 32 / C;
    const uint32_t n_short = a.n_short;
    const uint32_t group = lane / kLanes, rank = lane % kLanes;
    uint32_t base = first;
    if (base >= n_short && dynamic) {
        uint32_t c = 0;
        if (lane == 0)
            c = dyn_base + atomicAdd(a.claim, C);
        base = __shfl_sync(0xffffffffu, c, 0);
    }
    while (base < n_short) {
        uint32_t next = n_short;
        if (dynamic && lane == 0)
            next = dyn_base + atomicAdd(a.claim, C);
        const uint32_t i = base + group;
        if (i < n_short) {
            const WorkItem w = load_item(a.shorts + i);
            copy_range(reinterpret_cast<uint8_t *>(w.dst), reinterpret_cast<const uint8_t *>(w.src),
                       w.len, rank, kLanes);
        }
        base = __shfl_sync(0xffffffffu, next, 0);
    }
}

// A grid of up to kBatchWaves waves of resident CTAs (short-lived CTAs let
// the scheduler balance the SMs' finishing times).
//   Long copies: their bytes form one stream of `chunks` equal chunks; CTA b
//   owns chunks b, b + G, ... (the same number for every CTA, the grid
//   sweeping the stream front to back).  Thread 0 moves the 16-byte-aligned
//   bodies with a bulk-copy pipeline through shared memory; warps 1.. copy
//   the leftover edges.
//   Short copies (short_copies): the warps free at the start (all of them,
//   or warps 1.. when there are long chunks) take a first claim_items items
//   each by warp index; the rest are claimed from a counter in global memory
//   by whichever warp is free, warp 0 joining once its pipeline has
//   drained, which balances the work without any ordering on the host.
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

    // Warps that start on short copies, and this warp's index among them.
    const uint32_t wpc = blockDim.x >> 5;
    const bool busy0 = a.chunks > 0;  // warp 0 runs the bulk pipeline first
    const uint32_t starters = gridDim.x * (busy0 ? wpc - 1 : wpc);
    const bool starter = !(busy0 && warp == 0);
    const uint32_t sidx = blockIdx.x * (busy0 ? wpc - 1 : wpc) + (busy0 ? warp - 1 : warp);
    const uint32_t C = a.claim_items;
    const uint32_t fixed = starters * C;  // items taken by index
    const bool dynamic = fixed < a.n_short;
    const uint32_t first = starter ? sidx * C : a.n_short;
    if (C == 1)
        short_copies<1>(a, first, fixed, dynamic, lane);
    else
        short_copies<2>(a, first, fixed, dynamic, lane);
}

}  // namespace

int batch_ctas_per_sm()
{
    return resident_ctas((const void *)k_batch, kBatchThreads, kBatchSmem);
}

cudaError_t launch_batch(const void *dev, const BatchPlan &plan, cudaStream_t stream,
                         uint32_t *status, uint64_t wait_ns)
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
    a.claim_items = batch_claim_items(plan);
    a.wait_ns = wait_ns;
    // Short copies only: no shared memory needed.
    const size_t smem = plan.chunks ? kBatchSmem : 0;
    k_batch<<<plan.grid, kBatchThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace tb

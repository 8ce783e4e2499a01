// K2, the batched descriptor copy of libtb (sm_103a): one launch over a
// packed (src, dst, len) work list (Mooncake RFC #5041, "Design of #5040").
// Long copies stream through a bulk (TMA) pipeline in shared memory; short
// copies go to warps, through shared memory by asynchronous copies.

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
// The unrolls are the largest that compiled without spilling at 64
// registers; spilling variants (4 or 8 wide vectors) measured 1.3-1.7x
// slower on the short copies.  Short copies whose src and dst are equal
// modulo 16 no longer come here: they go through the shared-memory pipe
// below, which keeps more bytes in flight than a round of registers.
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

// A short copy whose src and dst differ modulo 16, by one warp: the same
// steps as copy_range takes for such a pair (head bytes to a 16-byte
// destination boundary, one funnel-shifted 16-byte vector per lane and
// round, tail bytes) without the branches a warp never reaches there, so
// the short-copy kernels keep few registers (the general form took the
// short-only kernel from 69 to 80 registers and into spills).
__device__ __forceinline__ void copy_shifted_warp(uint8_t *dst, const uint8_t *src, uint64_t len,
                                                  uint32_t lane)
{
    uint64_t h = (16u - ((uintptr_t)dst & 15u)) & 15u;
    if (h > len)
        h = len;
    if (lane < h)
        dst[lane] = src[lane];
    dst += h;
    src += h;
    len -= h;
    const uint64_t nv = len >> 4;
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    const uint32_t sh = (uint32_t)((uintptr_t)src & 15u);
    const uint4 *s = reinterpret_cast<const uint4 *>(src - sh);
    const uint32_t q = sh >> 2, rbits = (sh & 3u) * 8u;
    for (uint64_t v = lane; v < nv; v += 32) {
        // Both aligned words hold bytes of the range when sh != 0.
        const uint4 lo = ld16(s + v);
        const uint4 hi = sh ? ld16(s + v + 1) : lo;
        st16(d + v, sh ? shift_pair(lo, hi, q, rbits) : lo);
    }
    const uint64_t done = nv << 4;
    if (lane < len - done)
        dst[done + lane] = src[done + lane];
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
    uint32_t claim_items;        // short copies a warp takes by its index: 1 or 2
    uint64_t wait_ns;            // limit of each wait for a block's load
    uint32_t *done_count;        // nullable: completion signal (BatchDone)
    uint32_t *done_word;
    uint32_t done_base;
    uint32_t done_seq;
};

// The completion signal: called by every thread of a CTA at its end.  Every
// warp's reads of the work list have returned their values (they were used)
// before the barrier, so thread 0's add comes after all of them; the add
// that returns done_base + grid - 1 is the launch's last.
__device__ __forceinline__ void signal_done(const BatchArgs &a)
{
    if (!a.done_count)
        return;
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(a.done_count, 1u) == a.done_base + gridDim.x - 1u)
        *reinterpret_cast<volatile uint32_t *>(a.done_word) = a.done_seq;
}

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

// Short copies through shared memory.  Each warp streams its copies as
// pieces of up to 32 * U 16-byte units through a ring of S piece slots:
// every lane issues asynchronous 16-byte global -> shared copies (cp.async,
// no registers held) for its units of a piece and commits them as a group,
// then waits for the oldest piece in the ring and stores that one from
// shared memory.  A warp so keeps S - 1 pieces landing while it stores one,
// and no register holds data in flight.  Each lane reads back only the
// units it loaded, so no barrier is needed.  Measured on GB300 (47,520
// short copies of 64 B - 16 KiB alone / the 47,540 batch with long copies):
// register rounds 62.5 / 142.7 us; S = 2: U = 8 55.4, U = 4 57.0 /
// U = 4 141.6, U = 8 143.7; S = 4: U = 4 54.5 / U = 2 141.0; S = 8: U = 2
// 58.4 / U = 1 143.5; U = 16 (one CTA per SM) 71.1.  Launches with long
// copies take 4 KiB of slots per warp beside the bulk stages (two CTAs per
// SM); launches of short copies only take one of the k_short shapes.
constexpr int kMixedUnits = 2;  // U beside the long copies' bulk stages
constexpr int kMixedSlots = 4;
// Short copies a warp claims from the counter with one atomic: fewer
// atomics on the one counter address (47,540 batch: 138.2 us at 4, 2 or 8
// against 141.3 at 1; its short copies alone 52.1 against 54.9).
constexpr uint32_t kClaimBlock = 4;

template <int U>
__host__ __device__ constexpr uint32_t piece_bytes()
{
    return 32u * U * 16u;
}

template <int U, int S>
__host__ __device__ constexpr size_t warp_stage_bytes()
{
    return S * (size_t)piece_bytes<U>();
}

template <int U, int S>
__host__ __device__ constexpr size_t short_smem_bytes()
{
    return (kBatchThreads / 32) * warp_stage_bytes<U, S>();
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void *g)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(g) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds16(uint32_t smem)
{
    uint4 r;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem)
                 : "memory");
    return r;
}

// The ring: slot `cur` is free; the S - 1 pieces in flight are q[0]
// (oldest, in slot cur + 1) .. q[S - 2] (newest, in slot cur - 1), slots
// taken mod S.  It starts with S - 1 empty pieces (nv = 0), so every push
// runs the same steps: load into slot cur, commit, wait until at most S - 1
// groups are pending (the oldest piece has landed), store q[0], shift.
// While fewer than S groups were ever committed the oldest entry is an
// empty piece and the wait returns at once.
template <int U, int S>
struct ShortPipe {
    struct Piece {
        uint64_t dst;  // 16-byte aligned
        uint32_t nv;   // 16-byte units, 0 = nothing
    };
    uint32_t base;  // this warp's S slots
    uint32_t lane;
    uint32_t cur;
    Piece q[S - 1];

    __device__ ShortPipe(uint32_t b, uint32_t l) : base(b), lane(l), cur(0)
    {
#pragma unroll
        for (int j = 0; j < S - 1; ++j)
            q[j] = Piece{0ull, 0u};
    }
    __device__ uint32_t unit(uint32_t slot, int u) const
    {
        return base + (((slot * U + (uint32_t)u) * 32u + lane) << 4);
    }
    __device__ void store(const Piece &p, uint32_t slot) const
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t k = lane + 32u * u;
            if (k < p.nv)
                st16(reinterpret_cast<uint4 *>(p.dst) + k, lds16(unit(slot, u)));
        }
    }
    // Loads a piece of nv <= 32 * U units (src and dst 16-byte aligned)
    // into slot cur, then stores the oldest piece in flight.
    __device__ void push(const uint8_t *src, uint64_t dst, uint32_t nv)
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t k = lane + 32u * u;
            if (k < nv)
                cp_async16(unit(cur, u), src + 16ull * k);
        }
        cp_async_commit();
        const uint32_t oldest = cur + 1 == S ? 0u : cur + 1;
        cp_async_wait<S - 1>();
        store(q[0], oldest);
#pragma unroll
        for (int j = 0; j + 1 < S - 1; ++j)
            q[j] = q[j + 1];
        q[S - 2] = Piece{dst, nv};
        cur = oldest;
    }
    // Stores every piece still in flight, oldest first.
    __device__ void flush()
    {
        cp_async_wait<0>();
#pragma unroll
        for (int j = 0; j < S - 1; ++j) {
            const uint32_t slot = (cur + 1 + (uint32_t)j) % S;
            store(q[j], slot);
            q[j] = Piece{0ull, 0u};
        }
    }
};

// One short copy by a whole warp.  src and dst equal modulo 16: up to 15
// head bytes (lanes 0..14) and 15 tail bytes (lanes 16..30) go a byte per
// lane, loaded before the body's pieces are pushed and stored after, so
// their latency overlaps the pipe's; the body goes through the pipe.  Any
// other alignment: copy_shifted_warp through registers.
template <int U, int S>
__device__ __forceinline__ void short_item(ShortPipe<U, S> &p, const WorkItem &w, uint32_t lane)
{
    const uint8_t *s = reinterpret_cast<const uint8_t *>(w.src);
    uint8_t *d = reinterpret_cast<uint8_t *>(w.dst);
    if (((w.src ^ w.dst) & 15u) != 0) {
        copy_shifted_warp(d, s, w.len, lane);
        return;
    }
    const uint64_t h = min((uint64_t)((16u - (w.dst & 15u)) & 15u), w.len);
    const uint64_t body = (w.len - h) & ~(uint64_t)15;
    const uint64_t t = w.len - h - body;
    const bool edge = lane < h || (lane >= 16 && lane - 16 < t);
    const uint64_t eoff = lane < 16 ? lane : h + body + (lane - 16);
    uint8_t eb = 0;
    if (edge)
        eb = s[eoff];
    for (uint64_t off = 0; off < body; off += piece_bytes<U>()) {
        const uint32_t nv = (uint32_t)min((body - off) >> 4, (uint64_t)(32u * U));
        p.push(s + h + off, w.dst + h + off, nv);
    }
    if (edge)
        d[eoff] = eb;
}

// The short copies of one warp: up to claim_items items by its index
// among the warps that start on short copies (first, first + stride, ...;
// no atomic), then blocks of kClaimBlock items claimed from the counter.
// Lane 0 keeps one claim in flight and the descriptor of the next item is
// loaded before the current item is copied, so neither latency stalls the
// pipe.
template <int U, int S>
__device__ __forceinline__ void short_copies(const BatchArgs &a, uint32_t first, uint32_t stride,
                                             uint32_t dyn_base, bool dynamic, uint32_t lane,
                                             uint32_t pipe_smem)
{
    const uint32_t n = a.n_short;
    const uint64_t fixed_end = min(dyn_base, n);  // copies taken by index
    uint32_t pending = n;  // lane 0: the claim in flight
    if (dynamic && lane == 0)
        pending = dyn_base + atomicAdd(a.claim, kClaimBlock);
    uint64_t blk_end = 0;  // end of the claimed block being copied
    auto after = [&](uint32_t i) -> uint32_t {
        if ((uint64_t)i + stride < fixed_end)
            return i + stride;
        if (i >= dyn_base && (uint64_t)i + 1 < blk_end)
            return i + 1;
        const uint32_t v = __shfl_sync(0xffffffffu, pending, 0);
        if (dynamic && v < n && lane == 0)
            pending = dyn_base + atomicAdd(a.claim, kClaimBlock);
        blk_end = min((uint64_t)v + kClaimBlock, (uint64_t)n);
        return v;
    };
    uint32_t cur = first < n ? first : after(UINT32_MAX - 1);
    if (cur >= n)
        return;
    ShortPipe<U, S> p(pipe_smem, lane);
    WorkItem w = load_item(a.shorts + cur);
    // A launch that follows another on its stream may have started early
    // (programmatic dependent launch): its own work list is read already,
    // but no source or destination byte is touched before the launch ahead
    // has finished and its writes are visible.
    pdl_wait_prerequisite();
    for (;;) {
        const uint32_t nx = after(cur);
        WorkItem wn{0, 0, 0};
        if (nx < n)
            wn = load_item(a.shorts + nx);
        short_item(p, w, lane);
        if (nx >= n)
            break;
        cur = nx;
        w = wn;
    }
    p.flush();
}

// k_batch: a launch with long copies, over up to kBatchWaves waves of
// resident CTAs (short-lived CTAs let the scheduler balance the SMs'
// finishing times).  U, S: the short copies' ring (see ShortPipe).
//   Long copies: their bytes form one stream of `chunks` equal chunks; CTA b
//   owns chunks b, b + G, ... (the same number for every CTA, the grid
//   sweeping the stream front to back).  Thread 0 moves the 16-byte-aligned
//   bodies with a bulk-copy pipeline through shared memory; warps 1.. copy
//   the leftover edges.
//   Short copies (short_copies, each warp through its own shared-memory
//   pipe): warps 1.. take up to claim_items items each by warp index
//   (warp w: w, w + starters); the rest are claimed kClaimBlock at a time
//   from a counter in global memory by whichever warp is free, warp 0
//   joining once its pipeline has drained, which balances the work without
//   any ordering on the host.
template <int U, int S>
__global__ void __launch_bounds__(kBatchThreads, 3) k_batch(const BatchArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_launch_dependents();
    pdl_wait_prerequisite();
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
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

    // Warps 1.. start on short copies; warp 0 only claims.
    const uint32_t wpc = blockDim.x >> 5;
    const uint32_t starters = gridDim.x * (wpc - 1);
    const uint32_t fixed = starters * a.claim_items;  // items taken by index
    const uint32_t first = warp == 0 ? a.n_short : blockIdx.x * (wpc - 1) + warp - 1;
    short_copies<U, S>(a, first, starters, fixed, fixed < a.n_short, lane,
                       smem_u32(smem) + (uint32_t)kBatchSmem +
                           warp * (uint32_t)warp_stage_bytes<U, S>());
    signal_done(a);
}

// k_short: a launch of short copies only, over up to kShortWaves waves.
// Every warp starts on short copies: up to claim_items by warp index, then
// blocks claimed from the counter.  Its ring (U units per lane and piece, S
// slots) and the CTAs it keeps per SM (MINB, which bounds its registers)
// form a shape, chosen per launch (see short_shape_for).  Measured on GB300
// (kernel events, median of 40; shapes 1 / 2 / four 1 KiB slots at 5 CTAs
// per SM): 3840 x 2112 B 8.9-9.7 / 8.4-8.6 / 9.8-9.9 us; 7200 x 512 B-16 KiB
// 14.5-14.6 / 14.9 / 16.6 us; 47,520 x 64 B-16 KiB 50.8 us for all three.
// The old short-only launch (k_batch with four 2 KiB slots, 80 registers)
// took 6.1-8.5 us on the 3840 pages by ncu, shape 2 takes 5.4-6.1.
template <int U, int S, int MINB>
__global__ void __launch_bounds__(kBatchThreads, MINB) k_short(const BatchArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_launch_dependents();
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t wpc = blockDim.x >> 5;
    const uint32_t starters = gridDim.x * wpc;
    const uint32_t fixed = starters * a.claim_items;
    short_copies<U, S>(a, blockIdx.x * wpc + warp, starters, fixed, fixed < a.n_short, lane,
                       smem_u32(smem) + warp * (uint32_t)warp_stage_bytes<U, S>());
    signal_done(a);
}

// The shapes of k_short, by number (1-based; 0 names k_batch).
struct ShapeInfo {
    const void *kernel;
    size_t smem;
};

template <int U, int S, int MINB>
ShapeInfo shape_info()
{
    return ShapeInfo{(const void *)k_short<U, S, MINB>, short_smem_bytes<U, S>()};
}

ShapeInfo shape(int k)
{
    switch (k) {
    case 1:
        return shape_info<4, 4, 3>();  // 4 slots of 2 KiB per warp, 3 CTAs per SM
    case 2:
        return shape_info<4, 2, 5>();  // 2 slots of 2 KiB per warp, 5 CTAs per SM
    default:
        return ShapeInfo{(const void *)k_batch<kMixedUnits, kMixedSlots>,
                         kBatchSmem + short_smem_bytes<kMixedUnits, kMixedSlots>()};
    }
}

}  // namespace

int batch_ctas_per_sm(int k)
{
    if (k < 0 || k > kShortShapes)
        return 0;
    const ShapeInfo info = shape(k);
    return resident_ctas(info.kernel, kBatchThreads, info.smem);
}

cudaError_t launch_batch(const void *dev, const BatchPlan &plan, cudaStream_t stream,
                         uint32_t *status, uint64_t wait_ns, const BatchDone &done, bool pdl)
{
    if (plan.n_short == 0 && plan.n_long == 0)
        return cudaSuccess;
    // A launch with long copies runs k_batch, one of short copies only a
    // k_short shape.
    const int k = plan.chunks ? 0 : plan.shape;
    if ((plan.chunks == 0) == (k == 0) || batch_ctas_per_sm(k) < 1)
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
    a.done_count = done.count && done.word ? done.count : nullptr;
    a.done_word = done.word;
    a.done_base = done.base;
    a.done_seq = done.seq;
    const ShapeInfo info = shape(k);
    void *args[] = {&a};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kBatchThreads);
    cfg.dynamicSmemBytes = info.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, info.kernel, args);
}

}  // namespace tb

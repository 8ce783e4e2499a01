// Host-side packing of the batched copy: turns a (src, dst, len) descriptor
// array into the work list one k_batch launch reads.
//
// Layout of a packed launch (one device buffer):
//   uint32_t claim; (16-byte header)  work counter of the short copies,
//                                      uploaded as 0 with every launch
//   WorkItem shorts[n_short]          copies of at most small_max bytes, in
//                                      descriptor order (warps claim them)
//   WorkItem longs[n_long]            the longer copies, in descriptor order
//   uint64_t prefix[n_long + 1]       offset of each long copy in the stream
//                                      of all long-copy bytes; last = total
//   uint32_t chunk_desc[C + 1]        the long copy holding chunk c's first byte
// The long-copy stream is cut into C = grid * m chunks of equal size (cuts
// on 64-byte stream offsets); CTA b copies chunks b, b + grid, ... so every
// CTA gets exactly m chunks and the grid sweeps the stream front to back.
//
// Packing is one pass over the descriptors (check, count, append) plus a
// pass over the long copies; nothing is sorted, because the kernel balances
// the short copies itself by claiming them from the counter.

#include <algorithm>
#include <cstring>
#include <vector>

#include "tb_internal.h"

namespace tb {

size_t batch_buffer_bytes(uint64_t descs)
{
    return kBatchHeader + (size_t)descs * (sizeof(WorkItem) + sizeof(uint64_t)) +
           sizeof(uint64_t) + ((size_t)kMaxChunks + 1) * sizeof(uint32_t);
}

static inline bool bad_range(uint64_t src, uint64_t dst, uint64_t len)
{
    return src == 0 || dst == 0 || src + len < src || dst + len < dst;
}

int count_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, BatchCounts *c,
                size_t *bad, uint64_t ce_min)
{
    const tb_copy_desc *__restrict__ d = desc;
    const uint64_t ce = ce_min ? ce_min : UINT64_MAX;
    uint64_t descs = 0, bytes = 0, n_short = 0, n_long = 0, long_bytes = 0, n_ce = 0, ce_bytes = 0;
    for (size_t i = 0; i < n; ++i) {
        const uint64_t src = d[i].src, dst = d[i].dst, len = d[i].len;
        if (len == 0)
            continue;
        if (bad_range(src, dst, len)) {
            if (bad)
                *bad = i;
            return TB_EINVAL;
        }
        ++descs;
        bytes += len;
        if (len >= ce) {
            ++n_ce;
            ce_bytes += len;
        } else if (len <= small_max) {
            ++n_short;
        } else {
            ++n_long;
            long_bytes += len;
        }
    }
    *c = BatchCounts{descs, n_short, n_long, long_bytes, bytes, n_ce, ce_bytes};
    return TB_OK;
}

int gather_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, uint64_t ce_min,
                 void *buf, WorkItem *longs, BatchCounts *c, size_t *bad)
{
    const tb_copy_desc *__restrict__ d = desc;
    WorkItem *__restrict__ shorts =
        reinterpret_cast<WorkItem *>(static_cast<char *>(buf) + kBatchHeader);
    WorkItem *__restrict__ lg = longs;
    const uint64_t ce = ce_min ? ce_min : UINT64_MAX;
    uint64_t descs = 0, bytes = 0, ns = 0, nl = 0, long_bytes = 0, n_ce = 0, ce_bytes = 0;
    for (size_t i = 0; i < n; ++i) {
        const uint64_t src = d[i].src, dst = d[i].dst, len = d[i].len;
        if (len == 0)
            continue;
        if (bad_range(src, dst, len)) {
            if (bad)
                *bad = i;
            return TB_EINVAL;
        }
        ++descs;
        bytes += len;
        if (len >= ce) {
            ++n_ce;
            ce_bytes += len;
        } else if (len <= small_max) {
            shorts[ns++] = WorkItem{src, dst, len};
        } else {
            lg[nl++] = WorkItem{src, dst, len};
            long_bytes += len;
        }
    }
    *c = BatchCounts{descs, ns, nl, long_bytes, bytes, n_ce, ce_bytes};
    return TB_OK;
}

int batch_grid(const BatchCounts &c, int full_grid)
{
    const uint64_t warps = kBatchThreads / 32;
    const uint64_t for_short = (c.n_short + warps - 1) / warps;
    const uint64_t for_long = (c.long_bytes + kChunkBytes - 1) / kChunkBytes;
    uint64_t want = std::max<uint64_t>(1, std::max(for_short, for_long));
    if (c.n_long == 0 && want > (uint64_t)full_grid) {
        // Short copies only, more than one wave's warps: whole waves, the
        // warps taking the copies past the first one each (a partial wave
        // would run after the first one has finished).
        want = (uint64_t)full_grid * std::min<uint64_t>(kShortWaves, want / (uint64_t)full_grid);
    }
    const uint64_t waves = c.n_long ? kBatchWaves : kShortWaves;
    return (int)std::min<uint64_t>(std::min<uint64_t>((uint64_t)full_grid * waves, kMaxChunks), want);
}

int short_shape_for(const BatchCounts &c, int forced, uint64_t wide_warps)
{
    if (c.n_long > 0)
        return 0;
    if (forced >= 1 && forced <= kShortShapes)
        return forced;
    return c.n_short <= wide_warps ? 2 : 1;
}

void finish_batch(const BatchCounts &c, const WorkItem *longs, int grid, void *buf, BatchPlan *out)
{
    char *base = static_cast<char *>(buf);
    std::memset(base, 0, kBatchHeader);  // the claim counter starts at 0
    WorkItem *lg = reinterpret_cast<WorkItem *>(base + kBatchHeader) + c.n_short;
    uint64_t *prefix = reinterpret_cast<uint64_t *>(lg + c.n_long);
    uint32_t *chunk_desc = reinterpret_cast<uint32_t *>(prefix + c.n_long + 1);

    // Chunks: about kChunkBytes each, a whole number per CTA.
    const uint64_t G = (uint64_t)grid;
    uint64_t m = (c.long_bytes + G * kChunkBytes / 2) / (G * kChunkBytes);
    m = std::max<uint64_t>(1, std::min<uint64_t>(m, kMaxChunks / G));
    const uint64_t chunks = c.n_long ? G * m : 0;

    uint64_t pos = 0;
    for (uint64_t k = 0; k < c.n_long; ++k) {
        lg[k] = longs[k];
        prefix[k] = pos;
        pos += longs[k].len;
    }
    prefix[c.n_long] = pos;
    // Chunk -> first long copy it touches.  Chunk starts are chunk_start()
    // walked incrementally: raw_k = q k + floor(r k / chunks).
    uint32_t dcur = 0;
    const uint64_t q = chunks ? pos / chunks : 0, r = chunks ? pos % chunks : 0;
    uint64_t raw = 0, rem = 0;
    for (uint64_t k = 0; k < chunks; ++k) {
        const uint64_t s0 = raw & ~(uint64_t)63;
        while (dcur + 1 < c.n_long && prefix[dcur + 1] <= s0)
            ++dcur;
        chunk_desc[k] = dcur;
        raw += q;
        rem += r;
        if (rem >= chunks) {
            rem -= chunks;
            raw += 1;
        }
    }
    chunk_desc[chunks] = (uint32_t)c.n_long;

    out->n_short = (uint32_t)c.n_short;
    out->n_long = (uint32_t)c.n_long;
    out->grid = (uint32_t)grid;
    out->chunks = (uint32_t)chunks;
    out->long_bytes = pos;
    out->prefix_offset = (size_t)((const char *)prefix - base);
    out->chunk_offset = (size_t)((const char *)chunk_desc - base);
    out->upload_bytes = out->chunk_offset + ((size_t)chunks + 1) * sizeof(uint32_t);
}

bool find_overlap(const tb_copy_desc *desc, size_t n, size_t *first, size_t *second)
{
    // Every non-empty range, sorted by start; one sweep keeps the furthest
    // end among the destinations and among the sources seen so far.  A
    // range that starts before such an end overlaps that range.
    struct Range {
        uint64_t begin, end;
        size_t index;
        bool dst;
    };
    std::vector<Range> r;
    r.reserve(2 * n);
    for (size_t i = 0; i < n; ++i) {
        if (desc[i].len == 0)
            continue;
        r.push_back(Range{desc[i].dst, desc[i].dst + desc[i].len, i, true});
        r.push_back(Range{desc[i].src, desc[i].src + desc[i].len, i, false});
    }
    std::sort(r.begin(), r.end(), [](const Range &a, const Range &b) { return a.begin < b.begin; });
    uint64_t dst_end = 0, src_end = 0;
    size_t dst_at = 0, src_at = 0;
    bool any_dst = false, any_src = false;
    for (const Range &x : r) {
        if (any_dst && x.begin < dst_end) {  // overlaps an earlier destination
            *first = dst_at;
            *second = x.index;
            return true;
        }
        if (x.dst && any_src && x.begin < src_end) {  // a destination over an earlier source
            *first = src_at;
            *second = x.index;
            return true;
        }
        if (x.dst) {
            if (!any_dst || x.end > dst_end) {
                dst_end = x.end;
                dst_at = x.index;
            }
            any_dst = true;
        } else {
            if (!any_src || x.end > src_end) {
                src_end = x.end;
                src_at = x.index;
            }
            any_src = true;
        }
    }
    return false;
}

uint32_t batch_claim_items(const BatchPlan &plan)
{
    const uint64_t warps = kBatchThreads / 32;
    const uint64_t starters = (uint64_t)plan.grid * (plan.chunks ? warps - 1 : warps);
    return (uint64_t)plan.n_short <= starters ? 1u : 2u;
}

bool batch_direct(const BatchPlan &plan)
{
    const uint64_t warps = kBatchThreads / 32;
    const uint64_t fixed = (uint64_t)plan.grid * warps * batch_claim_items(plan);
    return plan.chunks == 0 && plan.n_short > 0 && plan.upload_bytes <= kDirectMaxBytes &&
           (uint64_t)plan.n_short <= fixed;
}

}  // namespace tb

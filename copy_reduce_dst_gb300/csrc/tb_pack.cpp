// Host-side packing of the batched copy: turns a (src, dst, len) descriptor
// array into the work list one k_batch launch reads.
//
// Layout of a packed launch (one device buffer):
//   WorkItem shorts[n_short]     copies of at most small_max bytes, longest
//                                first (one warp each)
//   WorkItem longs[n_long]       the longer copies, in descriptor order
//   uint64_t prefix[n_long + 1]  offset of each long copy in the stream of
//                                all long-copy bytes; prefix[n_long] = total
//   uint32_t chunk_desc[C + 1]   the long copy holding chunk c's first byte
// The long-copy stream is cut into C = grid * m chunks of equal size (cuts
// on 64-byte stream offsets); CTA b copies chunks b, b + grid, ... so every
// CTA gets exactly m chunks and the grid sweeps the stream front to back.

#include <algorithm>
#include <cstring>

#include "tb_internal.h"

namespace tb {

unsigned bucket_shift(uint64_t small_max)
{
    unsigned shift = 6;
    while ((small_max >> shift) > 4096)
        ++shift;
    return shift;
}

size_t bucket_count(uint64_t small_max)
{
    return (size_t)(small_max >> bucket_shift(small_max)) + 1;
}

size_t batch_buffer_bytes(uint64_t descs)
{
    return (size_t)descs * (sizeof(WorkItem) + sizeof(uint64_t)) + sizeof(uint64_t) +
           ((size_t)kMaxChunks + 1) * sizeof(uint32_t);
}

int count_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, BatchCounts *c,
                size_t *bad, uint32_t *bucket)
{
    *c = BatchCounts{};
    const unsigned shift = bucket_shift(small_max);
    const size_t nb = bucket_count(small_max);
    if (bucket)
        std::fill(bucket, bucket + nb, 0u);
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len == 0)
            continue;
        if (d.src == 0 || d.dst == 0 || d.src + d.len < d.src || d.dst + d.len < d.dst) {
            if (bad)
                *bad = i;
            return TB_EINVAL;
        }
        ++c->descs;
        c->bytes += d.len;
        if (d.len <= small_max) {
            ++c->n_short;
            if (bucket)
                ++bucket[nb - 1 - (size_t)(d.len >> shift)];
        } else {
            ++c->n_long;
            c->long_bytes += d.len;
        }
    }
    return TB_OK;
}

int batch_grid(const BatchCounts &c, int full_grid)
{
    const uint64_t warps = kBatchThreads / 32;
    const uint64_t for_short = (c.n_short + warps - 1) / warps;
    const uint64_t for_long = (c.long_bytes + kChunkBytes - 1) / kChunkBytes;
    const uint64_t want = std::max<uint64_t>(1, std::max(for_short, for_long));
    return (int)std::min<uint64_t>(std::min<uint64_t>((uint64_t)full_grid, kMaxChunks), want);
}

void pack_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, const BatchCounts &c,
                int grid, void *buf, uint32_t *bucket, BatchPlan *out)
{
    const unsigned shift = bucket_shift(small_max);
    const size_t nb = bucket_count(small_max);

    // Chunks: about kChunkBytes each, a whole number per CTA.
    uint64_t m = (c.long_bytes + (uint64_t)grid * kChunkBytes / 2) / ((uint64_t)grid * kChunkBytes);
    m = std::max<uint64_t>(1, std::min<uint64_t>(m, kMaxChunks / (uint64_t)grid));
    const uint64_t chunks = c.n_long ? (uint64_t)grid * m : 0;

    WorkItem *shorts = static_cast<WorkItem *>(buf);
    WorkItem *longs = shorts + c.n_short;
    uint64_t *prefix = reinterpret_cast<uint64_t *>(longs + c.n_long);
    uint32_t *chunk_desc = reinterpret_cast<uint32_t *>(prefix + c.n_long + 1);

    // Bucket counts (from count_batch) -> starts; short copies longest first.
    uint32_t run = 0;
    for (size_t k = 0; k < nb; ++k) {
        const uint32_t cnt = bucket[k];
        bucket[k] = run;
        run += cnt;
    }
    // Place every copy.
    uint32_t nl = 0;
    uint64_t pos = 0;
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len == 0)
            continue;
        if (d.len <= small_max) {
            uint32_t &p = bucket[nb - 1 - (size_t)(d.len >> shift)];
            shorts[p++] = WorkItem{d.src, d.dst, d.len};
        } else {
            prefix[nl] = pos;
            longs[nl++] = WorkItem{d.src, d.dst, d.len};
            pos += d.len;
        }
    }
    prefix[nl] = pos;
    // Chunk -> first long copy it touches.
    uint32_t dcur = 0;
    for (uint64_t k = 0; k < chunks; ++k) {
        const uint64_t s0 = chunk_start(pos, chunks, k);
        while (dcur + 1 < nl && prefix[dcur + 1] <= s0)
            ++dcur;
        chunk_desc[k] = dcur;
    }
    chunk_desc[chunks] = nl;

    out->n_short = (uint32_t)c.n_short;
    out->n_long = nl;
    out->grid = (uint32_t)grid;
    out->chunks = (uint32_t)chunks;
    out->long_bytes = pos;
    out->prefix_offset = (size_t)((const char *)prefix - (const char *)buf);
    out->chunk_offset = (size_t)((const char *)chunk_desc - (const char *)buf);
    out->upload_bytes = out->chunk_offset + ((size_t)chunks + 1) * sizeof(uint32_t);
}

}  // namespace tb

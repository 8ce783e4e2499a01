// Host-side packing of the batched copy: turns a (src, dst, len) descriptor
// array into the work list one k_batch launch reads.
//
// Layout of a packed launch (one device buffer):
//   WorkItem items[n_long_items + n_short]   pieces of long copies, then
//                                            short copies longest first
//   uint32_t cta_first[grid + 1]             CTA b copies long pieces
//                                            [cta_first[b], cta_first[b+1])
// The bytes of all long copies (len > small_max) form one stream, cut into
// grid shares of equal size (cuts on 64-byte stream offsets), so every CTA
// leaves the long-copy phase at the same time; a cut inside a copy splits it
// into two pieces.  Short copies are then dealt to warps by the kernel.

#include <algorithm>
#include <cstring>

#include "tb_internal.h"

namespace tb {

size_t bucket_count(uint64_t small_max)
{
    return (size_t)(small_max >> bucket_shift(small_max)) + 1;
}

unsigned bucket_shift(uint64_t small_max)
{
    unsigned shift = 6;
    while ((small_max >> shift) > 4096)
        ++shift;
    return shift;
}

size_t batch_buffer_bytes(uint64_t items, int grid)
{
    return (size_t)(items + (uint64_t)grid) * sizeof(WorkItem) + ((size_t)grid + 1) * sizeof(uint32_t);
}

int count_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, BatchCounts *c,
                size_t *bad)
{
    *c = BatchCounts{};
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
    const uint64_t for_long = (c.long_bytes + 65535) / 65536;  // at least 64 KiB per CTA
    const uint64_t want = std::max<uint64_t>(1, std::max(for_short, for_long));
    return (int)std::min<uint64_t>((uint64_t)full_grid, want);
}

// Start of CTA b's share of a T-byte stream over G CTAs, on a 64-byte offset.
static uint64_t share_start(uint64_t T, uint32_t G, uint32_t b)
{
    if (b >= G)
        return T;
    const uint64_t raw = (T / G) * b + ((T % G) * b) / G;
    return raw & ~(uint64_t)63;
}

void pack_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, const BatchCounts &c,
                int grid, void *buf, uint32_t *bucket, BatchPlan *out)
{
    const unsigned shift = bucket_shift(small_max);
    const size_t nb = bucket_count(small_max);
    const uint32_t G = (uint32_t)grid;

    // Long copies: walk the stream, cutting at every CTA share boundary.
    WorkItem *items = static_cast<WorkItem *>(buf);
    uint32_t n_long_items = 0;
    {
        // The table goes after the items; its position needs the item count,
        // which is at most n_long + G - 1, so fill it in a local pass first.
        uint64_t pos = 0;
        uint32_t b = 0;
        uint64_t next = share_start(c.long_bytes, G, 1);
        std::fill(bucket, bucket + nb, 0u);
        for (size_t i = 0; i < n; ++i) {
            const tb_copy_desc &d = desc[i];
            if (d.len == 0)
                continue;
            if (d.len <= small_max) {
                ++bucket[nb - 1 - (size_t)(d.len >> shift)];
                continue;
            }
            uint64_t off = 0;
            while (off < d.len) {
                while (next <= pos) {  // CTA b's share is complete
                    ++b;
                    next = share_start(c.long_bytes, G, b + 1);
                }
                const uint64_t take = std::min(d.len - off, next - pos);
                items[n_long_items++] = WorkItem{d.src + off, d.dst + off, take};
                off += take;
                pos += take;
            }
        }
    }
    // Per-CTA table: second walk over the pieces (cheap: at most n_long + G).
    uint32_t *first = reinterpret_cast<uint32_t *>(items + n_long_items + c.n_short);
    {
        uint64_t pos = 0;
        uint32_t b = 0;
        first[0] = 0;
        uint64_t next = share_start(c.long_bytes, G, 1);
        for (uint32_t k = 0; k < n_long_items; ++k) {
            while (next <= pos && b < G) {
                ++b;
                first[b] = k;
                next = share_start(c.long_bytes, G, b + 1);
            }
            pos += items[k].len;
        }
        while (b < G)
            first[++b] = n_long_items;
    }

    // Short copies, longest first (counting sort on 2^shift-byte buckets).
    uint32_t run = 0;
    for (size_t k = 0; k < nb; ++k) {
        const uint32_t cnt = bucket[k];
        bucket[k] = run;
        run += cnt;
    }
    WorkItem *shorts = items + n_long_items;
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len == 0 || d.len > small_max)
            continue;
        uint32_t &p = bucket[nb - 1 - (size_t)(d.len >> shift)];
        shorts[p++] = WorkItem{d.src, d.dst, d.len};
    }

    out->n_long_items = n_long_items;
    out->n_short = (uint32_t)c.n_short;
    out->grid = G;
    out->table_offset = (size_t)(n_long_items + c.n_short) * sizeof(WorkItem);
    out->upload_bytes = out->table_offset + ((size_t)G + 1) * sizeof(uint32_t);
}

}  // namespace tb

// Test harness: exposes the batched copy's host packer to the CPU tests.
#include <vector>

#include "tb_internal.h"

extern "C" int harness_pack(const tb_copy_desc *desc, size_t n, uint64_t small_max, uint64_t ce_min,
                            int full_grid, void *buf, uint64_t *out)
{
    tb::BatchCounts c, c2;
    size_t bad = 0;
    if (tb::count_batch(desc, n, small_max, &c2, &bad, ce_min) != TB_OK)
        return -1;
    std::vector<tb::WorkItem> longs(n + 1);
    if (tb::gather_batch(desc, n, small_max, ce_min, buf, longs.data(), &c, &bad) != TB_OK)
        return -2;
    if (c.descs != c2.descs || c.n_short != c2.n_short || c.n_long != c2.n_long ||
        c.long_bytes != c2.long_bytes || c.n_ce != c2.n_ce)
        return -3;
    const int grid = tb::batch_grid(c, full_grid);
    tb::BatchPlan plan;
    tb::finish_batch(c, longs.data(), grid, buf, &plan);
    out[0] = plan.n_short;
    out[1] = plan.n_long;
    out[2] = plan.grid;
    out[3] = plan.chunks;
    out[4] = plan.long_bytes;
    out[5] = plan.prefix_offset;
    out[6] = plan.chunk_offset;
    out[7] = plan.upload_bytes;
    out[8] = tb::batch_buffer_bytes(c.descs);
    out[9] = c.n_ce;
    out[10] = tb::batch_claim_items(plan);
    out[11] = tb::batch_direct(plan) ? 1 : 0;
    return 0;
}

extern "C" int harness_bad(const tb_copy_desc *desc, size_t n, uint64_t *bad_out)
{
    tb::BatchCounts c;
    size_t bad = 0;
    std::vector<tb::WorkItem> longs(n + 1);
    std::vector<char> buf(tb::batch_buffer_bytes(n));
    const int rc = tb::gather_batch(desc, n, 16384, 0, buf.data(), longs.data(), &c, &bad);
    *bad_out = bad;
    return rc;
}

extern "C" int harness_overlap(const tb_copy_desc *desc, size_t n, uint64_t *pair)
{
    size_t a = 0, b = 0;
    const bool found = tb::find_overlap(desc, n, &a, &b);
    pair[0] = a;
    pair[1] = b;
    return found ? 1 : 0;
}

extern "C" int harness_short_shape(uint64_t n_short, uint64_t n_long, int forced,
                                   uint64_t wide_warps)
{
    tb::BatchCounts c{};
    c.n_short = n_short;
    c.n_long = n_long;
    c.descs = n_short + n_long;
    return tb::short_shape_for(c, forced, wide_warps);
}

extern "C" uint64_t harness_chunk_start(uint64_t total, uint64_t chunks, uint64_t c)
{
    return tb::chunk_start(total, chunks, c);
}

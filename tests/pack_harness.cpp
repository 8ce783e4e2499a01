// Test harness: exposes the batched copy's host packer to the CPU tests.
#include "tb_internal.h"

extern "C" int harness_pack(const tb_copy_desc *desc, size_t n, uint64_t small_max, int full_grid,
                            void *buf, uint32_t *bucket, uint64_t *out)
{
    tb::BatchCounts c;
    size_t bad = 0;
    if (tb::count_batch(desc, n, small_max, &c, &bad, bucket) != TB_OK)
        return -1;
    const int grid = tb::batch_grid(c, full_grid);
    tb::BatchPlan plan;
    tb::pack_batch(desc, n, small_max, c, grid, buf, bucket, &plan);
    out[0] = plan.n_short;
    out[1] = plan.n_long;
    out[2] = plan.grid;
    out[3] = plan.chunks;
    out[4] = plan.long_bytes;
    out[5] = plan.prefix_offset;
    out[6] = plan.chunk_offset;
    out[7] = plan.upload_bytes;
    out[8] = tb::batch_buffer_bytes(c.descs);
    return 0;
}

extern "C" uint64_t harness_chunk_start(uint64_t total, uint64_t chunks, uint64_t c)
{
    return tb::chunk_start(total, chunks, c);
}

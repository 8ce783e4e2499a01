// Internal interface between the host side of libtb (tb_host.cpp,
// tb_pack.cpp, tb_static.cu) and its kernels (tb_reduce.cu, tb_batch.cu,
// tb_fill.cu).  Not installed; the public ABI is include/tb.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tb.h"

namespace tb {

// ---------------------------------------------------------------------------
// Reduce-copy (K1)
// ---------------------------------------------------------------------------

// One reduce-copy launch, fully resolved on the host.  The element range
// [0, n) splits into head (scalar, until dst reaches vector alignment), body
// (nvec vectors of vec_bytes) and tail (scalar).  The grid's CTAs are dealt to
// the num_subexec sub-executors as evenly as integers allow; each
// sub-executor owns a contiguous run of body vectors in proportion to its
// CTAs (equal runs when num_subexec divides the grid).
struct ReducePlan {
    const float *src[TB_MAX_SRCS];
    float *dst;
    uint64_t n;            // elements
    uint64_t head;         // scalar elements before the body
    uint64_t nvec;         // body vectors
    int n_src;
    int vec_bytes;         // 32, 16, or 4 (no common 16-byte alignment: scalar)
    int num_subexec;
    int grid;              // CTAs of the launch (>= num_subexec)
    int block_threads;
    int unroll;            // vectors per source a thread holds in flight
    int engine;            // 1 = vector loads, 2 = bulk copies through shared memory
    size_t smem_bytes;     // dynamic shared memory of the launch
    uint32_t memset_word;  // 0-source fill, the memset byte repeated
    uint32_t *status;      // nullable, device-visible: 1 if a bounded wait expired
    int pdl;               // 1 = launch with programmatic dependent launch
    int stages;            // bulk form: shared-memory pipeline stages
    int bulk_deep;         // bulk form: 1 = the deep pipeline's tile (CTAs alone on SMs)
    uint64_t wait_ns = 2000000000ull;  // bulk form: limit of each wait for a tile's loads
    // 1 = the launch may start reading its sources before the launch ahead
    // of it on the stream has finished: only for a launch that follows
    // another of the same transfer, which reads the same (unmodified)
    // sources and writes only dst.
    int early = 0;
};

// Picks engine, vector width, head/tail, sub-executor split, grid and unroll
// for one launch.  num_subexec, ctas_per_subexec, block_threads, vec_bytes,
// unroll and engine of 0 take the defaults.  Returns TB_OK, TB_EINVAL or
// TB_ENOTSUP (a forced vector width or engine the sources or the pointers'
// alignment do not allow).
int plan_reduce(ReducePlan *p, const void *const *srcs, int n_src, void *dst, uint64_t num_bytes,
                int num_subexec, int ctas_per_subexec, int block_threads, int vec_bytes, int unroll,
                uint32_t memset_byte, int num_sms, int engine);

// Launches the plan on `stream` (asynchronous).
cudaError_t launch_reduce(const ReducePlan &p, cudaStream_t stream);
// Bulk form: bytes per source of one tile of the plan's kernel; 0 otherwise.
uint32_t plan_tile_bytes(const ReducePlan &p);

// Default CTAs resident per SM for the reduce kernel of this plan shape.
int reduce_ctas_per_sm(int n_src, int vec_bytes, int block_threads, int unroll);

// ---------------------------------------------------------------------------
// Source patterns
// ---------------------------------------------------------------------------
cudaError_t launch_fill_source(float *dst, uint64_t n, const tb_pattern &pat, int buffer_idx,
                               int num_sms, cudaStream_t stream);

// Device-side compare of n bytes: *first (device memory) becomes the
// smallest differing byte index, or stays UINT64_MAX.
cudaError_t launch_compare(const void *a, const void *b, uint64_t n, unsigned long long *first,
                           int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Gate kernel: waits, with a %globaltimer deadline, until *flag != 0.
// Writes *status = 1 when released, 2 when the deadline passed first.
// ---------------------------------------------------------------------------
cudaError_t launch_gate(const volatile uint32_t *flag, uint32_t *status, uint64_t timeout_ns,
                        cudaStream_t stream);

// ---------------------------------------------------------------------------
// Batched copy (K2)
// ---------------------------------------------------------------------------

// One packed work item: copy len bytes from src to dst.
struct WorkItem {
    uint64_t src;
    uint64_t dst;
    uint64_t len;
};
static_assert(sizeof(WorkItem) == 24, "WorkItem is packed as three 64-bit words");

constexpr int kBatchThreads = 256;
constexpr uint64_t kChunkBytes = 65536;  // target size of a long-copy chunk
constexpr uint32_t kMaxChunks = 16384;   // chunks of one launch at most
// Waves of resident CTAs a batch launch may span.  Short-lived CTAs over
// several waves let the CTA scheduler balance the SMs' finishing times
// (47,540 batch: 141 us at 8 waves against 145 at one; one 2 GiB copy
// 6.86 against 6.45 TB/s).
constexpr uint64_t kBatchWaves = 8;
// Waves of a launch of short copies only: fewer CTAs leave more of the
// copies to the claim counter, which balances them (47,520 short copies:
// 55.4 us at 4 waves, 61.0 at 8, 57.3 at 2, 58.5 at 1).
constexpr uint64_t kShortWaves = 4;
constexpr size_t kBatchHeader = 16;      // claim counter of the short copies

// Descriptor counts of a batch (descriptors with len == 0 are skipped).
struct BatchCounts {
    uint64_t descs;       // len > 0
    uint64_t n_short;     // len <= small_max: one warp each
    uint64_t n_long;      // len > small_max: CTA phase
    uint64_t long_bytes;  // sum of the long lengths
    uint64_t bytes;       // sum of all lengths
    uint64_t n_ce;        // len >= ce_min: left to the copy engines
    uint64_t ce_bytes;
};

// One packed launch (see tb_pack.cpp for the buffer layout).
struct BatchPlan {
    uint32_t n_short;       // short copies
    uint32_t n_long;        // long copies
    uint32_t grid;          // CTAs of the launch
    uint32_t chunks;        // long-stream chunks (a multiple of grid)
    uint64_t long_bytes;    // bytes of the long-copy stream
    size_t prefix_offset;   // byte offsets of prefix[] and chunk_desc[]
    size_t chunk_offset;
    size_t upload_bytes;    // bytes of the packed buffer
    int shape = 0;          // kernel: 0 = k_batch (long copies), 1.. = a k_short shape
};

// Shapes of the kernel of a launch of short copies only (k_short), numbered
// 1..kShortShapes: 1 = four 2 KiB slots per warp, 3 CTAs per SM (deeper
// rings, for batches of more copies than one round of warps); 2 = two 2 KiB
// slots, 5 CTAs per SM (more warps, each copy in the first round).
constexpr int kShortShapes = 2;

// Start of chunk c of `chunks` equal chunks of a `total`-byte stream, on a
// 64-byte offset; chunk `chunks` starts at total.
__host__ __device__ inline uint64_t chunk_start(uint64_t total, uint64_t chunks, uint64_t c)
{
    if (c >= chunks)
        return total;
    const uint64_t raw = (total / chunks) * c + ((total % chunks) * c) / chunks;
    return raw & ~(uint64_t)63;
}

// Bytes a packed launch of at most `descs` non-empty descriptors needs.
size_t batch_buffer_bytes(uint64_t descs);
// Checks and counts descriptors; TB_EINVAL (index in *bad) for a null or
// wrapping range.  Descriptors with len >= ce_min (when ce_min > 0) are
// counted apart: the caller sends them to the copy engines.
int count_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, BatchCounts *c,
                size_t *bad, uint64_t ce_min = 0);
// One pass: checks and counts like count_batch, appends the short copies to
// buf (after the header) and the long ones to `longs` (room for n).
int gather_batch(const tb_copy_desc *desc, size_t n, uint64_t small_max, uint64_t ce_min,
                 void *buf, WorkItem *longs, BatchCounts *c, size_t *bad);
// CTAs for a batch: kBatchWaves full waves at most, fewer for small batches;
// full_grid = the CTAs of one wave of the launch's kernel shape.
int batch_grid(const BatchCounts &c, int full_grid);
// Kernel shape of a launch: 0 (k_batch) when it has long copies, else
// `forced` when it names a k_short shape, else shape 2 when every short copy
// gets a warp of shape 2's first wave (wide_warps of them), else shape 1.
int short_shape_for(const BatchCounts &c, int forced, uint64_t wide_warps);
// Completes a buffer gather_batch filled: header, long copies, prefix and
// chunk table; fills *out.
void finish_batch(const BatchCounts &c, const WorkItem *longs, int grid, void *buf, BatchPlan *out);
// Looks for two descriptors whose ranges make the batch's result depend on
// the order of the copies: two overlapping destinations, or a destination
// overlapping a source (its own included).  Sources may overlap one
// another.  Returns true with their indices (in either order).
bool find_overlap(const tb_copy_desc *desc, size_t n, size_t *first, size_t *second);
// Short copies each warp that starts on short copies takes by its index
// (no atomic; warp w of `starters` takes copies w, w + starters, ...)
// before it claims more, a few at a time, from the counter: 1 when those
// warps outnumber the short copies, else 2.
uint32_t batch_claim_items(const BatchPlan &plan);
// Work lists up to this size may be read by the kernel in place.
constexpr size_t kDirectMaxBytes = 256 * 1024;
// True when the launch can read its work list in place from pinned host
// memory instead of a device copy: short copies only, every one of them in
// the fixed first round (so the kernel never touches the claim counter),
// and a work list of at most kDirectMaxBytes.
bool batch_direct(const BatchPlan &plan);

// CTAs of `kernel` resident per SM at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device; raises the kernel's shared
// memory limit there first when it needs more than 48 KiB.  Cached per
// (device, kernel, threads, smem); 0 when a CUDA call fails.
int resident_ctas(const void *kernel, int threads, size_t smem);

// Completion signal of a batch launch (all fields null: none).  Every CTA
// adds one to *count (device memory that only grows) once it has finished
// reading the work list; the CTA whose add returns base + grid - 1 (base:
// the count before the launch, which the host tracks) is the last, and
// writes seq to *word (the device address of a host-mapped word), so the
// host learns with one read of host memory that the launch no longer reads
// its work list.
struct BatchDone {
    uint32_t *count = nullptr;
    uint32_t *word = nullptr;
    uint32_t base = 0;
    uint32_t seq = 0;
};

// Launches k_batch over a packed buffer (device copy at `dev`).  status
// (nullable, device-visible) is set to 1 if a bounded wait inside the kernel
// expired; wait_ns limits each wait of its bulk pipeline for a block's load
// (0: one non-blocking probe).
// With pdl the launch may be scheduled before the kernel ahead of it on the
// stream has finished (programmatic dependent launch): it reads its work
// list early, and every access to the copies' bytes waits for that kernel.
cudaError_t launch_batch(const void *dev, const BatchPlan &plan, cudaStream_t stream,
                         uint32_t *status = nullptr, uint64_t wait_ns = 2000000000ull,
                         const BatchDone &done = BatchDone{}, bool pdl = false);

// CTAs resident per SM for kernel shape k (0 = k_batch, 1..kShortShapes =
// k_short); 0 for an unknown shape or when a CUDA call fails.
int batch_ctas_per_sm(int k);

}  // namespace tb

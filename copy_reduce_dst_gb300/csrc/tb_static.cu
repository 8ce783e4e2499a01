// tb_batch_copy_noalloc: the batched copy for callers that cannot allocate
// device memory.
//
// tb_batch_copy keeps its packed work items in descriptor slots that
// tb_create allocates with cudaMalloc.  Some callers cannot make that call:
// a serving engine that has handed all free HBM to its own allocator (a KV
// cache reserved up front) has nothing left for an extra cudaMalloc, and a
// latency-sensitive loop cannot afford cudaMalloc / cudaFree, which may
// synchronize the whole device and stall every other stream.  This entry
// point needs no context and allocates nothing: its work items live in a
// file-scope __device__ array of fixed size, which every GPU that loads the
// library holds until the process exits.
//
// Host code must not pass the array's name to a kernel - in host code that
// name is only a host-side stand-in, not a device address.  The device
// address comes from cudaGetSymbolAddress, taken once per device with that
// device current, on the first call on the device.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "tb_internal.h"

namespace {

using tb::WorkItem;

constexpr uint64_t kSmallMax = 16384;   // one warp per copy up to this size
constexpr uint64_t kChunk = 65536;      // longer copies: 64 KiB CTA chunks
constexpr unsigned kShift = 6;          // length buckets of 64 bytes
constexpr size_t kBuckets = (kSmallMax >> kShift) + 1;
constexpr int kMaxDevices = 64;

// The scratch: packed work items of the batch in flight.
static __device__ __align__(256) WorkItem g_scratch_items[TB_NOALLOC_MAX_ITEMS];

// Host-side packing area (static storage, no heap) and its lock.
WorkItem g_host_items[TB_NOALLOC_MAX_ITEMS];
uint32_t g_bucket[kBuckets];
std::mutex g_lock;

// Per-device set-up: the scratch array's device address and the grid size.
WorkItem *g_dev_items[kMaxDevices];
int g_dev_grid[kMaxDevices];

int setup_current_device(int *device)
{
    if (cudaGetDevice(device) != cudaSuccess || *device < 0 || *device >= kMaxDevices)
        return TB_ECUDA;
    if (g_dev_items[*device])
        return TB_OK;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch_items) != cudaSuccess || !ptr)
        return TB_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess)
        return TB_ECUDA;
    g_dev_grid[*device] = sms * tb::batch_ctas_per_sm();
    g_dev_items[*device] = static_cast<WorkItem *>(ptr);
    return TB_OK;
}

}  // namespace

extern "C" int tb_batch_copy_noalloc(const tb_copy_desc *desc, size_t n, tb_stream stream)
{
    if (n > 0 && !desc)
        return TB_EINVAL;
    std::lock_guard<std::mutex> hold(g_lock);
    int device = -1;
    int rc = setup_current_device(&device);
    if (rc != TB_OK)
        return rc;

    // Pass 1: check, count long-copy chunks and short copies per length bucket.
    std::fill(g_bucket, g_bucket + kBuckets, 0u);
    uint64_t n_cta = 0, n_warp = 0;
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len == 0)
            continue;
        if (d.src == 0 || d.dst == 0 || d.src + d.len < d.src || d.dst + d.len < d.dst)
            return TB_EINVAL;
        if (d.len <= kSmallMax) {
            ++g_bucket[kBuckets - 1 - (size_t)(d.len >> kShift)];
            ++n_warp;
        } else {
            n_cta += (d.len + kChunk - 1) / kChunk;
        }
    }
    const uint64_t total = n_cta + n_warp;
    if (total > TB_NOALLOC_MAX_ITEMS)
        return TB_ENOTSUP;
    if (total == 0)
        return TB_OK;

    // Pass 2: chunks first, then short copies longest first.
    uint32_t run = 0;
    for (size_t b = 0; b < kBuckets; ++b) {
        const uint32_t c = g_bucket[b];
        g_bucket[b] = run;
        run += c;
    }
    uint64_t ci = 0;
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len == 0)
            continue;
        if (d.len <= kSmallMax) {
            uint32_t &pos = g_bucket[kBuckets - 1 - (size_t)(d.len >> kShift)];
            g_host_items[n_cta + pos++] = WorkItem{d.src, d.dst, d.len};
        } else {
            for (uint64_t off = 0; off < d.len; off += kChunk)
                g_host_items[ci++] = WorkItem{d.src + off, d.dst + off, std::min(kChunk, d.len - off)};
        }
    }

    // The copy from pageable host memory returns once the bytes are staged,
    // so the host area is free again when this call returns.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WorkItem *items = g_dev_items[device];
    if (cudaMemcpyAsync(items, g_host_items, total * sizeof(WorkItem), cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return TB_ECUDA;
    const uint64_t warps_per_cta = tb::kBatchThreads / 32;
    const uint64_t want = std::max<uint64_t>(n_cta, (n_warp + warps_per_cta - 1) / warps_per_cta);
    const int grid = (int)std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)g_dev_grid[device], want));
    if (tb::launch_batch(items, (uint32_t)n_cta, (uint32_t)n_warp, grid, s) != cudaSuccess)
        return TB_ECUDA;
    return TB_OK;
}

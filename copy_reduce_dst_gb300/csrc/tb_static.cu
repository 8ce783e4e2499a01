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
//
// A bounded wait inside the kernel that runs out (the long copies' bulk
// pipeline) is recorded in a status word per device.  The words sit in one
// page of static host memory, page-locked and mapped into the devices'
// address space once (cudaHostRegister pins the library's own page; nothing
// is allocated), so every call can read them without synchronizing.

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "tb_internal.h"

namespace {

using tb::WorkItem;

constexpr uint64_t kSmallMax = 16384;  // one warp per copy up to this size
constexpr int kMaxDevices = 64;
constexpr int kMaxGrid = 2048;         // CTAs of one wave at most (a launch spans up to
                                       // kBatchWaves waves; nothing is sized by the grid)
// Bytes of one packed launch of TB_NOALLOC_MAX_ITEMS descriptors: the claim
// counter header, the work items and the long copies' stream prefix, the
// prefix's end, and the chunk table.
constexpr size_t kScratchBytes =
    tb::kBatchHeader + TB_NOALLOC_MAX_ITEMS * (sizeof(WorkItem) + sizeof(uint64_t)) +
    sizeof(uint64_t) + ((size_t)tb::kMaxChunks + 1) * sizeof(uint32_t);
constexpr size_t kScratchItems = (kScratchBytes + sizeof(WorkItem) - 1) / sizeof(WorkItem);
// The size include/tb.h states for this array.
static_assert(kScratchItems * sizeof(WorkItem) == 2162736, "update the documented size");

// The scratch: the packed launch of the batch in flight.
static __device__ __align__(256) WorkItem g_scratch_items[kScratchItems];

// Host-side packing area and long-copy list (static storage, no heap), and
// their lock.
WorkItem g_host_items[kScratchItems];
WorkItem g_longs[TB_NOALLOC_MAX_ITEMS];
std::mutex g_lock;

// Status words, one per device: 1 once a kernel's bounded wait ran out.
// One page, page-locked and mapped on first use.
alignas(4096) volatile uint32_t g_status[1024];
bool g_status_mapped = false;

// Per-device set-up: the scratch array's device address, the device's view
// of its status word, the limit of each bounded wait, and the CTAs of one
// resident wave of each batch-kernel shape.
WorkItem *g_dev_items[kMaxDevices];
uint32_t *g_dev_status[kMaxDevices];
uint64_t g_dev_wait_ns[kMaxDevices];
int g_dev_grid[kMaxDevices][tb::kShortShapes + 1];

int setup_current_device(int *device)
{
    if (cudaGetDevice(device) != cudaSuccess || *device < 0 || *device >= kMaxDevices)
        return TB_ECUDA;
    if (g_dev_items[*device])
        return TB_OK;
    if (!g_status_mapped) {
        if (cudaHostRegister(const_cast<uint32_t *>(g_status), sizeof(g_status),
                             cudaHostRegisterPortable | cudaHostRegisterMapped) != cudaSuccess)
            return TB_ECUDA;
        g_status_mapped = true;
    }
    void *status = nullptr;
    if (cudaHostGetDevicePointer(&status, const_cast<uint32_t *>(g_status), 0) != cudaSuccess ||
        !status)
        return TB_ECUDA;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch_items) != cudaSuccess || !ptr)
        return TB_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess)
        return TB_ECUDA;
    int grid[tb::kShortShapes + 1];
    for (int k = 0; k <= tb::kShortShapes; ++k) {
        const int per_sm = tb::batch_ctas_per_sm(k);
        if (per_sm < 1)
            return TB_ECUDA;
        grid[k] = std::min(kMaxGrid, sms * per_sm);
    }
    // The wait limit follows the contexts' default: environment variable
    // TB_KERNEL_WAIT_NS (parsed like the contexts' options), else 2 s, read
    // once here.  No other variable is read.
    tb_options o;
    tb_options_default(&o);
    if (const char *v = getenv("TB_KERNEL_WAIT_NS"))
        if (tb_parse_bytes(v, &o.kernel_wait_ns) != TB_OK)
            return TB_EINVAL;
    g_dev_wait_ns[*device] = o.kernel_wait_ns;
    for (int k = 0; k <= tb::kShortShapes; ++k)
        g_dev_grid[*device][k] = grid[k];
    g_dev_status[*device] = static_cast<uint32_t *>(status) + *device;
    g_status[*device] = 0u;
    g_dev_items[*device] = static_cast<WorkItem *>(ptr);
    return TB_OK;
}

}  // namespace

extern "C" int tb_batch_copy_noalloc(const tb_copy_desc *desc, size_t n, tb_stream stream)
{
    if (n > 0 && !desc)
        return TB_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The work list is copied from a host array that the next call rewrites,
    // so a copy recorded into a graph would replay another call's list.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capturing) != cudaSuccess)
        return TB_ECUDA;
    if (capturing != cudaStreamCaptureStatusNone)
        return TB_ENOTSUP;
    std::lock_guard<std::mutex> hold(g_lock);
    tb::BatchCounts c;
    if (tb::count_batch(desc, n, kSmallMax, &c, nullptr) != TB_OK)
        return TB_EINVAL;
    if (c.descs > TB_NOALLOC_MAX_ITEMS)
        return TB_ENOTSUP;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return TB_ECUDA;
    if (!g_dev_items[device]) {
        if (c.descs == 0)
            return TB_OK;  // nothing to copy and nothing launched on this device yet
        const int rc = setup_current_device(&device);
        if (rc != TB_OK)
            return rc;
    }
    // A kernel of an earlier call whose bounded wait ran out stopped before
    // copying everything: report it once, launch nothing.
    if (g_status[device] != 0u) {
        g_status[device] = 0u;
        return TB_ETIMEOUT;
    }
    if (c.descs == 0)
        return TB_OK;

    // Packing writes the whole launch, including a zero for the work
    // counter the kernel claims short copies from.
    tb::gather_batch(desc, n, kSmallMax, 0, g_host_items, g_longs, &c, nullptr);
    tb::BatchPlan plan;
    const int shape =
        tb::short_shape_for(c, 0, (uint64_t)g_dev_grid[device][2] * (tb::kBatchThreads / 32));
    tb::finish_batch(c, g_longs, tb::batch_grid(c, g_dev_grid[device][shape]), g_host_items,
                     &plan);
    plan.shape = shape;
    // The copy from pageable host memory returns once the bytes are staged,
    // so the host area is free again when this call returns.
    WorkItem *items = g_dev_items[device];
    if (cudaMemcpyAsync(items, g_host_items, plan.upload_bytes, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return TB_ECUDA;
    if (tb::launch_batch(items, plan, s, g_dev_status[device], g_dev_wait_ns[device],
                         tb::BatchDone{}, true) !=
        cudaSuccess)
        return TB_ECUDA;
    return TB_OK;
}

// Host runtime of libtb: options, contexts, the rotation allocator's plan and
// slice fill, TransferBench's timed iteration loop, the end-to-end transfer
// from host memory, the descriptor-slot ring of the batched copy, and
// validation.  Every GPU step is one of the kernels in tb_reduce.cu,
// tb_batch.cu and tb_fill.cu (or a CUDA copy where the API says so); this
// file only plans, enqueues and times them.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <functional>
#include <string>
#include <thread>
#include <vector>

#include "tb_internal.h"

using tb::WorkItem;

namespace {

constexpr uint64_t kMiB = 1ull << 20;
constexpr uint64_t kValidateChunk = 64 * kMiB;
// Most launches queued behind the gate kernel; beyond this the launch queue
// could fill while the gate holds the stream, so longer loops run ungated.
constexpr int kMaxGatedLaunches = 256;

struct Slot {
    void *dev = nullptr;       // device copy of one packed launch
    void *host = nullptr;      // pinned staging of it (mapped)
    void *host_dev = nullptr;  // device address of the staging
    cudaEvent_t done_event = nullptr;
    cudaEvent_t uploaded = nullptr;  // the work list is on the device (upload stream)
    bool pending = false;      // `done_event` recorded and maybe not reached yet
    cudaEvent_t t0 = nullptr;  // kernel timing (time_kernels only)
    cudaEvent_t t1 = nullptr;
    volatile uint32_t *status = nullptr;  // host-mapped: 1 if a kernel wait expired
    uint32_t *status_dev = nullptr;
    // Completion signal (tb::BatchDone): the launch's last CTA writes `seq`
    // into the host-mapped `done_word`, so wait_slot usually learns the slot
    // is free from one read of host memory instead of an event query.
    volatile uint32_t *done_word = nullptr;
    uint32_t *done_word_dev = nullptr;
    uint32_t *count_dev = nullptr;        // device counter of finished CTAs (only grows)
    uint32_t count = 0;                   // its value once every launch so far has finished
    uint32_t seq = 0;                     // of the slot's latest launch
};

// Chunk size of the staged tb_reduce_copy_host pipeline.
constexpr uint64_t kStageChunk = 32 * kMiB;

// Streams and events of the staged host <-> device pipeline, made on first use.
struct Pipeline {
    cudaStream_t h2d = nullptr, cmp = nullptr, d2h = nullptr;
    cudaEvent_t begin = nullptr, end = nullptr;
    std::vector<cudaEvent_t> in, out;  // per chunk
};

}  // namespace

struct tb_ctx {
    int device = 0;
    int num_sms = 0;
    tb_options opt{};
    cudaStream_t stream = nullptr;  // internal stream of the synchronous calls

    // Gate: host-mapped words the gate kernel polls and reports through.
    volatile uint32_t *gate_flag = nullptr;
    volatile uint32_t *gate_status = nullptr;
    uint32_t *gate_flag_dev = nullptr;
    uint32_t *gate_status_dev = nullptr;
    // Host-mapped word the bulk reduce kernel sets if a bounded wait expired.
    volatile uint32_t *reduce_status = nullptr;
    uint32_t *reduce_status_dev = nullptr;

    std::vector<cudaEvent_t> events;  // timing events of tb_run_transfer
    std::vector<float> iter_ms;

    std::vector<Slot> slots;
    void *slot_status = nullptr;      // host-mapped status and done words, two per slot
    uint32_t *slot_counts = nullptr;  // device counters of the completion signal, one per slot
    uint32_t next_slot = 0;
    // CTAs of one resident wave of each batch-kernel shape (0 = k_batch, a
    // launch with long copies; 1.. = the k_short shapes of short-only ones).
    int batch_grid[tb::kShortShapes + 1] = {};
    std::vector<WorkItem> longs;      // long copies of the run being packed
    tb_batch_stats last_batch{};
    std::vector<uint32_t> last_slots;  // slots the last batch launched on

    Pipeline pipe;                    // staged host <-> device transfers
    cudaStream_t up = nullptr;        // upload stream of batch work lists
    cudaStream_t ce = nullptr;        // copy-engine stream of routed batch copies
    cudaEvent_t ce_fork = nullptr, ce_join = nullptr;

    void *val_stage = nullptr;        // pinned validation staging
    void *direct_expected = nullptr;  // device copy of `expected` (validate_direct)
    uint64_t direct_bytes = 0;
    unsigned long long *first_diff = nullptr;  // device word of the device-side compare
    uint64_t prep_h2d = 0;
    std::string err;
};

namespace {

// Records a message on ctx and returns code.
int fail(tb_ctx *ctx, int code, const char *fmt, ...) __attribute__((format(printf, 3, 4)));
int fail(tb_ctx *ctx, int code, const char *fmt, ...)
{
    if (ctx) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        ctx->err = buf;
    }
    return code;
}

int cuda_fail(tb_ctx *ctx, cudaError_t e, const char *what)
{
    return fail(ctx, TB_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

#define TB_CUDA(ctx, call)                                   \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess)                               \
            return cuda_fail((ctx), e_, #call);              \
    } while (0)

// Makes ctx's device current for the scope and restores the caller's after.
class DeviceScope {
  public:
    explicit DeviceScope(int device)
    {
        if (cudaGetDevice(&prev_) == cudaSuccess && prev_ != device)
            ok_ = cudaSetDevice(device) == cudaSuccess;
        else
            prev_ = -1;
    }
    ~DeviceScope()
    {
        if (prev_ >= 0)
            cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

  private:
    int prev_ = -1;
    bool ok_ = true;
};

bool env_u64(const char *name, uint64_t *out, bool *bad)
{
    const char *v = getenv(name);
    if (!v)
        return false;
    if (tb_parse_bytes(v, out) != TB_OK)
        *bad = true;
    return true;
}

bool env_i32(const char *name, int32_t *out, bool *bad)
{
    uint64_t v = 0;
    if (!env_u64(name, &v, bad))
        return false;
    if (v > (uint64_t)INT32_MAX)
        *bad = true;
    else
        *out = (int32_t)v;
    return true;
}

bool env_u32(const char *name, uint32_t *out, bool *bad)
{
    uint64_t v = 0;
    if (!env_u64(name, &v, bad))
        return false;
    if (v > (uint64_t)UINT32_MAX)
        *bad = true;
    else
        *out = (uint32_t)v;
    return true;
}

int check_options(tb_ctx *ctx, const tb_options &o)
{
    if (o.byte_offset % 4 != 0)
        return fail(ctx, TB_EINVAL, "byte_offset must be a multiple of 4");
    if (o.warmup < 0)
        return fail(ctx, TB_EINVAL, "warmup must be >= 0");
    if (o.memset_byte > 255)
        return fail(ctx, TB_EINVAL, "memset_byte must be a byte");
    if (o.ctas_per_subexec < 0)
        return fail(ctx, TB_EINVAL, "ctas_per_subexec must be >= 0");
    if (o.block_threads < 0 || o.block_threads > 512 || o.block_threads % 32 != 0)
        return fail(ctx, TB_EINVAL, "block_threads must be a multiple of 32 up to 512");
    if (o.small_max_bytes == 0 || o.small_max_bytes > 16 * kMiB)
        return fail(ctx, TB_EINVAL, "small_max_bytes must be in [1, 16 MiB]");
    if (o.slot_items < 1024 || o.slot_items > (1u << 24))
        return fail(ctx, TB_EINVAL, "slot_items must be in [1024, 2^24]");
    if (o.num_slots < 1 || o.num_slots > 64)
        return fail(ctx, TB_EINVAL, "num_slots must be in [1, 64]");
    if (o.batch_min_copies < 0)
        return fail(ctx, TB_EINVAL, "batch_min_copies must be >= 0");
    if (o.batch_short_shape < 0 || o.batch_short_shape > tb::kShortShapes)
        return fail(ctx, TB_EINVAL, "batch_short_shape must be 0..%d", tb::kShortShapes);
    if (o.batch_max_ctas < 0)
        return fail(ctx, TB_EINVAL, "batch_max_ctas must be >= 0");
    if (o.early_reads != 0 && o.early_reads != 1)
        return fail(ctx, TB_EINVAL, "early_reads must be 0 or 1");
    if (o.wait_timeout_ns == 0)
        return fail(ctx, TB_EINVAL, "wait_timeout_ns must be > 0");
    if (o.vec_bytes != 0 && o.vec_bytes != 4 && o.vec_bytes != 16 && o.vec_bytes != 32)
        return fail(ctx, TB_EINVAL, "vec_bytes must be 0, 4, 16 or 32");
    if (o.unroll != 0 && o.unroll != 1 && o.unroll != 2 && o.unroll != 4)
        return fail(ctx, TB_EINVAL, "unroll must be 0, 1, 2 or 4");
    if (o.reduce_engine < 0 || o.reduce_engine > 2)
        return fail(ctx, TB_EINVAL, "reduce_engine must be 0, 1 or 2");
    return TB_OK;
}

// CUDA profiling tools (ncu, nsys) are injected through CUDA_INJECTION64_PATH
// and run each launch to completion before the launch call returns; a gate
// kernel would then hold the host inside its own launch until its deadline.
bool profiler_attached()
{
    const char *v = getenv("CUDA_INJECTION64_PATH");
    return v && *v;
}

uint64_t now_ns()
{
    return (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(
               std::chrono::steady_clock::now().time_since_epoch())
        .count();
}

// Waits for a slot's previous launch, bounded by the context's timeout.
int wait_slot(tb_ctx *ctx, Slot &s)
{
    if (!s.pending)
        return TB_OK;
    const uint64_t deadline = now_ns() + ctx->opt.wait_timeout_ns;
    // The kernel's completion word first (one read of host memory), the
    // slot's event as the fallback: the launch may still be running, or
    // may not have written the word (a kernel without the signal).
    while (*s.done_word != s.seq) {
        cudaError_t e = cudaEventQuery(s.done_event);
        if (e == cudaSuccess)
            break;
        if (e != cudaErrorNotReady)
            return cuda_fail(ctx, e, "cudaEventQuery(slot)");
        if (now_ns() > deadline)
            return fail(ctx, TB_ETIMEOUT, "no descriptor slot came free within %llu ns",
                        (unsigned long long)ctx->opt.wait_timeout_ns);
        std::this_thread::yield();
    }
    s.pending = false;
    if (s.status && *s.status != 0u) {
        *s.status = 0u;
        return fail(ctx, TB_ETIMEOUT,
                    "an earlier batch on this descriptor slot stopped early: a bounded wait "
                    "inside the kernel expired");
    }
    return TB_OK;
}

int plan_for(tb_ctx *ctx, tb::ReducePlan *p, const void *const *srcs, int n_src, void *dst,
             uint64_t num_bytes, int num_subexec)
{
    const tb_options &o = ctx->opt;
    int rc = tb::plan_reduce(p, srcs, n_src, dst, num_bytes, num_subexec, o.ctas_per_subexec,
                             o.block_threads, o.vec_bytes, o.unroll, o.memset_byte, ctx->num_sms,
                             o.reduce_engine);
    p->status = ctx->reduce_status_dev;
    p->pdl = o.use_pdl ? 1 : 0;
    p->wait_ns = o.kernel_wait_ns;
    if (rc == TB_EINVAL)
        return fail(ctx, rc,
                    "reduce-copy arguments rejected (nSrc in [0,%d], numBytes %% 4 == 0, "
                    "4-byte aligned non-null pointers, dst not overlapping a source, "
                    "numSubExec >= 0)",
                    TB_MAX_SRCS);
    if (rc != TB_OK)
        return fail(ctx, rc,
                    "vec_bytes=%d / reduce_engine=%d not possible for %d sources at these "
                    "pointers' alignment",
                    o.vec_bytes, o.reduce_engine, n_src);
    return TB_OK;
}

// Device address of a page-locked host buffer mapped into the device's
// address space, or nullptr for any other memory.
void *mapped_host_pointer(const void *p)
{
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer)
        return nullptr;
    return attr.devicePointer;
}

int ensure_pipeline(tb_ctx *ctx)
{
    Pipeline &pl = ctx->pipe;
    if (pl.h2d)
        return TB_OK;
    for (cudaStream_t *s : {&pl.h2d, &pl.cmp, &pl.d2h})
        TB_CUDA(ctx, cudaStreamCreateWithFlags(s, cudaStreamNonBlocking));
    TB_CUDA(ctx, cudaEventCreateWithFlags(&pl.begin, cudaEventDisableTiming));
    TB_CUDA(ctx, cudaEventCreateWithFlags(&pl.end, cudaEventDisableTiming));
    return TB_OK;
}

// Grows the per-chunk events of the staged pipeline to n.
int pipeline_events(tb_ctx *ctx, uint64_t n)
{
    Pipeline &pl = ctx->pipe;
    while (pl.in.size() < n) {
        cudaEvent_t a = nullptr, b = nullptr;
        TB_CUDA(ctx, cudaEventCreateWithFlags(&a, cudaEventDisableTiming));
        pl.in.push_back(a);
        TB_CUDA(ctx, cudaEventCreateWithFlags(&b, cudaEventDisableTiming));
        pl.out.push_back(b);
    }
    return TB_OK;
}

// Captures the iteration loop of tb_run_transfer (warm-up launches, an
// external event record, the timed launches, a second external event
// record) on ctx->stream, launches the graph and waits for it.  Only the
// span of the timed launches is recorded: an event node between every two
// launches costs more GPU time than the graph saves.  set_iteration(it)
// points the plan's sources at the slice iteration `it` reads.
int run_graphed(tb_ctx *ctx, int iters, const std::function<void(int64_t)> &set_iteration,
                const std::function<cudaError_t(cudaStream_t)> &issue)
{
    cudaStream_t st = ctx->stream;
    TB_CUDA(ctx, cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    cudaError_t err = cudaSuccess;
    for (int64_t it = -(int64_t)ctx->opt.warmup; it < iters && err == cudaSuccess; ++it) {
        set_iteration(it);
        if (it == 0)
            err = cudaEventRecordWithFlags(ctx->events[0], st, cudaEventRecordExternal);
        if (err == cudaSuccess)
            err = issue(st);
        if (err == cudaSuccess && it == iters - 1)
            err = cudaEventRecordWithFlags(ctx->events[iters], st, cudaEventRecordExternal);
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t end = cudaStreamEndCapture(st, &graph);
    if (err != cudaSuccess || end != cudaSuccess) {
        if (graph)
            cudaGraphDestroy(graph);
        cudaGetLastError();
        return cuda_fail(ctx, err != cudaSuccess ? err : end, "capturing the iteration graph");
    }
    cudaGraphExec_t exec = nullptr;
    err = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (err != cudaSuccess)
        return cuda_fail(ctx, err, "cudaGraphInstantiate");
    err = cudaGraphLaunch(exec, st);
    if (err == cudaSuccess)
        err = cudaStreamSynchronize(st);
    cudaGraphExecDestroy(exec);
    if (err != cudaSuccess)
        return cuda_fail(ctx, err, "iteration graph");
    return TB_OK;
}

double median_of(std::vector<float> v)
{
    if (v.empty())
        return 0.0;
    std::sort(v.begin(), v.end());
    const size_t m = v.size() / 2;
    return v.size() % 2 ? v[m] : 0.5 * ((double)v[m - 1] + (double)v[m]);
}

int validate_impl(tb_ctx *ctx, const void *dev, const void *expected, uint64_t num_bytes,
                  uint32_t elem, tb_mismatch *out)
{
    if (out) {
        out->index = -1;
        out->expected = out->actual = 0;
    }
    if (!ctx->val_stage)
        TB_CUDA(ctx, cudaHostAlloc(&ctx->val_stage, kValidateChunk, cudaHostAllocDefault));
    const uint8_t *d = static_cast<const uint8_t *>(dev);
    const uint8_t *e = static_cast<const uint8_t *>(expected);
    uint8_t *h = static_cast<uint8_t *>(ctx->val_stage);
    for (uint64_t off = 0; off < num_bytes; off += kValidateChunk) {
        const uint64_t len = std::min<uint64_t>(kValidateChunk, num_bytes - off);
        TB_CUDA(ctx, cudaMemcpyAsync(h, d + off, len, cudaMemcpyDeviceToHost, ctx->stream));
        TB_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
        if (memcmp(h, e + off, len) == 0)
            continue;
        uint64_t b = 0;
        while (h[b] == e[off + b])
            ++b;
        const uint64_t byte = off + b;
        const uint64_t idx = byte / elem;
        if (out) {
            out->index = (int64_t)idx;
            // The element's bytes, fetched whole (it may straddle two chunks).
            uint32_t act = 0, exp = 0;
            TB_CUDA(ctx, cudaMemcpy(&act, d + idx * elem, elem, cudaMemcpyDeviceToHost));
            memcpy(&exp, e + idx * elem, elem);
            out->expected = exp;
            out->actual = act;
        }
        return fail(ctx, TB_EVALIDATE, "destination differs from expected at element %llu",
                    (unsigned long long)idx);
    }
    return TB_OK;
}

// Device-side compare of two device ranges on ctx's stream (synchronous).
int validate_device_impl(tb_ctx *ctx, const void *dev, const void *expected_dev, uint64_t num_bytes,
                         uint32_t elem, tb_mismatch *out)
{
    if (out) {
        out->index = -1;
        out->expected = out->actual = 0;
    }
    if (!ctx->first_diff)
        TB_CUDA(ctx, cudaMalloc(&ctx->first_diff, sizeof(unsigned long long)));
    TB_CUDA(ctx, tb::launch_compare(dev, expected_dev, num_bytes, ctx->first_diff, ctx->num_sms,
                                    ctx->stream));
    unsigned long long first = 0;
    TB_CUDA(ctx, cudaMemcpyAsync(&first, ctx->first_diff, sizeof first, cudaMemcpyDeviceToHost,
                                 ctx->stream));
    TB_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
    if (first == ~0ull)
        return TB_OK;
    const uint64_t idx = first / elem;
    if (out) {
        uint32_t act = 0, exp = 0;
        TB_CUDA(ctx, cudaMemcpy(&act, static_cast<const char *>(dev) + idx * elem, elem,
                                cudaMemcpyDeviceToHost));
        TB_CUDA(ctx, cudaMemcpy(&exp, static_cast<const char *>(expected_dev) + idx * elem, elem,
                                cudaMemcpyDeviceToHost));
        out->index = (int64_t)idx;
        out->expected = exp;
        out->actual = act;
    }
    return fail(ctx, TB_EVALIDATE, "destination differs from expected at element %llu",
                (unsigned long long)idx);
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char *tb_strerror(int code)
{
    switch (code) {
    case TB_OK: return "TB_OK";
    case TB_EINVAL: return "TB_EINVAL: invalid argument";
    case TB_ENOMEM: return "TB_ENOMEM: out of memory";
    case TB_ECUDA: return "TB_ECUDA: CUDA error";
    case TB_EVALIDATE: return "TB_EVALIDATE: destination differs from expected";
    case TB_ETIMEOUT: return "TB_ETIMEOUT: bounded wait expired";
    case TB_ENOTSUP: return "TB_ENOTSUP: not supported";
    default: return "unknown tb error code";
    }
}

const char *tb_last_error(const tb_ctx *ctx)
{
    return ctx ? ctx->err.c_str() : "";
}

void tb_options_default(tb_options *o)
{
    if (!o)
        return;
    memset(o, 0, sizeof *o);
    o->rotate_bytes = 256 * kMiB;
    o->byte_offset = 0;
    o->warmup = 3;
    o->always_validate = 0;
    o->memset_byte = 0;
    o->ctas_per_subexec = 0;
    o->block_threads = 0;
    o->small_max_bytes = 16384;
    o->slot_items = 65536;
    o->num_slots = 4;
    o->wait_timeout_ns = 5000000000ull;
    o->use_gate = 1;
    o->vec_bytes = 0;
    o->unroll = 0;
    o->time_kernels = 0;
    o->reduce_engine = 0;
    o->ce_min_bytes = 0;
    o->use_graph = 1;
    o->use_pdl = 1;
    o->kernel_wait_ns = 2000000000ull;
    o->validate_direct = 0;
    o->validate_source = 0;
    o->check_overlap = 0;
    o->batch_min_copies = 0;
    o->batch_short_shape = 0;
    o->batch_max_ctas = 0;
    o->early_reads = 0;
}

int tb_parse_bytes(const char *text, uint64_t *out)
{
    if (!text || !out)
        return TB_EINVAL;
    const char *p = text;
    while (*p == ' ' || *p == '\t')
        ++p;
    if (*p < '0' || *p > '9')
        return TB_EINVAL;
    uint64_t v = 0;
    for (; *p >= '0' && *p <= '9'; ++p) {
        const uint64_t digit = (uint64_t)(*p - '0');
        if (v > (UINT64_MAX - digit) / 10)
            return TB_EINVAL;
        v = v * 10 + digit;
    }
    unsigned shift = 0;
    switch (*p) {
    case 'k': case 'K': shift = 10; break;
    case 'm': case 'M': shift = 20; break;
    case 'g': case 'G': shift = 30; break;
    case 't': case 'T': shift = 40; break;
    default: break;
    }
    if (shift) {
        ++p;
        if (*p == 'i' || *p == 'I')
            ++p;
    }
    if (*p == 'b' || *p == 'B')
        ++p;
    while (*p == ' ' || *p == '\t' || *p == '\n')
        ++p;
    if (*p != '\0')
        return TB_EINVAL;
    if (shift && v > (UINT64_MAX >> shift))
        return TB_EINVAL;
    *out = v << shift;
    return TB_OK;
}

int tb_options_from_env(tb_options *o)
{
    if (!o)
        return TB_EINVAL;
    bool bad = false;
    if (!env_u64("TB_SRC_ROTATE_BYTES", &o->rotate_bytes, &bad))
        env_u64("SRC_ROTATE_BYTES", &o->rotate_bytes, &bad);
    env_u64("TB_BYTE_OFFSET", &o->byte_offset, &bad);
    env_i32("TB_WARMUP", &o->warmup, &bad);
    if (!env_i32("TB_ALWAYS_VALIDATE", &o->always_validate, &bad))
        env_i32("ALWAYS_VALIDATE", &o->always_validate, &bad);
    if (!env_u32("TB_MEMSET_CHAR", &o->memset_byte, &bad))
        env_u32("MEMSET_CHAR", &o->memset_byte, &bad);
    env_i32("TB_CTAS_PER_SUBEXEC", &o->ctas_per_subexec, &bad);
    env_i32("TB_BLOCK_THREADS", &o->block_threads, &bad);
    env_u64("TB_SMALL_MAX_BYTES", &o->small_max_bytes, &bad);
    env_u32("TB_SLOT_ITEMS", &o->slot_items, &bad);
    env_u32("TB_NUM_SLOTS", &o->num_slots, &bad);
    env_u64("TB_WAIT_TIMEOUT_NS", &o->wait_timeout_ns, &bad);
    env_i32("TB_USE_GATE", &o->use_gate, &bad);
    env_i32("TB_VEC_BYTES", &o->vec_bytes, &bad);
    env_i32("TB_UNROLL", &o->unroll, &bad);
    env_i32("TB_TIME_KERNELS", &o->time_kernels, &bad);
    env_i32("TB_REDUCE_ENGINE", &o->reduce_engine, &bad);
    env_u64("TB_CE_MIN_BYTES", &o->ce_min_bytes, &bad);
    env_i32("TB_USE_GRAPH", &o->use_graph, &bad);
    env_i32("TB_USE_PDL", &o->use_pdl, &bad);
    env_u64("TB_KERNEL_WAIT_NS", &o->kernel_wait_ns, &bad);
    if (!env_i32("TB_VALIDATE_DIRECT", &o->validate_direct, &bad))
        env_i32("VALIDATE_DIRECT", &o->validate_direct, &bad);
    if (!env_i32("TB_VALIDATE_SOURCE", &o->validate_source, &bad))
        env_i32("VALIDATE_SOURCE", &o->validate_source, &bad);
    env_i32("TB_CHECK_OVERLAP", &o->check_overlap, &bad);
    if (!env_i32("TB_BATCH_COPY_MIN", &o->batch_min_copies, &bad))
        env_i32("MC_HIP_BATCH_COPY_MIN", &o->batch_min_copies, &bad);
    env_i32("TB_BATCH_SHORT_SHAPE", &o->batch_short_shape, &bad);
    env_i32("TB_BATCH_MAX_CTAS", &o->batch_max_ctas, &bad);
    env_i32("TB_EARLY_READS", &o->early_reads, &bad);
    return bad ? TB_EINVAL : TB_OK;
}

int tb_rotation_plan(uint64_t num_bytes, uint64_t rotate_bytes, uint64_t byte_offset, uint64_t *K,
                     uint64_t *slice_stride, uint64_t *alloc_bytes)
{
    if (num_bytes == 0 || num_bytes > UINT64_MAX - 255)
        return TB_EINVAL;
    // K = ceil(rotateBytes / numBytes); 0 disables rotation.
    const uint64_t k = rotate_bytes == 0 ? 1 : rotate_bytes / num_bytes + (rotate_bytes % num_bytes != 0);
    const uint64_t stride = (num_bytes + 255) & ~(uint64_t)255;
    if (k - 1 > (UINT64_MAX - num_bytes) / stride)
        return TB_EINVAL;
    const uint64_t span = (k - 1) * stride + num_bytes;
    if (span > UINT64_MAX - byte_offset)
        return TB_EINVAL;
    if (K)
        *K = k;
    if (slice_stride)
        *slice_stride = stride;
    if (alloc_bytes)
        *alloc_bytes = span + byte_offset;
    return TB_OK;
}

uint64_t tb_slice_for_iteration(int64_t iteration, uint64_t K)
{
    if (K == 0)
        return 0;
    if (iteration >= 0)
        return (uint64_t)iteration % K;
    // -1 -> K-1, -2 -> K-2, ...: fold the magnitude, then reflect.
    const uint64_t mag = (uint64_t)(-(iteration + 1)) + 1;
    const uint64_t r = mag % K;
    return r == 0 ? 0 : K - r;
}

int tb_create(tb_ctx **out, int device, const tb_options *opt)
{
    if (!out)
        return TB_EINVAL;
    tb_options o;
    if (opt) {
        o = *opt;
    } else {
        tb_options_default(&o);
        if (tb_options_from_env(&o) != TB_OK)
            return TB_EINVAL;
    }
    if (check_options(nullptr, o) != TB_OK)
        return TB_EINVAL;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
        return device < 0 ? TB_EINVAL : TB_ECUDA;

    tb_ctx *ctx = new (std::nothrow) tb_ctx;
    if (!ctx)
        return TB_ENOMEM;
    ctx->device = device;
    ctx->opt = o;
    DeviceScope scope(device);
    auto bail = [&](int code) {
        tb_destroy(ctx);
        return code;
    };
    if (!scope.ok())
        return bail(TB_ECUDA);
    if (cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return bail(TB_ECUDA);
    if (cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&ctx->up, cudaStreamNonBlocking) != cudaSuccess)
        return bail(TB_ECUDA);

    void *gate = nullptr;
    if (cudaHostAlloc(&gate, 4 * sizeof(uint32_t), cudaHostAllocMapped) != cudaSuccess)
        return bail(TB_ENOMEM);
    ctx->gate_flag = static_cast<volatile uint32_t *>(gate);
    ctx->gate_status = ctx->gate_flag + 1;
    ctx->reduce_status = ctx->gate_flag + 2;
    ctx->gate_flag[0] = 0;
    ctx->gate_status[0] = 0;
    ctx->reduce_status[0] = 0;
    void *dgate = nullptr;
    if (cudaHostGetDevicePointer(&dgate, gate, 0) != cudaSuccess)
        return bail(TB_ECUDA);
    ctx->gate_flag_dev = static_cast<uint32_t *>(dgate);
    ctx->gate_status_dev = ctx->gate_flag_dev + 1;
    ctx->reduce_status_dev = ctx->gate_flag_dev + 2;

    for (int k = 0; k <= tb::kShortShapes; ++k) {
        const int per_sm = tb::batch_ctas_per_sm(k);
        if (per_sm < 1)
            return bail(TB_ECUDA);
        ctx->batch_grid[k] = ctx->num_sms * per_sm;
    }
    ctx->slots.resize(o.num_slots);
    const size_t slot_bytes = tb::batch_buffer_bytes(o.slot_items);
    void *status_dev = nullptr;
    if (cudaHostAlloc(&ctx->slot_status, 2 * o.num_slots * sizeof(uint32_t), cudaHostAllocMapped) !=
            cudaSuccess ||
        cudaHostGetDevicePointer(&status_dev, ctx->slot_status, 0) != cudaSuccess)
        return bail(TB_ENOMEM);
    if (cudaMalloc(&ctx->slot_counts, o.num_slots * sizeof(uint32_t)) != cudaSuccess)
        return bail(TB_ENOMEM);
    if (cudaMemset(ctx->slot_counts, 0, o.num_slots * sizeof(uint32_t)) != cudaSuccess)
        return bail(TB_ECUDA);
    for (uint32_t i = 0; i < o.num_slots; ++i) {
        Slot &sl = ctx->slots[i];
        sl.status = static_cast<volatile uint32_t *>(ctx->slot_status) + i;
        sl.status_dev = static_cast<uint32_t *>(status_dev) + i;
        sl.done_word = static_cast<volatile uint32_t *>(ctx->slot_status) + o.num_slots + i;
        sl.done_word_dev = static_cast<uint32_t *>(status_dev) + o.num_slots + i;
        sl.count_dev = ctx->slot_counts + i;
        *sl.status = 0u;
        *sl.done_word = 0u;
    }
    for (Slot &s : ctx->slots) {
        if (cudaMalloc(&s.dev, slot_bytes) != cudaSuccess)
            return bail(TB_ENOMEM);
        if (cudaHostAlloc(&s.host, slot_bytes, cudaHostAllocMapped) != cudaSuccess)
            return bail(TB_ENOMEM);
        if (cudaHostGetDevicePointer(&s.host_dev, s.host, 0) != cudaSuccess)
            return bail(TB_ECUDA);
        if (cudaEventCreateWithFlags(&s.done_event, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.uploaded, cudaEventDisableTiming) != cudaSuccess)
            return bail(TB_ECUDA);
        if (o.time_kernels &&
            (cudaEventCreate(&s.t0) != cudaSuccess || cudaEventCreate(&s.t1) != cudaSuccess))
            return bail(TB_ECUDA);
    }
    *out = ctx;
    return TB_OK;
}

void tb_destroy(tb_ctx *ctx)
{
    if (!ctx)
        return;
    DeviceScope scope(ctx->device);
    // Quiesce first: the launches on slots, then every internal stream
    // (an upload may be queued on `up` even when its launch failed), and
    // only then free what they may still read or write.
    for (Slot &s : ctx->slots)
        if (s.done_event && s.pending)
            cudaEventSynchronize(s.done_event);
    for (cudaStream_t s : {ctx->stream, ctx->up, ctx->ce, ctx->pipe.h2d, ctx->pipe.cmp,
                           ctx->pipe.d2h})
        if (s)
            cudaStreamSynchronize(s);
    for (Slot &s : ctx->slots) {
        if (s.done_event)
            cudaEventDestroy(s.done_event);
        if (s.uploaded)
            cudaEventDestroy(s.uploaded);
        if (s.t0)
            cudaEventDestroy(s.t0);
        if (s.t1)
            cudaEventDestroy(s.t1);
        if (s.dev)
            cudaFree(s.dev);
        if (s.host)
            cudaFreeHost(s.host);
    }
    for (cudaStream_t s : {ctx->stream, ctx->up, ctx->ce})
        if (s)
            cudaStreamDestroy(s);
    for (cudaEvent_t e : ctx->events)
        cudaEventDestroy(e);
    for (cudaEvent_t e : {ctx->ce_fork, ctx->ce_join})
        if (e)
            cudaEventDestroy(e);
    Pipeline &pl = ctx->pipe;
    for (cudaStream_t s : {pl.h2d, pl.cmp, pl.d2h})
        if (s)
            cudaStreamDestroy(s);
    for (cudaEvent_t e : {pl.begin, pl.end})
        if (e)
            cudaEventDestroy(e);
    for (cudaEvent_t e : pl.in)
        cudaEventDestroy(e);
    for (cudaEvent_t e : pl.out)
        cudaEventDestroy(e);
    if (ctx->gate_flag)
        cudaFreeHost((void *)ctx->gate_flag);
    if (ctx->slot_status)
        cudaFreeHost(ctx->slot_status);
    if (ctx->slot_counts)
        cudaFree(ctx->slot_counts);
    if (ctx->val_stage)
        cudaFreeHost(ctx->val_stage);
    if (ctx->direct_expected)
        cudaFree(ctx->direct_expected);
    if (ctx->first_diff)
        cudaFree(ctx->first_diff);
    delete ctx;
}

int tb_get_options(const tb_ctx *ctx, tb_options *opt)
{
    if (!ctx || !opt)
        return TB_EINVAL;
    *opt = ctx->opt;
    return TB_OK;
}

int tb_fill_source(tb_ctx *ctx, void *dst, uint64_t num_bytes, const tb_pattern *pat,
                   int buffer_idx, tb_stream stream)
{
    if (!ctx)
        return TB_EINVAL;
    if (!dst || !pat || num_bytes % 4 != 0 || ((uintptr_t)dst & 3u) || buffer_idx < 0 ||
        buffer_idx > 40000)
        return fail(ctx, TB_EINVAL,
                    "fill_source: dst 4-byte aligned, numBytes %% 4 == 0, bufferIdx in [0, 40000]");
    if (pat->kind == TB_PATTERN_COMPRESS) {
        uint32_t total = 0;
        for (int m = 0; m < 5; ++m) {
            if (pat->compress_pct[m] > 100)
                return fail(ctx, TB_EINVAL, "fillCompress percentage above 100");
            total += pat->compress_pct[m];
        }
        if (total != 100)
            return fail(ctx, TB_EINVAL, "fillCompress percentages sum to %u, not 100", total);
    } else if (pat->kind == TB_PATTERN_REPEAT) {
        if (!pat->repeat || pat->repeat_len == 0 || pat->repeat_len > 4096)
            return fail(ctx, TB_EINVAL, "fillPattern needs 1..4096 values");
    } else if (pat->kind != TB_PATTERN_DEFAULT) {
        return fail(ctx, TB_EINVAL, "unknown pattern kind %d", pat->kind);
    }
    DeviceScope scope(ctx->device);
    TB_CUDA(ctx, tb::launch_fill_source(static_cast<float *>(dst), num_bytes / 4, *pat, buffer_idx,
                                        ctx->num_sms, static_cast<cudaStream_t>(stream)));
    return TB_OK;
}

int tb_upload_sources(tb_ctx *ctx, void *const *srcs, const void *const *host_srcs, int n_src,
                      uint64_t num_bytes)
{
    if (!ctx)
        return TB_EINVAL;
    if (n_src < 0 || n_src > TB_MAX_SRCS || (n_src > 0 && (!srcs || !host_srcs)))
        return fail(ctx, TB_EINVAL, "upload_sources: bad source list");
    DeviceScope scope(ctx->device);
    TB_CUDA(ctx, cudaDeviceSynchronize());
    for (int k = 0; k < n_src; ++k) {
        if (!srcs[k] || !host_srcs[k])
            return fail(ctx, TB_EINVAL, "upload_sources: null pointer");
        char *d = static_cast<char *>(srcs[k]) + ctx->opt.byte_offset;
        TB_CUDA(ctx, cudaMemcpyAsync(d, host_srcs[k], num_bytes, cudaMemcpyHostToDevice, ctx->stream));
        ctx->prep_h2d += num_bytes;
    }
    TB_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
    // validateSource: every device source against the host copy it came from.
    if (ctx->opt.validate_source) {
        for (int k = 0; k < n_src; ++k) {
            const char *d = static_cast<const char *>(srcs[k]) + ctx->opt.byte_offset;
            tb_mismatch mm;
            const int rc = validate_impl(ctx, d, host_srcs[k], num_bytes, 4, &mm);
            if (rc == TB_EVALIDATE)
                return fail(ctx, rc, "source %d differs from its host copy at element %lld", k,
                            (long long)mm.index);
            if (rc != TB_OK)
                return rc;
        }
    }
    return TB_OK;
}

int tb_prepare_sources(tb_ctx *ctx, void *const *srcs, int n_src, uint64_t num_bytes,
                       uint64_t rotate_bytes)
{
    if (!ctx)
        return TB_EINVAL;
    if (n_src < 0 || n_src > TB_MAX_SRCS || (n_src > 0 && !srcs) || num_bytes % 4 != 0)
        return fail(ctx, TB_EINVAL, "prepare_sources: bad arguments");
    uint64_t K = 0, stride = 0;
    if (tb_rotation_plan(num_bytes, rotate_bytes, ctx->opt.byte_offset, &K, &stride, nullptr) != TB_OK)
        return fail(ctx, TB_EINVAL, "prepare_sources: rotation plan overflows");
    DeviceScope scope(ctx->device);
    TB_CUDA(ctx, cudaDeviceSynchronize());
    // Slices [0, m) are valid; copy them onto [m, 2m) until all K are.
    const uint64_t span = (K - 1) * stride + num_bytes;
    for (int k = 0; k < n_src; ++k) {
        if (!srcs[k])
            return fail(ctx, TB_EINVAL, "prepare_sources: null source");
        char *base = static_cast<char *>(srcs[k]) + ctx->opt.byte_offset;
        for (uint64_t m = 1; m < K; m *= 2) {
            const uint64_t len = std::min<uint64_t>(m * stride, span - m * stride);
            const void *from[1] = {base};
            tb::ReducePlan p;
            int rc = plan_for(ctx, &p, from, 1, base + m * stride, len, 0);
            if (rc != TB_OK)
                return rc;
            TB_CUDA(ctx, tb::launch_reduce(p, ctx->stream));
        }
    }
    TB_CUDA(ctx, cudaStreamSynchronize(ctx->stream));
    // validateSource: every filled slice against slice 0, on the device.
    if (ctx->opt.validate_source) {
        for (int k = 0; k < n_src; ++k) {
            const char *base = static_cast<const char *>(srcs[k]) + ctx->opt.byte_offset;
            for (uint64_t j = 1; j < K; ++j) {
                tb_mismatch mm;
                const int rc = validate_device_impl(ctx, base + j * stride, base, num_bytes, 4, &mm);
                if (rc == TB_EVALIDATE)
                    return fail(ctx, rc, "source %d slice %llu differs from slice 0 at element %lld",
                                k, (unsigned long long)j, (long long)mm.index);
                if (rc != TB_OK)
                    return rc;
            }
        }
    }
    return TB_OK;
}

uint64_t tb_prep_h2d_bytes(const tb_ctx *ctx)
{
    return ctx ? ctx->prep_h2d : 0;
}

int tb_reduce_copy(tb_ctx *ctx, const void *const *srcs, int n_src, void *dst, uint64_t num_bytes,
                   int num_subexec, tb_stream stream)
{
    if (!ctx)
        return TB_EINVAL;
    DeviceScope scope(ctx->device);
    if (ctx->reduce_status[0] != 0u) {
        ctx->reduce_status[0] = 0u;
        return fail(ctx, TB_ETIMEOUT, "an earlier reduce-copy on this context stopped early: a "
                                      "bounded wait inside the kernel expired");
    }
    tb::ReducePlan p;
    int rc = plan_for(ctx, &p, srcs, n_src, dst, num_bytes, num_subexec);
    if (rc != TB_OK)
        return rc;
    p.early = ctx->opt.early_reads && p.pdl ? 1 : 0;
    TB_CUDA(ctx, tb::launch_reduce(p, static_cast<cudaStream_t>(stream)));
    return TB_OK;
}

int tb_reduce_plan(tb_ctx *ctx, const void *const *srcs, int n_src, const void *dst,
                   uint64_t num_bytes, int num_subexec, tb_launch_info *out)
{
    if (!ctx)
        return TB_EINVAL;
    if (!out)
        return fail(ctx, TB_EINVAL, "reduce_plan: null output");
    DeviceScope scope(ctx->device);
    tb::ReducePlan p;
    int rc = plan_for(ctx, &p, srcs, n_src, const_cast<void *>(dst), num_bytes, num_subexec);
    if (rc != TB_OK)
        return rc;
    out->engine = p.engine;
    out->vec_bytes = p.vec_bytes;
    out->unroll = p.unroll;
    out->block_threads = p.block_threads;
    out->grid = p.grid;
    out->num_subexec = p.num_subexec;
    out->head_elems = p.head;
    out->body_vectors = p.nvec;
    out->tail_elems = p.n - p.head - p.nvec * ((uint64_t)p.vec_bytes / 4);
    out->smem_bytes = p.smem_bytes;
    out->stages = p.engine == 2 ? p.stages : 0;
    out->tile_bytes = (int32_t)tb::plan_tile_bytes(p);
    return TB_OK;
}

int tb_reduce_copy_host(tb_ctx *ctx, const void *const *host_srcs, int n_src, void *host_dst,
                        uint64_t num_bytes, void *const *dev_srcs, void *dev_dst, int num_subexec,
                        tb_stream stream)
{
    if (!ctx)
        return TB_EINVAL;
    if (n_src < 0 || n_src > TB_MAX_SRCS || !host_dst || (n_src > 0 && !host_srcs))
        return fail(ctx, TB_EINVAL, "reduce_copy_host: bad arguments");
    for (int k = 0; k < n_src; ++k)
        if (!host_srcs[k])
            return fail(ctx, TB_EINVAL, "reduce_copy_host: null host source");
    DeviceScope scope(ctx->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Direct: every host buffer is page-locked and mapped into the device's
    // address space, so one reduce-copy kernel reads the sources and writes
    // the destination across the host link (both directions at once).
    const void *mapped[TB_MAX_SRCS];
    void *mapped_dst = mapped_host_pointer(host_dst);
    bool direct = mapped_dst != nullptr;
    for (int k = 0; direct && k < n_src; ++k)
        direct = (mapped[k] = mapped_host_pointer(host_srcs[k])) != nullptr;
    if (direct) {
        tb::ReducePlan p;
        int rc = plan_for(ctx, &p, mapped, n_src, mapped_dst, num_bytes, num_subexec);
        if (rc != TB_OK)
            return rc;
        TB_CUDA(ctx, tb::launch_reduce(p, st));
        return TB_OK;
    }

    // Staged: chunks flow host -> device copies, kernel, device -> host copy
    // on three streams, so copies in both directions overlap the kernels.
    if (!dev_dst || (n_src > 0 && !dev_srcs))
        return fail(ctx, TB_EINVAL, "reduce_copy_host: device buffers are needed for host "
                                    "memory that is not page-locked and mapped");
    for (int k = 0; k < n_src; ++k)
        if (!dev_srcs[k])
            return fail(ctx, TB_EINVAL, "reduce_copy_host: null device source");
    // Every chunk starts at a multiple of kStageChunk, so all chunks share
    // the pointers' alignments: one plan checks the arguments of all of
    // them before anything is queued.
    if (num_bytes > 0) {
        tb::ReducePlan probe;
        const int prc = plan_for(ctx, &probe, const_cast<const void *const *>(dev_srcs), n_src,
                                 dev_dst, std::min<uint64_t>(kStageChunk, num_bytes), num_subexec);
        if (prc != TB_OK)
            return prc;
        if (num_bytes % 4 != 0)
            return fail(ctx, TB_EINVAL, "reduce_copy_host: numBytes must be a multiple of 4");
    }
    int rc = ensure_pipeline(ctx);
    if (rc != TB_OK)
        return rc;
    const uint64_t chunk = kStageChunk;
    const uint64_t nchunks = num_bytes ? (num_bytes + chunk - 1) / chunk : 0;
    rc = pipeline_events(ctx, nchunks);
    if (rc != TB_OK)
        return rc;
    Pipeline &pl = ctx->pipe;
    TB_CUDA(ctx, cudaEventRecord(pl.begin, st));
    for (cudaStream_t s : {pl.h2d, pl.cmp, pl.d2h})
        TB_CUDA(ctx, cudaStreamWaitEvent(s, pl.begin, 0));
    for (uint64_t c = 0; c < nchunks; ++c) {
        const uint64_t off = c * chunk;
        const uint64_t len = std::min(chunk, num_bytes - off);
        const void *ds[TB_MAX_SRCS];
        for (int k = 0; k < n_src; ++k) {
            char *d = static_cast<char *>(dev_srcs[k]) + off;
            TB_CUDA(ctx, cudaMemcpyAsync(d, static_cast<const char *>(host_srcs[k]) + off, len,
                                         cudaMemcpyHostToDevice, pl.h2d));
            ds[k] = d;
        }
        TB_CUDA(ctx, cudaEventRecord(pl.in[c], pl.h2d));
        TB_CUDA(ctx, cudaStreamWaitEvent(pl.cmp, pl.in[c], 0));
        tb::ReducePlan p;
        rc = plan_for(ctx, &p, ds, n_src, static_cast<char *>(dev_dst) + off, len, num_subexec);
        if (rc != TB_OK)
            return rc;
        TB_CUDA(ctx, tb::launch_reduce(p, pl.cmp));
        TB_CUDA(ctx, cudaEventRecord(pl.out[c], pl.cmp));
        TB_CUDA(ctx, cudaStreamWaitEvent(pl.d2h, pl.out[c], 0));
        TB_CUDA(ctx, cudaMemcpyAsync(static_cast<char *>(host_dst) + off,
                                     static_cast<const char *>(dev_dst) + off, len,
                                     cudaMemcpyDeviceToHost, pl.d2h));
    }
    TB_CUDA(ctx, cudaEventRecord(pl.end, pl.d2h));
    TB_CUDA(ctx, cudaStreamWaitEvent(st, pl.end, 0));
    return TB_OK;
}

int tb_run_transfer_ex(tb_ctx *ctx, const tb_transfer *t, tb_result *out)
{
    if (!ctx)
        return TB_EINVAL;
    if (!t || !out || t->iters < 1 || t->n_src < 0 || t->n_src > TB_MAX_SRCS || !t->dst ||
        (t->n_src > 0 && !t->srcs))
        return fail(ctx, TB_EINVAL, "run_transfer: bad arguments");
    if (t->executor != TB_EXEC_GPU && t->executor != TB_EXEC_DMA)
        return fail(ctx, TB_EINVAL, "run_transfer: unknown executor %d", (int)t->executor);
    // The DMA executor copies one source to dst with the copy engines.
    const bool dma = t->executor == TB_EXEC_DMA;
    if (dma && t->n_src != 1)
        return fail(ctx, TB_ENOTSUP, "run_transfer: the DMA executor takes exactly one source");
    memset(out, 0, sizeof *out);
    out->mismatch_index = -1;
    const tb_options &o = ctx->opt;
    uint64_t K = 0, stride = 0, alloc = 0;
    if (tb_rotation_plan(t->num_bytes, t->rotate_bytes, o.byte_offset, &K, &stride, &alloc) != TB_OK)
        return fail(ctx, TB_EINVAL, "run_transfer: rotation plan overflows or numBytes == 0");
    DeviceScope scope(ctx->device);
    TB_CUDA(ctx, cudaDeviceSynchronize());

    // Slice-0 pointers; the plan is made once and only the source pointers
    // move between iterations (the stride keeps every slice's alignment).
    const void *base[TB_MAX_SRCS];
    for (int k = 0; k < t->n_src; ++k) {
        if (!t->srcs[k])
            return fail(ctx, TB_EINVAL, "run_transfer: null source");
        base[k] = static_cast<const char *>(t->srcs[k]) + o.byte_offset;
    }
    char *dst = static_cast<char *>(t->dst) + o.byte_offset;
    tb::ReducePlan plan;
    int rc = plan_for(ctx, &plan, base, t->n_src, dst, t->num_bytes, t->num_subexec);
    if (rc != TB_OK)
        return rc;
    auto at_iteration = [&](int64_t it) {
        const uint64_t off = tb_slice_for_iteration(it, K) * stride;
        for (int k = 0; k < t->n_src; ++k)
            plan.src[k] = reinterpret_cast<const float *>(static_cast<const char *>(base[k]) + off);
        // Every launch but the first follows one of this transfer.
        plan.early = it > -(int64_t)o.warmup;
    };
    // One iteration: the reduce-copy kernel, or on the DMA executor one
    // device-to-device copy of the iteration's slice (rotated inline).
    auto issue = [&](cudaStream_t s) -> cudaError_t {
        if (dma)
            return cudaMemcpyAsync(dst, plan.src[0], t->num_bytes, cudaMemcpyDeviceToDevice, s);
        return tb::launch_reduce(plan, s);
    };

    const int iters = t->iters;
    while ((int)ctx->events.size() < iters + 1) {
        cudaEvent_t e;
        TB_CUDA(ctx, cudaEventCreate(&e));
        ctx->events.push_back(e);
    }
    ctx->iter_ms.assign(iters, 0.0f);
    cudaStream_t st = ctx->stream;
    const bool has_expected = t->expected || t->expected_device;
    const bool per_iter_validate = o.always_validate && has_expected;
    // validateDirect: the host expected values go to the device once, before
    // the loop, and every validation compares on the GPU.
    const void *expected_dev = t->expected_device;
    if (!expected_dev && t->expected && o.validate_direct) {
        if (ctx->direct_bytes < t->num_bytes) {
            if (ctx->direct_expected)
                TB_CUDA(ctx, cudaFree(ctx->direct_expected));
            ctx->direct_expected = nullptr;
            ctx->direct_bytes = 0;
            TB_CUDA(ctx, cudaMalloc(&ctx->direct_expected, t->num_bytes));
            ctx->direct_bytes = t->num_bytes;
        }
        TB_CUDA(ctx, cudaMemcpy(ctx->direct_expected, t->expected, t->num_bytes,
                                cudaMemcpyHostToDevice));
        expected_dev = ctx->direct_expected;
    }
    auto check = [&](tb_mismatch *mm) {
        return expected_dev ? validate_device_impl(ctx, dst, expected_dev, t->num_bytes, 4, mm)
                            : validate_impl(ctx, dst, t->expected, t->num_bytes, 4, mm);
    };
    // Graph: the whole loop (warm-up and timed iterations, the per-iteration
    // event records as external event nodes) captured and launched as one
    // CUDA graph - no host launch gaps and less launch work on the GPU per
    // iteration.  Per-iteration validation needs the host between
    // iterations, so it keeps the stream loop.
    const bool graphed = o.use_graph && !per_iter_validate;
    if (graphed) {
        int rc2 = run_graphed(ctx, iters, at_iteration, issue);
        if (rc2 != TB_OK)
            return rc2;
    }
    const bool gated = !graphed && o.use_gate && !per_iter_validate &&
                       o.warmup + iters <= kMaxGatedLaunches && !profiler_attached();

    if (gated) {
        ctx->gate_flag[0] = 0;
        ctx->gate_status[0] = 0;
        TB_CUDA(ctx, tb::launch_gate(ctx->gate_flag_dev, ctx->gate_status_dev, o.wait_timeout_ns, st));
    }
    int first_err = TB_OK;
    // A failed call inside the loop releases the gate before returning, so
    // the launches already queued behind it run and the stream drains.
    auto abort_loop = [&](cudaError_t e, const char *what) {
        if (gated)
            __atomic_store_n(ctx->gate_flag, 1u, __ATOMIC_SEQ_CST);
        cudaStreamSynchronize(st);
        return cuda_fail(ctx, e, what);
    };
    for (int64_t it = graphed ? iters : -(int64_t)o.warmup; it < iters; ++it) {
        at_iteration(it);
        cudaError_t e = cudaSuccess;
        if (it == 0 || (per_iter_validate && it > 0))
            if ((e = cudaEventRecord(ctx->events[it], st)) != cudaSuccess)
                return abort_loop(e, "cudaEventRecord");
        if ((e = issue(st)) != cudaSuccess)
            return abort_loop(e, dma ? "DMA copy" : "reduce-copy launch");
        if (it >= 0 && (e = cudaEventRecord(ctx->events[it + 1], st)) != cudaSuccess)
            return abort_loop(e, "cudaEventRecord");
        if (per_iter_validate && it >= 0) {
            tb_mismatch mm;
            first_err = check(&mm);
            if (first_err != TB_OK) {
                out->mismatch_index = mm.index;
                out->mismatch_expected = mm.expected;
                out->mismatch_actual = mm.actual;
                out->iters = (int)it + 1;
                break;
            }
        }
    }
    if (gated)
        __atomic_store_n(ctx->gate_flag, 1u, __ATOMIC_SEQ_CST);
    TB_CUDA(ctx, cudaStreamSynchronize(st));
    if (gated && ctx->gate_status[0] != 1u)
        return fail(ctx, TB_ETIMEOUT, "gate kernel was not released within %llu ns",
                    (unsigned long long)o.wait_timeout_ns);
    if (ctx->reduce_status[0] != 0u) {
        ctx->reduce_status[0] = 0u;
        return fail(ctx, TB_ETIMEOUT, "a bounded wait inside the reduce-copy kernel expired");
    }

    const int done = first_err != TB_OK ? out->iters : iters;
    double total = 0.0;
    if (graphed) {
        // One span for all timed iterations; each iteration gets the mean.
        float ms = 0.0f;
        TB_CUDA(ctx, cudaEventElapsedTime(&ms, ctx->events[0], ctx->events[iters]));
        total = ms;
        for (int i = 0; i < done; ++i)
            ctx->iter_ms[i] = (float)(total / done);
    } else {
        for (int i = 0; i < done; ++i) {
            float ms = 0.0f;
            TB_CUDA(ctx, cudaEventElapsedTime(&ms, ctx->events[i], ctx->events[i + 1]));
            ctx->iter_ms[i] = ms;
            total += ms;
        }
    }
    out->K = K;
    out->slice_stride = stride;
    out->alloc_bytes = alloc;
    out->prep_h2d_bytes = ctx->prep_h2d;
    out->iters = done;
    out->num_subexec = dma ? 1 : plan.num_subexec;
    out->ctas = dma ? 0 : plan.grid;
    out->block_threads = dma ? 0 : plan.block_threads;
    out->gated = gated ? 1 : 0;
    out->graphed = graphed ? 1 : 0;
    out->engine = dma ? 0 : plan.engine;
    out->executor = t->executor;
    out->total_ms = total;
    if (done > 0) {
        std::vector<float> v(ctx->iter_ms.begin(), ctx->iter_ms.begin() + done);
        out->mean_ms = total / done;
        out->median_ms = median_of(v);
        out->min_ms = *std::min_element(v.begin(), v.end());
        out->max_ms = *std::max_element(v.begin(), v.end());
        out->gbps = total > 0 ? (double)(t->n_src + 1) * (double)t->num_bytes * done / (total * 1e6)
                              : 0.0;
    }
    out->iter_ms = ctx->iter_ms.data();
    if (first_err != TB_OK) {
        out->validated = 1;
        return first_err;
    }
    if (has_expected) {
        out->validated = 1;
        tb_mismatch mm;
        rc = check(&mm);
        if (rc != TB_OK) {
            out->mismatch_index = mm.index;
            out->mismatch_expected = mm.expected;
            out->mismatch_actual = mm.actual;
            return rc;
        }
    }
    return TB_OK;
}

int tb_run_transfer(tb_ctx *ctx, void *const *srcs, int n_src, void *dst, uint64_t num_bytes,
                    int num_subexec, int iters, uint64_t rotate_bytes, tb_result *out)
{
    tb_transfer t;
    t.srcs = srcs;
    t.n_src = n_src;
    t.dst = dst;
    t.num_bytes = num_bytes;
    t.num_subexec = num_subexec;
    t.iters = iters;
    t.rotate_bytes = rotate_bytes;
    t.expected = nullptr;
    t.expected_device = nullptr;
    t.executor = TB_EXEC_GPU;
    return tb_run_transfer_ex(ctx, &t, out);
}

int tb_batch_copy(tb_ctx *ctx, const tb_copy_desc *desc, size_t n, tb_stream stream)
{
    if (!ctx)
        return TB_EINVAL;
    if (n > 0 && !desc)
        return fail(ctx, TB_EINVAL, "batch_copy: null descriptor array");
    const tb_options &o = ctx->opt;
    const uint64_t small = o.small_max_bytes;
    const uint64_t ce_min = o.ce_min_bytes;
    DeviceScope scope(ctx->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // A captured call would leave the graph reading the slot's staging when
    // it is replayed, after later calls have packed other work lists into
    // it, and its completion event would never be recorded; so a capturing
    // stream is refused before anything is queued on it.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    TB_CUDA(ctx, cudaStreamIsCapturing(s, &capture));
    if (capture != cudaStreamCaptureStatusNone)
        return fail(ctx, TB_ENOTSUP,
                    "batch_copy: the stream is capturing a CUDA graph; the packed work list "
                    "lives in staging that later calls reuse");
    ctx->last_slots.clear();
    tb_batch_stats st{};
    // Work lists go up on the internal upload stream, so that a call's upload
    // overlaps the kernel of the call before it; the kernel waits for it on
    // the caller's stream.  The slot is free by then: wait_slot has seen its
    // previous kernel finish.

    // A batch that fits one slot is checked and packed in a single pass
    // straight into the slot's pinned staging.  A larger one is checked as a
    // whole first, so that no launch happens for a batch that is rejected.
    const bool one_slot = n <= o.slot_items;
    size_t bad = 0;
    if (!one_slot || o.check_overlap) {
        tb::BatchCounts all;
        if (tb::count_batch(desc, n, small, &all, &bad, ce_min) != TB_OK)
            return fail(ctx, TB_EINVAL, "batch_copy: descriptor %zu has a null or wrapping range",
                        bad);
    }
    // Fewer copies than batch_min_copies: one cudaMemcpyAsync each, no kernel.
    size_t nonempty = 0;
    for (size_t i = 0; i < n && nonempty < (size_t)o.batch_min_copies; ++i)
        nonempty += desc[i].len != 0;
    if (nonempty < (size_t)o.batch_min_copies) {
        tb::BatchCounts few;
        if (tb::count_batch(desc, n, small, &few, &bad, 0) != TB_OK)
            return fail(ctx, TB_EINVAL, "batch_copy: descriptor %zu has a null or wrapping range",
                        bad);
        if (o.check_overlap) {
            size_t a = 0, b = 0;
            if (tb::find_overlap(desc, n, &a, &b))
                return fail(ctx, TB_EINVAL, "batch_copy: descriptors %zu and %zu overlap",
                            std::min(a, b), std::max(a, b));
        }
        for (size_t i = 0; i < n; ++i)
            if (desc[i].len)
                TB_CUDA(ctx, cudaMemcpyAsync(reinterpret_cast<void *>(desc[i].dst),
                                             reinterpret_cast<const void *>(desc[i].src),
                                             desc[i].len, cudaMemcpyDeviceToDevice, s));
        st.descs = few.descs;
        st.bytes = few.bytes;
        st.ce_copies = few.descs;
        ctx->last_batch = st;
        return TB_OK;
    }
    if (o.check_overlap) {
        size_t a = 0, b = 0;
        if (tb::find_overlap(desc, n, &a, &b))
            return fail(ctx, TB_EINVAL,
                        "batch_copy: descriptors %zu and %zu overlap (a destination over another "
                        "destination or over a source)",
                        std::min(a, b), std::max(a, b));
    }
    if (ctx->longs.size() < std::min<size_t>(n, o.slot_items))
        ctx->longs.resize(std::min<size_t>(n, o.slot_items));

    // Copies forked to the copy-engine stream are joined back into the
    // caller's stream on every way out, a failed call's too, so that work
    // queued on it afterwards comes after them.
    bool forked = false;
    struct JoinOnExit {
        tb_ctx *ctx;
        cudaStream_t s;
        const bool &forked;
        ~JoinOnExit()
        {
            if (forked && cudaEventRecord(ctx->ce_join, ctx->ce) == cudaSuccess)
                cudaStreamWaitEvent(s, ctx->ce_join, 0);
        }
    } join_on_exit{ctx, s, forked};
    size_t begin = 0;
    do {
        // The next run of at most slot_items descriptors.
        const size_t end = std::min(n, begin + (size_t)o.slot_items);
        Slot &slot = ctx->slots[ctx->next_slot];
        int rc = wait_slot(ctx, slot);
        if (rc != TB_OK)
            return rc;
        tb::BatchCounts c;
        if (tb::gather_batch(desc + begin, end - begin, small, ce_min, slot.host, ctx->longs.data(),
                             &c, &bad) != TB_OK)
            return fail(ctx, TB_EINVAL, "batch_copy: descriptor %zu has a null or wrapping range",
                        begin + bad);
        st.descs += c.descs;
        st.bytes += c.bytes;
        st.ce_copies += c.n_ce;

        // Copies routed to the copy engines run on a stream forked from the
        // caller's, alongside the kernel, and are joined back at the end.
        if (c.n_ce) {
            if (!ctx->ce) {
                TB_CUDA(ctx, cudaStreamCreateWithFlags(&ctx->ce, cudaStreamNonBlocking));
                TB_CUDA(ctx, cudaEventCreateWithFlags(&ctx->ce_fork, cudaEventDisableTiming));
                TB_CUDA(ctx, cudaEventCreateWithFlags(&ctx->ce_join, cudaEventDisableTiming));
            }
            if (!forked) {
                TB_CUDA(ctx, cudaEventRecord(ctx->ce_fork, s));
                TB_CUDA(ctx, cudaStreamWaitEvent(ctx->ce, ctx->ce_fork, 0));
                forked = true;
            }
            for (size_t i = begin; i < end; ++i)
                if (desc[i].len && desc[i].len >= ce_min)
                    TB_CUDA(ctx, cudaMemcpyAsync(reinterpret_cast<void *>(desc[i].dst),
                                                 reinterpret_cast<const void *>(desc[i].src),
                                                 desc[i].len, cudaMemcpyDeviceToDevice, ctx->ce));
        }
        if (c.n_short + c.n_long > 0) {
            tb::BatchPlan plan;
            const int shape = tb::short_shape_for(
                c, o.batch_short_shape, (uint64_t)ctx->batch_grid[2] * (tb::kBatchThreads / 32));
            int grid = tb::batch_grid(c, ctx->batch_grid[shape]);
            if (o.batch_max_ctas > 0 && grid > o.batch_max_ctas)
                grid = o.batch_max_ctas;
            tb::finish_batch(c, ctx->longs.data(), grid, slot.host, &plan);
            plan.shape = shape;
            ctx->next_slot = (ctx->next_slot + 1) % (uint32_t)ctx->slots.size();
            // A small batch of short copies all assigned by warp index reads
            // its work list in place from the pinned staging: no upload and
            // no cross-stream event, which is most of a small call's cost.
            // The staging is not rewritten before the kernel has finished:
            // wait_slot waits for it first.
            const bool direct = tb::batch_direct(plan);
            if (direct) {
                st.direct_launches += 1;
            } else {
                TB_CUDA(ctx, cudaMemcpyAsync(slot.dev, slot.host, plan.upload_bytes,
                                             cudaMemcpyHostToDevice, ctx->up));
                TB_CUDA(ctx, cudaEventRecord(slot.uploaded, ctx->up));
                TB_CUDA(ctx, cudaStreamWaitEvent(s, slot.uploaded, 0));
            }
            if (slot.t0)
                TB_CUDA(ctx, cudaEventRecord(slot.t0, s));
            tb::BatchDone done;
            done.count = slot.count_dev;
            done.word = slot.done_word_dev;
            done.base = slot.count;
            done.seq = slot.seq + 1;
            const cudaError_t le = tb::launch_batch(direct ? slot.host_dev : slot.dev, plan, s,
                                                    slot.status_dev, o.kernel_wait_ns, done,
                                                    o.use_pdl != 0);
            if (le != cudaSuccess) {
                // The slot is not marked pending, so its staging may be
                // rewritten next: let a queued upload finish reading it.
                if (!direct)
                    cudaStreamSynchronize(ctx->up);
                return cuda_fail(ctx, le, "launch of the batch kernel");
            }
            // The kernel runs: the slot's staging stays untouched until it
            // has signalled (or its event has been reached).
            slot.seq = done.seq;
            slot.count += plan.grid;
            slot.pending = true;
            ctx->last_slots.push_back((uint32_t)(&slot - ctx->slots.data()));
            if (slot.t1)
                TB_CUDA(ctx, cudaEventRecord(slot.t1, s));
            TB_CUDA(ctx, cudaEventRecord(slot.done_event, s));
            st.launches += 1;
            st.warp_items += plan.n_short;
            st.cta_items += plan.chunks;
            st.upload_bytes += plan.upload_bytes;
        }
        begin = end;
    } while (begin < n);
    if (forked) {
        forked = false;
        TB_CUDA(ctx, cudaEventRecord(ctx->ce_join, ctx->ce));
        TB_CUDA(ctx, cudaStreamWaitEvent(s, ctx->ce_join, 0));
    }
    ctx->last_batch = st;
    return TB_OK;
}

int tb_last_batch_kernel_ms(tb_ctx *ctx, double *ms)
{
    if (!ctx || !ms)
        return TB_EINVAL;
    if (!ctx->opt.time_kernels)
        return fail(ctx, TB_ENOTSUP, "the context was created without time_kernels");
    DeviceScope scope(ctx->device);
    double total = 0.0;
    for (uint32_t i : ctx->last_slots) {
        Slot &s = ctx->slots[i];
        TB_CUDA(ctx, cudaEventSynchronize(s.t1));
        if (*s.status != 0u)
            return fail(ctx, TB_ETIMEOUT, "the last batch stopped early: a bounded wait inside "
                                          "the kernel expired");
        float t = 0.0f;
        TB_CUDA(ctx, cudaEventElapsedTime(&t, s.t0, s.t1));
        total += t;
    }
    *ms = total;
    return TB_OK;
}

int tb_copy_each(tb_ctx *ctx, const tb_copy_desc *desc, size_t n, tb_stream stream)
{
    if (!ctx)
        return TB_EINVAL;
    if (n > 0 && !desc)
        return fail(ctx, TB_EINVAL, "copy_each: null descriptor array");
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len && (d.src == 0 || d.dst == 0 || d.src + d.len < d.src || d.dst + d.len < d.dst))
            return fail(ctx, TB_EINVAL, "copy_each: descriptor %zu has a null or wrapping range", i);
    }
    DeviceScope scope(ctx->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (size_t i = 0; i < n; ++i) {
        const tb_copy_desc &d = desc[i];
        if (d.len)
            TB_CUDA(ctx, cudaMemcpyAsync(reinterpret_cast<void *>(d.dst),
                                         reinterpret_cast<const void *>(d.src), d.len,
                                         cudaMemcpyDeviceToDevice, s));
    }
    return TB_OK;
}

int tb_last_batch_stats(const tb_ctx *ctx, tb_batch_stats *out)
{
    if (!ctx || !out)
        return TB_EINVAL;
    *out = ctx->last_batch;
    return TB_OK;
}

int tb_validate_device(tb_ctx *ctx, const void *dst_device, const void *expected_device,
                       uint64_t num_bytes, uint32_t elem_size, tb_mismatch *out)
{
    if (!ctx)
        return TB_EINVAL;
    if ((num_bytes > 0 && (!dst_device || !expected_device)) ||
        (elem_size != 1 && elem_size != 2 && elem_size != 4) || num_bytes % elem_size != 0)
        return fail(ctx, TB_EINVAL, "validate_device: bad arguments");
    DeviceScope scope(ctx->device);
    TB_CUDA(ctx, cudaDeviceSynchronize());
    return validate_device_impl(ctx, dst_device, expected_device, num_bytes, elem_size, out);
}

int tb_validate(tb_ctx *ctx, const void *dst_device, const void *expected_host, uint64_t num_bytes,
                uint32_t elem_size, tb_mismatch *out)
{
    if (!ctx)
        return TB_EINVAL;
    if ((num_bytes > 0 && (!dst_device || !expected_host)) ||
        (elem_size != 1 && elem_size != 2 && elem_size != 4) || num_bytes % elem_size != 0)
        return fail(ctx, TB_EINVAL, "validate: bad arguments");
    DeviceScope scope(ctx->device);
    TB_CUDA(ctx, cudaDeviceSynchronize());
    return validate_impl(ctx, dst_device, expected_host, num_bytes, elem_size, out);
}

}  // extern "C"

/*
 * tb.h - C ABI of libtb, a single-GPU GB300 (sm_103a) reduce-copy and
 * batched-copy engine.
 *
 * Two operations sit on the hot path:
 *
 *  1. The GPU-executor transfer of TransferBench: dst[i] = src0[i] + ... +
 *     srcN-1[i] over float32 buffers, with source-slice rotation so that
 *     repeated iterations read HBM rather than L2.
 *       - "TransferBench data validation" (ROCm docs 1.66.02), table
 *         "Number of sources / Expected value" and section
 *         "Expected destination (dstReference)": 0 sources -> memset value,
 *         1 source -> dst == src0, N sources -> the left-to-right float sum.
 *       - TransferBench PR #365 "source-slice rotation (SRC_ROTATE_BYTES)",
 *         section "Technical Details": K = ceil(SRC_ROTATE_BYTES / numBytes),
 *         allocation K * numBytes + byteOffset, slices 1..K-1 filled
 *         device-to-device from slice 0, iteration i reads slice i % K, the
 *         rotation kept outside the timed region.
 *
 *  2. The batched descriptor copy of the Mooncake RFC #5041
 *     ("HipTransport: fast, correct intra-node XGMI", section
 *     "Design of #5040"): many scattered copies of 64 B - 16 MiB run as one
 *     kernel over a (src, dst, len) descriptor array instead of one memcpy
 *     call each; the caller's stream orders it (section "Item 4: ordering
 *     after the caller's stream", first option: an explicit stream argument).
 *
 * Conventions for every entry point:
 *   - Return 0 (TB_OK) or a negative TB_E* code; tb_strerror() names it and
 *     tb_last_error() returns a sentence about the last failure on a context.
 *   - Device pointers are plain CUDA device addresses of the context's device
 *     (interior pointers into caching-allocator blocks are fine).  The caller
 *     owns every buffer it passes; the library owns only what it allocates
 *     inside a context (staging, descriptor slots, events, timing arrays).
 *   - tb_stream is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.
 *   - Nothing falls back to a different copy method on failure: an error is
 *     returned instead, so a benchmark never silently measures something else.
 *   - Synchronous calls (tb_upload_sources, tb_prepare_sources,
 *     tb_run_transfer*, tb_validate*) first wait until all work already queued
 *     on the device has finished, so they see the results of earlier
 *     asynchronous calls on any stream.
 *   - A context is not thread-safe; use one context per host thread.
 */
#ifndef TB_H
#define TB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------------- */
/* Error codes                                                              */
/* ----------------------------------------------------------------------- */
#define TB_OK          0
#define TB_EINVAL     (-1)  /* bad argument: null pointer, bad size, overflow */
#define TB_ENOMEM     (-2)  /* a host or device allocation of the library failed */
#define TB_ECUDA      (-3)  /* a CUDA call failed; tb_last_error() has the text */
#define TB_EVALIDATE  (-4)  /* destination differs from the expected bytes */
#define TB_ETIMEOUT   (-5)  /* a bounded wait (descriptor slot, gate) expired */
#define TB_ENOTSUP    (-6)  /* request outside what the library supports */

/* Most sources one reduce-copy accepts. */
#define TB_MAX_SRCS 16

typedef struct tb_ctx tb_ctx;
typedef void *tb_stream;

/* ----------------------------------------------------------------------- */
/* Options                                                                  */
/* ----------------------------------------------------------------------- */
typedef struct {
    /* SRC_ROTATE_BYTES of PR #365: bytes of rotation per source.
       Default 256 MiB; 0 disables rotation (K = 1). */
    uint64_t rotate_bytes;
    /* Bytes between the start of each source allocation (and of dst) and the
       first data byte ("K * numBytes + byteOffset").  Multiple of 4. Default 0. */
    uint64_t byte_offset;
    /* Untimed iterations before the timed ones (indices -warmup .. -1).
       Default 3. */
    int32_t warmup;
    /* ALWAYS_VALIDATE: 1 = validate after every timed iteration and stop at
       the first error; 0 = once after the loop.  Default 0. */
    int32_t always_validate;
    /* MEMSET_CHAR: the byte a 0-source transfer writes.  Default 0. */
    uint32_t memset_byte;
    /* Reduce-copy CTAs per sub-executor.  0 = the library's grid dealt to
       the sub-executors as evenly as possible (at least one each): for the
       vector form one wave of resident CTAs (fewer for a small transfer),
       for the bulk form one CTA per ~4 tiles of work, at least one wave;
       1 gives TransferBench's one CTA per sub-executor.  Default 0. */
    int32_t ctas_per_subexec;
    /* Reduce-copy threads per CTA (multiple of 32, <= 512); 0 = the
       library's choice: 512 or 256, whichever keeps more threads resident
       per SM, or 1024 for a CTA alone on its SM (one CTA per sub-executor,
       no more CTAs than SMs) with 2 to 4 sources. */
    int32_t block_threads;
    /* Batched copy: descriptors up to this many bytes are copied by one
       warp; the bytes of all longer ones are shared equally among the CTAs.
       Default 16384, at most 16 MiB. */
    uint64_t small_max_bytes;
    /* Batched copy: non-empty descriptors one descriptor slot holds, and how
       many slots the ring has.  A batch with more runs as several launches.
       Defaults 65536 and 4. */
    uint32_t slot_items;
    uint32_t num_slots;
    /* Limit of every bounded wait (descriptor slot reuse, gate kernel), in
       nanoseconds.  Default 5e9. */
    uint64_t wait_timeout_ns;
    /* 1 = tb_run_transfer enqueues its iterations behind a gate kernel that
       the host releases once everything is queued, so host launch overhead
       never separates iterations (nvbandwidth's spin-kernel method).
       Ignored when a CUDA profiling tool is injected (CUDA_INJECTION64_PATH
       set): such tools finish each launch before the launch call returns.
       Default 1. */
    int32_t use_gate;
    /* Reduce-copy vector width in bytes: 32, 16, or 0 = the widest that every
       pointer of the launch shares the alignment of (4-byte scalar loads when
       they share no 16-byte alignment).  Default 0. */
    int32_t vec_bytes;
    /* Reduce-copy vectors per source each thread keeps in flight (1, 2 or 4);
       0 = chosen from the source count.  Default 0. */
    int32_t unroll;
    /* 1 = bracket every batched-copy kernel with CUDA events so that
       tb_last_batch_kernel_ms can report its device time.  Default 0. */
    int32_t time_kernels;
    /* Reduce-copy engine: 1 = vector loads and stores by every thread;
       2 = bulk copies (cp.async.bulk) through shared-memory stages with the
       adds done in shared memory (sources sharing a 16-byte alignment, else
       TB_ENOTSUP); 0 = the library's choice, by what measured faster on
       GB300: 2 where it applies, vec_bytes is 0 and each source holds at
       least 12 MiB (one or two sources), 8 MiB (three), 6 MiB (four),
       4 MiB (five), 3 MiB (six to eight), 1 MiB (nine to fourteen), or 1
       to 32 MiB (fifteen and sixteen); else 1.  A split of at most one CTA
       per SM (ctas_per_subexec with few sub-executors) with 2 to 4 sources
       sharing a 32-byte alignment takes 1 in 1024-thread CTAs, which stream
       more per SM than a lone bulk pipeline.  Default 0. */
    int32_t reduce_engine;
    /* Batched copy: descriptors of at least this many bytes go to the copy
       engines (one cudaMemcpyAsync each, on an internal stream forked from
       the caller's and joined back) while the kernel copies the rest, as the
       Mooncake RFC does for copies over 1 MiB.  0 = everything in the
       kernel.  Default 0. */
    uint64_t ce_min_bytes;
    /* 1 = tb_run_transfer captures its whole iteration loop (warm-up and
       timed launches) into one CUDA graph and launches that: no host gaps
       between iterations and less launch work per iteration on the GPU.
       Only the span of the timed iterations is recorded (an event between
       every two launches costs more than the graph saves), so every
       iteration reports the mean; use 0 for per-iteration events.  Not used
       with always_validate, which needs the host between iterations.
       Default 1. */
    int32_t use_graph;
    /* 1 = reduce-copy and batched-copy kernels are launched with
       programmatic dependent launch: a launch may be scheduled while the
       previous kernel on its stream drains, and every CTA waits for that
       kernel to complete and its writes to be visible before it touches the
       copies' bytes, so the results are those of serialised launches with
       less idle time between them.  A batched-copy launch reads its own
       work list before that wait.  Inside tb_run_transfer, where the launch
       before is one of the same transfer (same sources, writing only dst),
       a launch starts reading its sources before that wait; only its writes
       wait.  Default 1. */
    int32_t use_pdl;
    /* Limit, in nanoseconds, of each wait inside the kernels' shared-memory
       pipelines (bulk reduce-copy, batched copy) for a load to land.  A wait
       that runs out makes the kernel record the failure in a status word,
       wait (up to 2 s each) for the loads it has already issued, and stop;
       the call that reads the status returns TB_ETIMEOUT (tb_run_transfer;
       for batches, the next call that reuses the slot, or
       tb_last_batch_kernel_ms).  0 = never wait: a load that has not landed
       at the first check counts as expired.  Default 2e9. */
    uint64_t kernel_wait_ns;
    /* TransferBench's validateDirect: 1 = tb_run_transfer compares dst with
       the expected values on the GPU (the host `expected` copied once to a
       context-owned device buffer before the loop) instead of copying dst
       to the host for every validation.  Unused when the transfer gives
       expected_device.  Default 0. */
    int32_t validate_direct;
    /* TransferBench's validateSource: 1 = check the sources right after they
       are initialised: tb_upload_sources compares each device source with
       its host copy, tb_prepare_sources every filled slice with slice 0;
       a difference returns TB_EVALIDATE naming source, slice and element.
       Default 0. */
    int32_t validate_source;
    /* 1 = tb_batch_copy first sorts the descriptors' ranges and rejects,
       with TB_EINVAL naming two of them and nothing launched, a batch whose
       result would depend on the order of its copies: two overlapping
       destinations, or a destination overlapping a source.  O(n log n) on
       the host; a debugging aid.  Default 0. */
    int32_t check_overlap;
    /* The Mooncake RFC's MC_HIP_BATCH_COPY_MIN: a batch with fewer non-empty
       descriptors than this is copied with one cudaMemcpyAsync per
       descriptor on `stream` instead of a kernel launch (counted in
       tb_batch_stats.ce_copies).  0 = always the kernel.  Default 0. */
    int32_t batch_min_copies;
    /* Batched copy: the kernel shape of a launch of short copies only (the
       per-warp ring of shared-memory slots and the CTAs kept per SM):
       1 = four 2 KiB slots per warp, 3 CTAs per SM; 2 = two 2 KiB slots,
       5 CTAs per SM; 0 = the library's choice (2 when every copy gets a warp
       of one wave of shape 2, else 1).  Launches with long copies are not
       affected.  Default 0. */
    int32_t batch_short_shape;
    /* Batched copy: most CTAs one kernel launch may use (0 = no cap), the
       analogue of the CU mask the Mooncake RFC's open question 4 asks about
       for GPUs that also run compute.  Fewer CTAs copy more slowly and take
       fewer SMs at once; results do not change.  Default 0. */
    int32_t batch_max_ctas;
    /* 1 = a tb_reduce_copy launch (with use_pdl) may start reading its
       sources before the launch of this library queued ahead of it on the
       stream has finished, as every launch after the first does inside
       tb_run_transfer's loop; its writes still wait.  Only for callers whose
       earlier work on that stream never writes this launch's sources, for
       example successive reduce-copies over slices nothing writes: a launch
       reading the previous one's output must keep 0.  Default 0. */
    int32_t early_reads;
} tb_options;

/* Fills *opt with the defaults above. */
void tb_options_default(tb_options *opt);

/* Overrides fields of *opt from the environment:
     TB_SRC_ROTATE_BYTES (or SRC_ROTATE_BYTES), TB_BYTE_OFFSET, TB_WARMUP,
     TB_ALWAYS_VALIDATE (or ALWAYS_VALIDATE), TB_MEMSET_CHAR (or MEMSET_CHAR),
     TB_CTAS_PER_SUBEXEC,
     TB_BLOCK_THREADS, TB_SMALL_MAX_BYTES, TB_SLOT_ITEMS,
     TB_NUM_SLOTS, TB_WAIT_TIMEOUT_NS, TB_USE_GATE, TB_VEC_BYTES, TB_UNROLL,
     TB_TIME_KERNELS, TB_REDUCE_ENGINE, TB_CE_MIN_BYTES, TB_USE_GRAPH,
     TB_USE_PDL, TB_KERNEL_WAIT_NS, TB_VALIDATE_DIRECT (or VALIDATE_DIRECT),
     TB_VALIDATE_SOURCE (or VALIDATE_SOURCE), TB_CHECK_OVERLAP, TB_BATCH_COPY_MIN
     (or MC_HIP_BATCH_COPY_MIN; batch_min_copies), TB_BATCH_SHORT_SHAPE,
     TB_BATCH_MAX_CTAS, TB_EARLY_READS.
   A TB_ name, when set, wins over the bare name beside it; the bare names are
   the ones TransferBench and Mooncake read, so their users' environments
   carry over.  Byte counts go through tb_parse_bytes.  Returns TB_EINVAL
   (leaving *opt partly updated) if a variable does not parse. */
int tb_options_from_env(tb_options *opt);

/* Parses an unsigned byte count: decimal digits, optionally followed by one of
   K, M, G, T (binary: 2^10, 2^20, 2^30, 2^40), optionally followed by "B" or
   "iB", case-insensitive; surrounding blanks are allowed.  "256M" and "256MB"
   are 268,435,456.  Rejects signs, empty input, trailing junk and any value
   that does not fit in 64 bits (TB_EINVAL) - PR #365's review asks that
   SRC_ROTATE_BYTES never overflow a signed type. */
int tb_parse_bytes(const char *text, uint64_t *out);

/* ----------------------------------------------------------------------- */
/* Context                                                                  */
/* ----------------------------------------------------------------------- */

/* Creates a context on CUDA device `device`.  opt == NULL takes the defaults
   with environment overrides.  Allocates pinned staging, descriptor slots and
   events.  *out is set only on success. */
int tb_create(tb_ctx **out, int device, const tb_options *opt);

/* Waits for the context's outstanding work, then frees everything it owns.
   NULL is accepted. */
void tb_destroy(tb_ctx *ctx);

/* Copies the context's options to *opt. */
int tb_get_options(const tb_ctx *ctx, tb_options *opt);

/* Text of the last error recorded on ctx ("" if none). Valid until the next
   call on ctx. */
const char *tb_last_error(const tb_ctx *ctx);

/* Static name of an error code. */
const char *tb_strerror(int code);

/* ----------------------------------------------------------------------- */
/* Rotation plan (host only, no GPU needed)                                 */
/* ----------------------------------------------------------------------- */

/* PR #365 "Technical Details": K = ceil(rotateBytes / numBytes), or 1 when
   rotateBytes == 0.  Slice j starts at byteOffset + j * sliceStride, where
   sliceStride = numBytes rounded up to 256 bytes so every slice keeps the
   alignment of slice 0 for vector loads.  allocBytes = (K - 1) * sliceStride
   + numBytes + byteOffset, i.e. the page's K * numBytes + byteOffset whenever
   numBytes is a multiple of 256 (4 MiB at the 256 MiB default: K = 64,
   268,435,456 bytes).  Any output pointer may be NULL.  TB_EINVAL for
   numBytes == 0 or 64-bit overflow. */
int tb_rotation_plan(uint64_t numBytes, uint64_t rotateBytes, uint64_t byteOffset,
                     uint64_t *K, uint64_t *sliceStride, uint64_t *allocBytes);

/* The slice iteration `iteration` reads: iteration folded into [0, K), so the
   negative warm-up indices -warmup..-1 read slices K-warmup..K-1. */
uint64_t tb_slice_for_iteration(int64_t iteration, uint64_t K);

/* ----------------------------------------------------------------------- */
/* Source preparation ("TransferBench data validation", section            */
/* "Expected source pattern" and "Initializing source and destination       */
/* memories")                                                               */
/* ----------------------------------------------------------------------- */

#define TB_PATTERN_DEFAULT   0  /* PrepSrcValue(bufferIdx, i) */
#define TB_PATTERN_COMPRESS  1  /* fillCompress */
#define TB_PATTERN_REPEAT    2  /* fillPattern */

typedef struct {
    int32_t kind;             /* TB_PATTERN_* */
    /* TB_PATTERN_COMPRESS: percentages of 64-byte lines in mode 0 (random),
       1 (1B0), 2 (2B0), 3 (4B0), 4 (32B0); they must sum to 100.  Mode nB0
       zeroes every odd-numbered aligned n-byte chunk of its line.  Line L of
       buffer k draws SplitMix64 outputs number 17L .. 17L+16 of the stream
       seeded with seed + k: the first picks the mode ((draw % 100) against
       the running sum of the percentages), the next 16 give the floats
       (draw >> 40) * 2^-23 - 1 in [-1, 1). */
    uint32_t compress_pct[5];
    uint64_t seed;
    /* TB_PATTERN_REPEAT: host array of repeat_len floats, repeated over the
       buffer (copied by the call; at most 4096 values). */
    const float *repeat;
    uint32_t repeat_len;
} tb_pattern;

/* Writes source pattern `pat` for SRC number bufferIdx into numBytes bytes of
   device memory at dst (slice 0 of a source: the allocation base plus
   byte_offset), with a kernel on `stream`, asynchronously.  numBytes must be
   a multiple of 4 and dst 4-byte aligned.  Default pattern:
   PrepSrcValue(bufferIdx, i) = (((i % 383) * 517) % 383 + 31) * (bufferIdx+1)
   as a float32. */
int tb_fill_source(tb_ctx *ctx, void *dst, uint64_t numBytes, const tb_pattern *pat,
                   int bufferIdx, tb_stream stream);

/* Host-to-device prep copy: for each k, copies numBytes bytes from hostSrcs[k]
   into slice 0 of srcs[k] (srcs[k] + byte_offset).  Synchronous.  Adds
   nSrc * numBytes to the context's prep-H2D counter. */
int tb_upload_sources(tb_ctx *ctx, void *const *srcs, const void *const *hostSrcs,
                      int nSrc, uint64_t numBytes);

/* Prep fill of PR #365: with slice 0 of every source already written, fills
   slices 1..K-1 from slice 0 device-to-device (by doubling, log2(K) copies,
   with the library's own copy kernel), K from tb_rotation_plan(numBytes,
   rotateBytes, byte_offset).  srcs[k] are allocation bases of at least
   allocBytes.  Synchronous.  Moves no host data. */
int tb_prepare_sources(tb_ctx *ctx, void *const *srcs, int nSrc, uint64_t numBytes,
                       uint64_t rotateBytes);

/* Bytes the context has copied host-to-device to prepare sources so far. */
uint64_t tb_prep_h2d_bytes(const tb_ctx *ctx);

/* ----------------------------------------------------------------------- */
/* Reduce-copy                                                              */
/* ----------------------------------------------------------------------- */

/* One reduce-copy launch on `stream`, asynchronous:
     nSrc == 0: every byte of dst[0 .. numBytes) = memset_byte;
     nSrc == 1: dst = srcs[0], bit for bit;
     nSrc >= 2: dst[i] = (...((srcs[0][i] + srcs[1][i]) + srcs[2][i]) ...)
                in float32, each add rounded to nearest even, no fused
                multiply-add, subnormals kept.
   srcs[k] and dst point at the data itself (no byte_offset or slice offset
   is added).  numBytes must be a multiple of 4, every pointer 4-byte aligned,
   nSrc <= TB_MAX_SRCS.  The elements are split into numSubExec contiguous
   ranges (sub-executors), each served by its own CTAs and sized in
   proportion to them (equal when numSubExec divides the grid);
   numSubExec == 0 is the library's choice: one per CTA, except one for the
   whole grid of the bulk form when ctas_per_subexec is 0.  The split does
   not change the result.  dst must not overlap any source (TB_EINVAL).  TB_ETIMEOUT, with
   nothing launched, when an earlier launch of this context stopped early
   because a bounded wait inside the kernel expired (kernel_wait_ns); the
   call after that one launches again. */
int tb_reduce_copy(tb_ctx *ctx, const void *const *srcs, int nSrc, void *dst,
                   uint64_t numBytes, int numSubExec, tb_stream stream);

/* The launch tb_reduce_copy makes for given arguments. */
typedef struct {
    int32_t engine;           /* 1 = vector loads, 2 = bulk copies via shared memory */
    int32_t vec_bytes;        /* bytes per vector access: 32, 16 or 4 */
    int32_t unroll;           /* vectors per source in flight per thread (engine 1) */
    int32_t block_threads;    /* threads per CTA */
    int32_t grid;             /* CTAs */
    int32_t num_subexec;      /* sub-executors */
    uint64_t head_elems;      /* scalar elements before the vector body */
    uint64_t body_vectors;    /* vectors of vec_bytes in the body */
    uint64_t tail_elems;      /* scalar elements after it */
    uint64_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t stages;           /* shared-memory pipeline stages (engine 2), else 0 */
    int32_t tile_bytes;       /* bytes per source of one tile (engine 2), else 0 */
} tb_launch_info;

/* Describes, without launching, the launch tb_reduce_copy would make for
   these arguments (same checks and errors). */
int tb_reduce_plan(tb_ctx *ctx, const void *const *srcs, int nSrc, const void *dst,
                   uint64_t numBytes, int numSubExec, tb_launch_info *out);

typedef struct {
    uint64_t K;               /* slices per source */
    uint64_t slice_stride;    /* bytes between slices */
    uint64_t alloc_bytes;     /* bytes each source allocation needs */
    uint64_t prep_h2d_bytes;  /* the context's prep-H2D counter */
    int32_t  iters;           /* timed iterations run */
    int32_t  num_subexec;     /* sub-executors used */
    int32_t  ctas;            /* CTAs per launch (0 on the DMA executor) */
    int32_t  block_threads;   /* threads per CTA */
    int32_t  gated;           /* 1 if the iterations ran behind the gate */
    int32_t  graphed;         /* 1 if the iterations ran as one CUDA graph */
    int32_t  engine;          /* reduce-copy engine used (see tb_launch_info); 0 on DMA */
    int32_t  validated;       /* 1 if dst was compared with expected bytes */
    double   total_ms;        /* device time of all timed iterations */
    double   mean_ms, median_ms, min_ms, max_ms;
    double   gbps;            /* (nSrc + 1) * numBytes * iters / total, 1e9 B/s */
    const float *iter_ms;     /* iters per-iteration times (owned by ctx,
                                 valid until the next tb_run_transfer) */
    int64_t  mismatch_index;  /* first bad element when validation failed, else -1 */
    uint32_t mismatch_expected, mismatch_actual;  /* its bits */
    int32_t  executor;        /* TB_EXEC_* the iterations ran on */
} tb_result;

typedef struct {
    void *const *srcs;        /* nSrc device allocation bases (>= alloc_bytes) */
    int32_t n_src;
    void *dst;                /* device allocation base (>= numBytes + byte_offset) */
    uint64_t num_bytes;       /* bytes per source slice and of dst */
    int32_t num_subexec;      /* 0 = auto */
    int32_t iters;            /* timed iterations, >= 1 */
    uint64_t rotate_bytes;    /* SRC_ROTATE_BYTES for this transfer */
    const void *expected;     /* NULL, or host bytes dst must equal (validation
                                 after the loop, or after every iteration when
                                 always_validate is set) */
    const void *expected_device; /* NULL, or device bytes dst must equal,
                                 compared on the GPU (tb_validate_device);
                                 used instead of `expected` when set */
    int32_t executor;         /* TB_EXEC_GPU (0) or TB_EXEC_DMA (1), below */
} tb_transfer;

/* Executors of a transfer (TransferBench PR #365, section "Technical
   Details": rotation applies to the GFX and DMA executors; the DMA one reads
   its source directly and rotates inline).
     TB_EXEC_GPU  the reduce-copy kernel (tb_reduce_copy's launch).
     TB_EXEC_DMA  the copy engines: iteration it is one cudaMemcpyAsync,
                  device to device, of numBytes from slice
                  tb_slice_for_iteration(it, K) of the one source to dst.
                  Exactly one source (TB_ENOTSUP otherwise); numSubExec,
                  the reduce-copy options and use_pdl do not apply. */
#define TB_EXEC_GPU 0
#define TB_EXEC_DMA 1

/* TransferBench's timed iteration loop for one transfer, synchronous on an
   internal stream: for it = -warmup .. iters-1, iteration it reads slice
   tb_slice_for_iteration(it, K) of every source (the slice offset is a kernel
   argument, or the copy's source address on the DMA executor, so rotation
   costs no host-to-device traffic and sits outside the timed region) and
   writes dst + byte_offset.  The loop runs as one
   CUDA graph timed by events around the timed iterations (use_graph), or as
   stream launches, behind the gate (use_gate) or not, with CUDA events
   between every two iterations.  Sources must already hold their slices
   (tb_fill_source or tb_upload_sources, then tb_prepare_sources), and
   nothing else may write them during the call: every launch after the
   first starts reading its sources while the launch before it finishes.
   On a validation failure returns TB_EVALIDATE with the mismatch in *out. */
int tb_run_transfer_ex(tb_ctx *ctx, const tb_transfer *t, tb_result *out);

/* tb_run_transfer_ex without expected bytes. */
int tb_run_transfer(tb_ctx *ctx, void *const *srcs, int nSrc, void *dst,
                    uint64_t numBytes, int numSubExec, int iters, uint64_t rotateBytes,
                    tb_result *out);

/* The transfer with host buffers, end to end, asynchronous on `stream`
   (ordered after the caller's earlier work on it): hostDst = the reduce-copy
   of hostSrcs, numBytes each.
   - When every host buffer is page-locked and mapped into the device's
     address space (cudaHostAlloc, or cudaHostRegister with mapping), one
     reduce-copy kernel reads the sources and writes hostDst across the host
     link directly; devSrcs / devDst are not used and may be NULL.
   - Otherwise the bytes are staged through the caller's device buffers
     devSrcs[k] / devDst (numBytes each) in 32 MiB chunks: host-to-device
     copies, the kernel and the device-to-host copy of successive chunks run
     on three internal streams and overlap.  Pageable host memory makes the
     copies synchronous with the host. */
int tb_reduce_copy_host(tb_ctx *ctx, const void *const *hostSrcs, int nSrc, void *hostDst,
                        uint64_t numBytes, void *const *devSrcs, void *devDst,
                        int numSubExec, tb_stream stream);

/* ----------------------------------------------------------------------- */
/* Batched copy                                                             */
/* ----------------------------------------------------------------------- */

typedef struct {
    uint64_t src;  /* device address of the first source byte */
    uint64_t dst;  /* device address of the first destination byte */
    uint64_t len;  /* bytes; 0 is a no-op */
} tb_copy_desc;

/* Copies every descriptor's len bytes from src to dst, byte-exact, any
   alignment, with one kernel launch per descriptor slot, asynchronously on
   `stream` (ordered after the caller's earlier work on it).  The descriptor
   array is read and packed before return, so the caller may reuse it at
   once.  The packed work list goes to the device on an internal stream,
   overlapping earlier work, and the kernel waits for it on `stream`; a small
   batch of short copies only has its list read in place from pinned host
   memory.  The kernel runs at the priority of `stream`: on a high-priority
   stream its CTAs are scheduled ahead of waiting work of lower-priority
   streams, such as a GEMM loop.  The bytes of all descriptors longer than
   small_max_bytes form one stream cut into equal chunks, the same number
   for every CTA, moved with bulk copies through shared memory; descriptors
   of at most small_max_bytes go to a warp each, streamed through that
   warp's ring of shared-memory slots by asynchronous 16-byte copies, the
   first ones fixed by warp index and the rest claimed four at a time by free
   warps from a counter in the packed work list.  A launch of short copies
   only runs a kernel without the long-copy path, in the ring shape that
   batch_short_shape selects; batch_max_ctas caps the CTAs of any launch.
   Addresses may also be
   pinned host memory mapped into the device's address space.  Destinations
   must not overlap one another or any source of the batch (the order of
   copies is unspecified).  TB_EINVAL for a null
   address with len > 0 or an address range that wraps; TB_ETIMEOUT if no
   slot came free within wait_timeout_ns, or when the previous batch that
   used the chosen slot stopped early because a bounded wait inside the
   kernel (2 s per wait) expired (a batch of more than slot_items
   descriptors is launched one slot at a time, so when the wait for a later
   slot fails the launches before it stay queued and copy their part);
   TB_ENOTSUP, with nothing queued, while
   `stream` is capturing a CUDA graph (the packed work list lives in the
   context's staging, which later calls reuse, so a replayed graph would
   read another batch's list). */
int tb_batch_copy(tb_ctx *ctx, const tb_copy_desc *desc, size_t n, tb_stream stream);

typedef struct {
    uint64_t descs;        /* descriptors with len > 0 */
    uint64_t warp_items;   /* descriptors copied by one warp */
    uint64_t cta_items;    /* pieces of long descriptors copied by whole CTAs */
    uint64_t launches;     /* kernel launches (slots) used */
    uint64_t bytes;        /* sum of len */
    uint64_t upload_bytes; /* bytes of the packed work lists the kernels read */
    uint64_t ce_copies;    /* descriptors sent to the copy engines (ce_min_bytes) */
    uint64_t direct_launches; /* launches that read their work list in place from
                                 pinned host memory (small batches of short copies
                                 only: no upload, no event) */
} tb_batch_stats;

/* Statistics of the last tb_batch_copy on ctx. */
int tb_last_batch_stats(const tb_ctx *ctx, tb_batch_stats *out);

/* Device time, in milliseconds, of the kernel launches of the last
   tb_batch_copy (summed over its launches).  Waits for them to finish.
   TB_ENOTSUP unless the context was created with time_kernels = 1. */
int tb_last_batch_kernel_ms(tb_ctx *ctx, double *ms);

/* The per-copy baseline of the HipTransport RFC (section "Motivation": each
   request there costs one memcpy call): one cudaMemcpyAsync (device to device) per
   descriptor with len > 0, in array order, on `stream`.  Same arguments and
   checks as tb_batch_copy; provided so the two can be timed side by side. */
int tb_copy_each(tb_ctx *ctx, const tb_copy_desc *desc, size_t n, tb_stream stream);

/* Non-empty descriptors one tb_batch_copy_noalloc call can take. */
#define TB_NOALLOC_MAX_ITEMS 65536

/* The batched copy without any allocation.  The pages have no counterpart:
   it exists for callers that cannot call cudaMalloc - a serving engine that
   has handed all free HBM to its own allocator (a KV cache reserved up
   front) has nothing left for one, and a latency-sensitive loop cannot
   afford cudaMalloc / cudaFree, which may synchronize the whole device.
   Same copy semantics and scheduling as tb_batch_copy with default options
   (copies up to 16 KiB go to one warp each), on the current CUDA device,
   asynchronously on `stream`; no context is needed.
   Memory: the packed work items live in a fixed __device__ array of
   2,162,736 bytes (about 2.06 MiB: room for the work items, stream prefix
   and chunk table of TB_NOALLOC_MAX_ITEMS descriptors) that every GPU
   loading this library holds until the process exits.  The status words
   below sit in one 4 KiB page of the library's static host memory.
   Set-up: the first call on a device that has something to copy looks up
   that array's device address (with that device current), reads the wait
   limit of the long copies' bulk pipeline (environment variable
   TB_KERNEL_WAIT_NS, else 2 s) and, on the first device only, page-locks
   and maps the status page (cudaHostRegister of the library's own page);
   make that first call before any stream capture.
   Sharing: every call on a device uses the one array and leaves the last
   batch's items in it: calls whose work overlaps on the GPU (different
   streams, no ordering between them) race; calls on one stream run in
   order.  Host-side packing is serialized by a lock.
   Expired waits: when a bounded wait inside a kernel runs out, that kernel
   stops its long copies early and sets the device's status word.  The
   first call on the device that starts after that kernel has finished
   returns TB_ETIMEOUT, clears the word and enqueues nothing.  To learn
   whether a given batch completed, synchronize its stream and then call
   with n == 0, which copies nothing and only reports (and clears) the word.
   Errors: TB_EINVAL for a null or wrapping range, or on the first call on
   a device when TB_KERNEL_WAIT_NS does not parse; TB_ENOTSUP when the batch
   has more than TB_NOALLOC_MAX_ITEMS descriptors with len > 0, or when
   `stream` is capturing work into a graph (the work list is copied from a
   host array that the next call rewrites); TB_ETIMEOUT as above; TB_ECUDA
   when a CUDA call fails.  Nothing is copied after an error.  It calls no
   cudaMalloc, cudaFree or other allocating routine. */
int tb_batch_copy_noalloc(const tb_copy_desc *desc, size_t n, tb_stream stream);

/* ----------------------------------------------------------------------- */
/* Validation ("How validation (ValidateAllTransfers) works")               */
/* ----------------------------------------------------------------------- */

typedef struct {
    int64_t  index;     /* first differing element, -1 if none */
    uint32_t expected;  /* its expected bits (elemSize bytes, zero-extended) */
    uint32_t actual;    /* its actual bits */
} tb_mismatch;

/* Copies numBytes of device memory at dstDevice to the host (in bounded
   chunks through pinned staging) and compares it with expectedHost by
   memcmp; elemSize (1, 2 or 4) sets the unit of the reported index.
   Synchronous.  Returns TB_OK when equal, TB_EVALIDATE with *out filled at
   the first difference otherwise.  out may be NULL. */
int tb_validate(tb_ctx *ctx, const void *dstDevice, const void *expectedHost,
                uint64_t numBytes, uint32_t elemSize, tb_mismatch *out);

/* The validateDirect option of "TransferBench data validation" (which the
   page gives for AMD only, with NVIDIA falling back to a host copy): compares
   numBytes of dstDevice with expectedDevice on the GPU, without copying
   either to the host, and reports the first differing element (elemSize
   1, 2 or 4 bytes).  Synchronous; first waits for work already queued on
   the device.  TB_OK when equal, TB_EVALIDATE with *out filled otherwise. */
int tb_validate_device(tb_ctx *ctx, const void *dstDevice, const void *expectedDevice,
                       uint64_t numBytes, uint32_t elemSize, tb_mismatch *out);

#ifdef __cplusplus
}
#endif

#endif /* TB_H */

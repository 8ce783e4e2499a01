#!/usr/bin/env python3
"""Benchmark of the reduce-copy and batched-copy engine on GB300.

Default line (rank 0 prints one JSON object):
  workload  3-source reduce-copy, 3 x 67,108,864 float32 (256 MiB each),
            src_k = PrepSrcValue(k, i), SRC_ROTATE_BYTES = 256 MiB (K = 1);
  step      one reduce-copy launch over the whole transfer (1 GiB moved:
            3 x 256 MiB read + 256 MiB written); inputs (1 GiB) exceed the
            129 MB L2, so no flush is needed between steps; the K timed
            steps are captured into one CUDA graph and replayed once;
  value     HBM GB/s counting read + write bytes, summed over ranks;
  e2e       the same transfer through tb_reduce_copy_host from pinned host
            buffers: host-to-device sources, the kernel, device-to-host dst;
  batch     the 47,540-descriptor batch (47,520 head-sliced pages of
            64 B-16 KiB + 16 x 16 MiB + 4 x 8 MiB) through tb_batch_copy,
            with one cudaMemcpyAsync per copy (tb_copy_each) timed beside it;
  single_4mib_k64, dma_executor_256mib, rotation_sweep, index_pages_3840,
  block_pages_7200, interference, multi_source_fill_compress,
  validation_256mib
            the other configured workloads, a few seconds in all (leave
            them out with --no-extra): the 4 MiB K = 64 transfer on the
            kernel and on the copy engines, the DMA executor at 256 MiB,
            the fillCompress sweep 8-512 MiB with rotation on and off, the
            3840- and 7200-page batches, a bf16 GEMM beside the batches,
            2-8 fillCompress sources, and validation on the device against
            the host;
  roofline  achieved algorithmic GB/s of the reduce kernel against the
            measured HBM copy bandwidth (MEASURED_PEAKS.json);
  cpu_baseline  the CPU oracle on a bounded sample, one host core.

``--impl reference`` times the CPU oracle itself (the reference arm of this
benchmark) on the same metric.  Under torchrun every rank runs its own
replica on its own GPU (no data exchange); timings are the max over ranks.
``--study`` prints extra lines instead of the default line: the single
4 MiB transfer (graph with and without programmatic dependent launch,
events per launch), the fillCompress sweep with rotation on and off (cold,
warm, graphed), validation on the device against the host, end to end from
pinned and pageable host memory, tiny batches against per-copy memcpy,
small copies under a GEMM loop (normal and high-priority stream), the three
batch workloads, the batch's long and short parts, copy-engine routing, GEMM
interference, and GEMM interference with the batch kernel's grid capped.
``--profile reduce|batch|batch-short|batch-small|rotation`` runs one
workload for an ncu capture (commands in ``profiles/``).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MiB = 1 << 20
GiB = 1 << 30
METRIC = ("HBM GB/s (read+write) and % of GB300 HBM peak; copies/s for batched small copies")
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("3-source reduce-copy: 3 x 67,108,864 float32 (256 MiB each), src_k = "
            "PrepSrcValue(k, i), k = 0..2, dst = src0 + src1 + src2 left to right in fp32, "
            "SRC_ROTATE_BYTES = 256 MiB (K = 1)")


# ---------------------------------------------------------------------------
# Process group (torchrun) and timing helpers
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Ranks:
    """Barrier and max/sum over ranks; a no-op for one process."""

    def __init__(self, world: int, backend: str):
        self.world = world
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.dist = dist
            self.backend = backend

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def reduce(self, value: float, op: str) -> float:
        if not self.dist:
            return value
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([value], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=getattr(self.dist.ReduceOp, op))
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()


def combine(ranks: Ranks, units: float, seconds: float):
    """Whole-job throughput: units summed over ranks / the slowest rank's time."""
    total_units = ranks.reduce(units, "SUM")
    worst = ranks.reduce(seconds, "MAX")
    return total_units, worst


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def ctx_options(tb, **fields):
    """Context options: defaults, the given fields, then TB_* environment
    overrides (e.g. TB_USE_GATE=0 under a profiler)."""
    return tb.options_from_env(tb.options(**fields))


def kernel_source_sha(source: str) -> str:
    """SHA-256 of a kernel's source file together with the shared device
    header, so a recorded ncu figure goes stale when either changes."""
    h = hashlib.sha256()
    for name in (source, "tb_device.cuh"):
        with open(os.path.join(ROOT, "copy_reduce_dst_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(key: str):
    """Per-launch DRAM bytes (read + write) from the committed ncu summary,
    or None when the kernel's source changed after the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            entry = json.load(f)[key]
    except (OSError, KeyError, ValueError):
        return None
    try:
        if entry.get("kernel_source_sha256") != kernel_source_sha(entry["source"]):
            return None
    except (OSError, KeyError):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            self.out = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and time.time() - t0 < timeout:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# Reduce-copy (default line)
# ---------------------------------------------------------------------------
def run_reduce(args, tb, torch, ranks, local):
    nb = 256 * MiB
    n_src = 3
    rotate = 256 * MiB
    plan = tb.rotation_plan(nb, rotate)
    # early_reads: each timed step may read its sources before the step ahead
    # has finished, as TransferBench's loop inside tb_run_transfer does; no
    # step writes a source (the steps write dst only).
    ctx = tb.Context(local, ctx_options(tb, early_reads=1))
    stream = torch.cuda.current_stream()
    srcs = [torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda") for _ in range(n_src)]
    for k, s in enumerate(srcs):
        ctx.fill_source(s, nb, tb.default_pattern(), k, stream)
    ctx.prepare_sources(srcs, nb, rotate)
    dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
    bytes_per_step = (n_src + 1) * nb

    # Sub-executor sweep with the library's own per-iteration events
    # (TransferBench's loop: 3 warm-up + 20 timed iterations each).
    sweep = {}
    peak0 = read_peaks()[0]
    for se in (1, 4, 16, 32):
        r = ctx.run_transfer(srcs, dst, nb, num_subexec=se, iters=20, rotate_bytes=rotate)
        sweep[str(se)] = {"gbps": round(r["gbps"], 1), "ctas": r["ctas"],
                          "median_ms": round(r["median_ms"], 4),
                          "pct_of_peak": round(r["gbps"] / peak0 * 100, 1)}
    # The timed loop runs at the best sub-executor count of the sweep (every
    # count is reported in the line's config).
    subexec = max(sweep, key=lambda k: sweep[k]["gbps"])
    subexec = int(subexec)
    info = ctx.reduce_plan(srcs, dst, nb, subexec)
    kernel = (f"k_reduce_bulk<{n_src}, {info['tile_bytes']}> (bulk copies through shared memory, "
              f"{info['stages']} stages of {info['tile_bytes'] // 1024} KiB per source)"
              if info["engine"] == 2
              else f"k_reduce<{n_src}, {info['vec_bytes']}, {info['unroll']}> (vector loads)")
    # TransferBench's literal layout, one CTA per sub-executor (1 warm-up and
    # 3 timed iterations: a lone CTA's rate hardly varies, and at 1 GiB per
    # launch one CTA takes ~15 ms).
    strict = {}
    with tb.Context(local, ctx_options(tb, ctas_per_subexec=1, warmup=1)) as c1:
        for se in (1, 4, 16, 32):
            r = c1.run_transfer(srcs, dst, nb, num_subexec=se, iters=3, rotate_bytes=rotate)
            strict[str(se)] = {"gbps": round(r["gbps"], 1), "ctas": r["ctas"],
                               "pct_of_peak": round(r["gbps"] / peak0 * 100, 1)}

    def srcs_at(step):
        off = tb.slice_for_iteration(step, plan.K) * plan.slice_stride
        return [s.data_ptr() + off for s in srcs]

    def step(i, s=stream):
        ctx.reduce_copy(srcs_at(i), dst, nb, subexec, s)

    for i in range(-args.warmup, 0):
        step(i)
    # The K timed steps are captured into one CUDA graph (each step one
    # reduce-copy launch over the whole transfer, its rotated slice baked in)
    # and replayed once in the timed region: no launch gaps between steps.
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    gstream = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=gstream):
        for i in range(args.steps):
            step(i, gstream)
    with torch.cuda.stream(gstream):
        graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.wait_first()
    # Untimed soak so the clock samples cover a steady load, then the timed loop.
    t_end = time.time() + 0.5
    i = 0
    while time.time() < t_end:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    ranks.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gstream):
        torch.cuda.nvtx.range_push("timed")   # the launch list of the timed region: ncu --nvtx
        ev0.record(gstream)
        graph.replay()
        ev1.record(gstream)
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    ranks.barrier()
    clocks = sampler.stop()
    del graph
    ms = ev0.elapsed_time(ev1)
    units, worst_s = combine(ranks, bytes_per_step * args.steps, ms / 1e3)
    value = units / worst_s / 1e9
    per_launch_s = (ms / 1e3) / args.steps
    achieved = bytes_per_step / per_launch_s / 1e9
    peak, peak_kind = read_peaks()

    # End to end from pinned host memory (public API: tb_reduce_copy_host).
    hsrc = [torch.empty(nb, dtype=torch.uint8).pin_memory() for _ in range(n_src)]
    for h, s in zip(hsrc, srcs):
        h.copy_(s[:nb].cpu())
    hdst = torch.empty(nb, dtype=torch.uint8).pin_memory()
    dsrc = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(n_src)]
    for i in range(args.warmup):
        ctx.reduce_copy_host(hsrc, hdst, nb, dsrc, dst, subexec, stream)
    e_steps = max(1, min(args.steps, 10))
    torch.cuda.synchronize()
    ranks.barrier()
    t0 = time.perf_counter()
    ev0.record(stream)
    for i in range(e_steps):
        ctx.reduce_copy_host(hsrc, hdst, nb, dsrc, dst, subexec, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ranks.barrier()
    e_ms = ev0.elapsed_time(ev1)
    e_units, e_worst = combine(ranks, bytes_per_step * e_steps, max(e_ms / 1e3, wall))
    e2e = {"value": round(e_units / e_worst / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": n_src * nb, "d2h_bytes_per_step": nb,
           "api": "tb_reduce_copy_host", "steps": e_steps}
    ctx.close()
    del srcs, dsrc, hsrc, hdst
    torch.cuda.empty_cache()

    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": profiled_traffic("reduce_3src_256MiB"),
                "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": bytes_per_step,
                "kernel": kernel, "grid": info["grid"], "block_threads": info["block_threads"]}
    result = {"value": value, "ms_per_step": ms / args.steps, "roofline": roofline, "e2e": e2e,
              "clocks": clocks, "gpu_launches": args.steps,
              "subexec_sweep": sweep, "strict_one_cta_per_subexec": strict,
              "subexec": subexec}
    return result


# ---------------------------------------------------------------------------
# Batched copy (47,540 descriptors)
# ---------------------------------------------------------------------------
def run_batch(args, tb, torch, ranks, local):
    from copy_reduce_dst_gb300 import workloads
    layout = workloads.batch_head_sliced()
    src = device_random_bytes(torch, layout.src_pool_bytes, 41)
    dst = device_random_bytes(torch, layout.dst_pool_bytes, 42)
    desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
    stream = torch.cuda.current_stream()
    ctx = tb.Context(local, ctx_options(tb, time_kernels=1))
    n = layout.n
    payload = 2 * layout.total_bytes

    for _ in range(args.warmup):
        ctx.batch_copy(desc, stream)
    torch.cuda.synchronize()
    # device time of back-to-back calls (descriptor upload + kernel)
    ranks.barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record(stream)
    for _ in range(args.steps):
        ctx.batch_copy(desc, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall_total = time.perf_counter() - t0
    ranks.barrier()
    dev_ms = ev0.elapsed_time(ev1) / args.steps
    stats = ctx.last_batch_stats()
    # kernel-only device time and per-call wall time (pack + upload + kernel + sync)
    kern, walls = [], []
    for _ in range(max(3, min(args.steps, 10))):
        t0 = time.perf_counter()
        ctx.batch_copy(desc, stream)
        stream.synchronize()
        walls.append(time.perf_counter() - t0)
        kern.append(ctx.last_batch_kernel_ms())
    kernel_ms = statistics.median(kern)
    wall_ms = statistics.median(walls) * 1e3
    # one cudaMemcpyAsync per copy, timed the same way
    each = []
    for _ in range(2):
        t0 = time.perf_counter()
        ctx.copy_each(desc, stream)
        stream.synchronize()
        each.append(time.perf_counter() - t0)
    each_ms = min(each) * 1e3
    ctx.close()
    del src, dst
    torch.cuda.empty_cache()
    peak, peak_kind = read_peaks()
    algo = payload + stats["upload_bytes"]  # the kernel also reads each work item once
    units, worst = combine(ranks, n * args.steps, wall_total)
    return {
        "workload": layout.name + " (uint8 random from seed, two 2 GiB pools, seeded layout)",
        "descriptors": n, "bytes_copied": layout.total_bytes,
        "copies_per_s": round(units / worst, 1),
        "gbps_rw_device": round(payload / (dev_ms / 1e3) / 1e9, 1),
        "device_ms_per_batch": round(dev_ms, 4),
        "kernel_ms": round(kernel_ms, 4),
        "wall_ms_per_batch": round(wall_ms, 4),
        "memcpy_each_wall_ms": round(each_ms, 3),
        "speedup_vs_memcpy_each": round(each_ms / wall_ms, 1),
        "work_items": {"warp": stats["warp_items"], "cta": stats["cta_items"],
                       "launches": stats["launches"], "upload_bytes": stats["upload_bytes"]},
        "roofline": {"bound": "hbm", "achieved": round(algo / (kernel_ms / 1e3) / 1e9, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(algo / (kernel_ms / 1e3) / 1e9 / peak, 4),
                     "traffic": profiled_traffic("batch_head_sliced"),
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": algo,
                     "kernel": "k_batch<2, 4>"},
    }


def device_random_bytes(torch, n: int, seed: int):
    """A seeded uniform uint8 pool written on the device (input preparation,
    outside every timed region)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)


# ---------------------------------------------------------------------------
# The other workloads, bounded to a few seconds each, on the default line
# ---------------------------------------------------------------------------
def run_single_transfer(tb, torch, local):
    """The single 4 MiB transfer: 1 source of 1,048,576 float32 =
    PrepSrcValue(0, i), uploaded from the host into slice 0 (prep H2D 4 MiB),
    slices 1..63 filled on the device; SRC_ROTATE_BYTES 256 MiB, so K = 64 and
    a 268,435,456 B allocation; 3 warm-up + 10 timed iterations, dst validated
    against src0 on the device.  Median (and mean) of 15 runs, on the
    reduce-copy kernel (one CUDA graph) and on the copy engines (DMA
    executor): the event timer steps by 1-2 us on a ~25 us span, so one run
    says little; a full rotation of 64 iterations (median of 5) beside it,
    and the same 64-iteration loop on a 4 KiB transfer, which costs what the
    chain of dependent launches costs by itself."""
    nb, rot = 4 * MiB, 256 * MiB
    plan = tb.rotation_plan(nb, rot)
    with tb.Context(local, ctx_options(tb)) as ctx:
        src = torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda")
        ctx.fill_source(src, nb, tb.default_pattern(), 0)
        host = src[:nb].cpu().pin_memory()
        src.zero_()
        ctx.upload_sources([src], [host], nb)
        ctx.prepare_sources([src], nb, rot)
        dst = torch.zeros(nb, dtype=torch.uint8, device="cuda")

        def med(iters, executor, runs=15):
            rs = [ctx.run_transfer([src], dst, nb, iters=iters, rotate_bytes=rot,
                                   expected_device=src, executor=executor) for _ in range(runs)]
            rs.sort(key=lambda r: r["gbps"])
            r = dict(rs[len(rs) // 2])
            r["mean_us"] = statistics.mean(x["mean_ms"] for x in rs) * 1e3
            return r
        k1, k1_64 = med(10, tb.TB_EXEC_GPU), med(64, tb.TB_EXEC_GPU, 5)
        dma = med(10, tb.TB_EXEC_DMA)
        # The loop's own floor: a 4 KiB transfer through the same loop (its
        # K = 65,536 slices of 4 KiB fill the same 268,435,456 B allocation).
        floor = sorted(ctx.run_transfer([src], dst, 4096, iters=64, rotate_bytes=rot)["mean_ms"]
                       for _ in range(5))[2]
        out = {"workload": "1 source, 1,048,576 float32 = PrepSrcValue(0, i), SRC_ROTATE_BYTES "
                           "256 MiB, 3 warm-up + 10 timed iterations, dst == src0",
               "K": k1["K"], "alloc_bytes": k1["alloc_bytes"],
               "prep_h2d_bytes": k1["prep_h2d_bytes"], "validated": bool(k1["validated"]),
               "gbps": round(k1["gbps"], 1), "us_per_iteration": round(k1["mean_ms"] * 1e3, 3),
               "pct_of_peak": round(k1["gbps"] / read_peaks()[0] * 100, 1),
               "us_per_iteration_mean_of_runs": round(k1["mean_us"], 3),
               "graphed": bool(k1["graphed"]), "ctas": k1["ctas"],
               "gbps_64_iterations": round(k1_64["gbps"], 1),
               "us_per_iteration_64": round(k1_64["mean_ms"] * 1e3, 3),
               "floor_us_per_iteration_4kib_64": round(floor * 1e3, 3),
               "dma_gbps": round(dma["gbps"], 1),
               "dma_us_per_iteration": round(dma["mean_ms"] * 1e3, 3),
               "dma_us_per_iteration_mean_of_runs": round(dma["mean_us"], 3),
               "dma_validated": bool(dma["validated"])}
        del src, dst, host
    return out


def run_dma_large(tb, torch, local):
    """The copy-engine (DMA) executor beside the reduce-copy kernel on one
    256 MiB source (K = 1): 3 warm-up + 20 timed iterations, median of 3."""
    nb = 256 * MiB
    with tb.Context(local, ctx_options(tb)) as ctx:
        src = torch.empty(nb, dtype=torch.uint8, device="cuda")
        ctx.fill_source(src, nb, tb.default_pattern(), 0)
        dst = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        res = {}
        for name, ex in (("kernel", tb.TB_EXEC_GPU), ("dma", tb.TB_EXEC_DMA)):
            runs = [ctx.run_transfer([src], dst, nb, iters=20, rotate_bytes=256 * MiB,
                                     expected_device=src, executor=ex) for _ in range(3)]
            r = sorted(runs, key=lambda r: r["gbps"])[1]
            res[name + "_gbps"] = round(r["gbps"], 1)
            res[name + "_us_per_iteration"] = round(r["mean_ms"] * 1e3, 2)
        del src, dst
    res["workload"] = "1 source of 256 MiB (67,108,864 float32), K = 1, 20 iterations, dst == src0"
    return res


def run_rotation_sweep(tb, torch, local):
    """fillCompress sweep: 1 source, 8-512 MiB, 40% random / 20% 1B0 / 0% 2B0 /
    20% 4B0 / 20% 32B0 per 64-byte line (seed 0x5EED), rotation at 256 MiB
    and off.  cold = mean of 5 single iterations each after writing a 512 MiB
    buffer (> L2); warm = 20 iterations after 3 warm-ups with events around
    every launch; warm_graph = the same 20 as one CUDA graph; median of 3."""
    import statistics as st
    flush = torch.empty(512 * MiB, dtype=torch.uint8, device="cuda")
    pct = (40, 20, 0, 20, 20)
    rows = []
    with tb.Context(local, ctx_options(tb)) as ctx, \
            tb.Context(local, ctx_options(tb, use_graph=0)) as ev_ctx, \
            tb.Context(local, ctx_options(tb, warmup=0, use_graph=0)) as cold_ctx:
        for mib in (8, 16, 32, 64, 128, 256, 512):
            nb = mib * MiB
            row = {"MiB": mib}
            for rot in (256 * MiB, 0):
                plan = tb.rotation_plan(nb, rot)
                src = torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda")
                ctx.fill_source(src, nb, tb.compress_pattern(pct, 0x5EED), 0)
                ctx.prepare_sources([src], nb, rot)
                dst = torch.zeros(nb, dtype=torch.uint8, device="cuda")
                cold, warm, graph = [], [], []
                for rep in range(3):
                    c = []
                    for _ in range(5):
                        flush.fill_(rep)
                        c.append(cold_ctx.run_transfer([src], dst, nb, iters=1,
                                                       rotate_bytes=rot)["total_ms"])
                    cold.append(2 * nb / (st.mean(c) / 1e3) / 1e9)
                    warm.append(ev_ctx.run_transfer([src], dst, nb, iters=20,
                                                    rotate_bytes=rot)["gbps"])
                    graph.append(ctx.run_transfer([src], dst, nb, iters=20,
                                                  rotate_bytes=rot)["gbps"])
                tag = "on" if rot else "off"
                row[tag] = {"K": plan.K, "cold_gbps": round(st.median(cold), 1),
                            "warm_gbps": round(st.median(warm), 1),
                            "w_over_c": round(st.median(warm) / st.median(cold), 3),
                            "warm_graph_gbps": round(st.median(graph), 1)}
                del src, dst
            rows.append(row)
    del flush
    torch.cuda.empty_cache()
    return rows


def run_multi_source_compress(tb, torch, local):
    """Multi-source fillCompress reduce-copies (2, 4 and 8 sources of 64 MiB,
    40/20/0/20/20 %, seed 0x5EED + k, rotation at 256 MiB, so K = 4 and every
    iteration reads its sources from HBM): random floats with zeroed bytes,
    so the adds meet subnormals and the order of the adds decides the bits
    (bit-exactness is tested against the oracle).  GB/s (read + write) of 20
    graphed iterations, median of 3, and the engine."""
    import statistics as st
    nb, rot = 64 * MiB, 256 * MiB
    plan = tb.rotation_plan(nb, rot)
    pct = (40, 20, 0, 20, 20)
    rows = []
    with tb.Context(local, ctx_options(tb)) as ctx:
        srcs = [torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda") for _ in range(8)]
        for k, s_ in enumerate(srcs):
            ctx.fill_source(s_, nb, tb.compress_pattern(pct, 0x5EED), k)
        ctx.prepare_sources(srcs, nb, rot)
        dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
        for n in (2, 4, 8):
            runs = [ctx.run_transfer(srcs[:n], dst, nb, iters=20, rotate_bytes=rot)
                    for _ in range(3)]
            rows.append({"sources": n, "MiB_each": 64, "K": runs[0]["K"],
                         "gbps": round(st.median(r["gbps"] for r in runs), 1),
                         "engine": runs[0]["engine"], "ctas": runs[0]["ctas"]})
        del srcs, dst
    torch.cuda.empty_cache()
    return rows


def run_small_batch(tb, torch, local, make_layout, seed, variants):
    """One of the Mooncake RFC's small-copy shapes on seeded random pools.
    A single batch of this shape touches less than the 129 MB L2, so the
    calls cycle through `variants` layouts of the same shape (seeds seed,
    seed + 1, ...; sources in separate regions when the source pool is
    small), whose bytes together exceed L2: no call finds its data there.
    kernel_us = kernel-only events (median of 40); device_us = events around
    back-to-back calls (two passes over the variants); wall_us = one call
    with packing, upload, kernel and stream sync (median of 40);
    memcpy_each = one cudaMemcpyAsync per copy, wall-timed the same way
    (best of 2, the first layout)."""
    import statistics as st
    layouts = [make_layout(seed + r) for r in range(variants)]
    lay0 = layouts[0]
    own_src = lay0.src_pool_bytes * variants <= 1 << 30
    src = device_random_bytes(torch, lay0.src_pool_bytes * (variants if own_src else 1), seed)
    dst = device_random_bytes(torch, lay0.dst_pool_bytes, seed + 1000)
    descs = [lay.descriptors(src.data_ptr() + (r * lay0.src_pool_bytes if own_src else 0),
                             dst.data_ptr()) for r, lay in enumerate(layouts)]
    touched = sum(2 * int(lay.total_bytes) for lay in layouts)
    stream = torch.cuda.Stream()
    moved = 2 * int(lay0.total_bytes)
    with tb.Context(local, ctx_options(tb, time_kernels=1)) as kctx, \
            tb.Context(local, ctx_options(tb)) as ctx:
        for d in descs:
            kctx.batch_copy(d, stream)
        kern = []
        for i in range(40):
            kctx.batch_copy(descs[i % variants], stream)
            kern.append(kctx.last_batch_kernel_ms())
        for d in descs:
            ctx.batch_copy(d, stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        calls = 2 * variants
        stream.synchronize()
        a.record(stream)
        for i in range(calls):
            ctx.batch_copy(descs[i % variants], stream)
        b.record(stream)
        b.synchronize()
        dev_ms = a.elapsed_time(b) / calls
        walls = []
        for i in range(40):
            t0 = time.perf_counter()
            ctx.batch_copy(descs[i % variants], stream)
            stream.synchronize()
            walls.append(time.perf_counter() - t0)
        each = []
        for _ in range(2):
            t0 = time.perf_counter()
            ctx.copy_each(descs[0], stream)
            stream.synchronize()
            each.append(time.perf_counter() - t0)
        stats = kctx.last_batch_stats()
    k_ms = st.median(kern)
    wall = st.median(walls)
    del src, dst
    return {"workload": lay0.name + " (uint8 random from seed)", "descriptors": lay0.n,
            "bytes_copied": int(lay0.total_bytes),
            "variants": variants, "bytes_touched_per_cycle": touched,
            "kernel_us": round(k_ms * 1e3, 2),
            "kernel_gbps": round(moved / (k_ms / 1e3) / 1e9, 1),
            "device_us": round(dev_ms * 1e3, 2),
            "device_gbps": round(moved / (dev_ms / 1e3) / 1e9, 1),
            "copies_per_s_device": round(lay0.n / (dev_ms / 1e3), 1),
            "wall_us": round(wall * 1e6, 1), "copies_per_s_wall": round(lay0.n / wall, 1),
            "memcpy_each_wall_ms": round(min(each) * 1e3, 3),
            "speedup_vs_memcpy_each": round(min(each) / wall, 1),
            "direct_launches": stats["direct_launches"]}


def run_interference(tb, torch, local):
    """A bf16 GEMM (4096^3 torch.matmul) looping on one stream for ~0.4 s, alone
    and while the 47,540 batch is copied back to back on another stream (the
    Mooncake RFC's interference measurement); and the 3840-page batch's wall
    time per call on an idle GPU and under the GEMM loop, on a normal- and a
    high-priority stream."""
    import statistics as st
    from copy_reduce_dst_gb300 import workloads
    n = 4096
    a = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    b = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    flops = 2 * n ** 3
    gemm_s = torch.cuda.Stream()
    copy_s = torch.cuda.Stream()
    hi_s = torch.cuda.Stream(priority=-1)
    reps = 2400  # ~0.4 s of 4096^3 GEMMs

    def gemm_loop():
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(gemm_s)
        with torch.cuda.stream(gemm_s):
            for _ in range(reps):
                torch.matmul(a, b)
        e1.record(gemm_s)
        return e0, e1

    big = workloads.batch_head_sliced()
    src = device_random_bytes(torch, big.src_pool_bytes, 51)
    dst = device_random_bytes(torch, big.dst_pool_bytes, 52)
    desc = big.descriptors(src.data_ptr(), dst.data_ptr())
    out = {}
    with tb.Context(local, ctx_options(tb)) as ctx:
        with torch.cuda.stream(gemm_s):
            for _ in range(20):
                torch.matmul(a, b)
        torch.cuda.synchronize()
        e0, e1 = gemm_loop()
        torch.cuda.synchronize()
        alone = reps * flops / (e0.elapsed_time(e1) / 1e3) / 1e12
        e0, e1 = gemm_loop()
        batches, t0 = 0, time.perf_counter()
        while not e1.query():
            ctx.batch_copy(desc, copy_s)
            copy_s.synchronize()
            batches += 1
        wall = time.perf_counter() - t0
        torch.cuda.synchronize()
        shared = reps * flops / (e0.elapsed_time(e1) / 1e3) / 1e12
        gbps = 2 * big.total_bytes * batches / wall / 1e9
        out.update({"gemm": "4096^3 bf16 torch.matmul", "gemm_tflops_alone": round(alone, 1),
                    "gemm_tflops_with_batch": round(shared, 1), "batch_gbps": round(gbps, 1),
                    "gemm_loss_pct": round(100 * (1 - shared / alone), 2),
                    "batch": big.name + " back to back"})
        del src, dst
        small = workloads.batch_index_pages()
        src = device_random_bytes(torch, small.src_pool_bytes, 53)
        dst = device_random_bytes(torch, small.dst_pool_bytes, 54)
        desc = small.descriptors(src.data_ptr(), dst.data_ptr())
        for name, s in (("normal", copy_s), ("high", hi_s)):
            for busy in (False, True):
                torch.cuda.synchronize()
                e1 = gemm_loop()[1] if busy else None
                times = []
                while len(times) < 40 and (e1 is None or not e1.query()):
                    t = time.perf_counter()
                    ctx.batch_copy(desc, s)
                    s.synchronize()
                    times.append(time.perf_counter() - t)
                torch.cuda.synchronize()
                key = f"index_pages_{name}_priority_{'under_gemm' if busy else 'idle'}_us"
                out[key] = round(st.median(times) * 1e6, 1) if times else None
        del src, dst
    del a, b
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle timings
# ---------------------------------------------------------------------------
def oracle_sample(budget_s: float, n: int = 4 * MiB):
    """The oracle's dstReference over 3 default-pattern sources of n float32,
    repeated until budget_s has passed; returns (GB/s, reps, seconds)."""
    import oracle
    refs = [oracle.prepare_reference(n, k) for k in range(3)]
    oracle.dst_reference(refs)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.dst_reference(refs)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return 4 * 4 * n * reps / el / 1e9, reps, el


def host_cpu() -> dict:
    """The host the oracle ran on: CPU model (or Arm implementer / part
    numbers where the kernel reports no model name), architecture, logical
    CPUs and the current / maximum clock of CPU 0 where sysfs reports them."""
    import platform
    info = {"arch": platform.machine(), "logical_cpus": os.cpu_count()}
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k and v and k not in fields:
                    fields[k] = v
    except OSError:
        pass
    # Arm Ltd. (implementer 0x41) core part numbers
    arm_parts = {"0xd0c": "Neoverse N1", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2",
                 "0xd4f": "Neoverse V2"}
    if "model name" in fields:
        info["model"] = fields["model name"]
    elif "CPU part" in fields:
        impl, part = fields.get("CPU implementer", "?"), fields["CPU part"]
        named = arm_parts.get(part) if impl == "0x41" else None
        info["model"] = named or f"Arm implementer {impl} part {part}"
    for key, name in (("mhz", "scaling_cur_freq"), ("max_mhz", "cpuinfo_max_freq")):
        try:
            with open(f"/sys/devices/system/cpu/cpu0/cpufreq/{name}") as f:
                info[key] = round(int(f.read().strip()) / 1000)
        except (OSError, ValueError):
            pass
    return info


def oracle_batch_sample(reps: int = 5):
    """The oracle's batch apply (one memcpy per descriptor, in order) of the
    3840- and 7200-page layouts on their host pools, single thread: one
    untimed apply to touch the pages, then the best of `reps` for each."""
    import numpy as np
    import oracle
    from copy_reduce_dst_gb300 import workloads
    out = {"unit": "copies/s", "cores": 1, "kind": "oracle"}
    for key, layout in (("index_pages_3840", workloads.batch_index_pages()),
                        ("block_pages_7200", workloads.batch_block_pages())):
        src = np.zeros(layout.src_pool_bytes, dtype=np.uint8)
        dst = np.zeros(layout.dst_pool_bytes, dtype=np.uint8)
        oracle.apply_batch(dst, src, layout.src_off, layout.dst_off, layout.lens)
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            oracle.apply_batch(dst, src, layout.src_off, layout.dst_off, layout.lens)
            best = min(best, time.perf_counter() - t0)
        out[key] = {"value": round(layout.n / best, 1), "us_per_batch": round(best * 1e6, 1),
                    "gbps": round(2 * layout.total_bytes / best / 1e9, 3)}
        del src, dst
    out["value"] = out["index_pages_3840"]["value"]
    out["sample"] = (f"the 3840- and 7200-page batches applied to their host pools, best of "
                     f"{reps} each, single thread; value = the 3840-page batch")
    return out


def parallel_cpu_sample(budget_s: float, n: int = 16 * MiB):
    """A second CPU baseline, on every host core (not the oracle): the same
    3-source reduce-copy as numpy adds, (src0 + src1) + src2 in float32, over
    chunks taken by a pool of threads (numpy releases the interpreter lock
    inside its loops).  Sources of n float32 each (256 MiB moved per call,
    above the host's last-level cache); one result is compared bit for bit
    with the oracle's dstReference first."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import oracle
    threads = os.cpu_count() or 1
    srcs = [oracle.prepare_reference(n, k) for k in range(3)]
    dst = np.empty(n, dtype=np.float32)
    step = -(-n // (4 * threads))
    bounds = [(a, min(n, a + step)) for a in range(0, n, step)]

    def part(ab):
        a, b = ab
        np.add(srcs[0][a:b], srcs[1][a:b], out=dst[a:b])
        np.add(dst[a:b], srcs[2][a:b], out=dst[a:b])

    with ThreadPoolExecutor(threads) as pool:
        list(pool.map(part, bounds))
        exact = bool(np.array_equal(dst.view(np.uint32),
                                    oracle.dst_reference(srcs).view(np.uint32)))
        calls, t0 = 0, time.perf_counter()
        while True:
            list(pool.map(part, bounds))
            calls += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return {"value": round(4 * 4 * n * calls / el / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "numpy adds on a thread pool (not the oracle)", "bit_exact_vs_oracle": exact,
            "sample": f"3 x {n:,} float32 default-pattern sources (256 MiB moved per call), "
                      f"{calls} calls in {el:.1f} s, {len(bounds)} chunks on {threads} threads"}


def cpu_baseline(budget_s: float):
    gbps, reps, el = oracle_sample(budget_s)
    return {"value": round(gbps, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"dstReference[3] over 3 x 4,194,304 float32 default-pattern sources "
                      f"(64 MiB moved per call), {reps} calls in {el:.1f} s, single thread",
            "host": host_cpu(), "batch": oracle_batch_sample(),
            "parallel": parallel_cpu_sample(min(2.0, budget_s))}


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    n = 4 * MiB
    refs = [oracle.prepare_reference(n, k) for k in range(3)]
    for _ in range(args.warmup):
        oracle.dst_reference(refs)
    times = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.dst_reference(refs)
        times.append(time.perf_counter() - t)
    el = time.perf_counter() - t0
    value = 4 * 4 * n * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "3 x 4,194,304 float32 per step",
                   "parallelism": "none (CPU, 1 thread)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"dstReference[3] over 3 x 4,194,304 float32 per step, "
                                   f"{args.steps} steps", "host": host_cpu()},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Study lines (not the default): single transfer and the fillCompress sweep
# ---------------------------------------------------------------------------
def study(args, tb, torch, local):
    """Single 4 MiB transfer (K = 64) and the fillCompress sweep with rotation
    on and off.  Like-for-like cold / warm, both with CUDA events around every
    launch: cold = mean of 10 single iterations, each after writing a 512 MiB
    buffer (> L2); warm = 20 back-to-back iterations after 3 warm-ups (their
    events telescope, so the ~1 us event resolution does not bias the sum).
    warm_graph = the same 20 iterations as one CUDA graph (no launch gaps).
    Each figure is the median of 3 reps."""
    import statistics as st
    flush = torch.empty(512 * MiB, dtype=torch.uint8, device="cuda")
    with tb.Context(local, ctx_options(tb)) as ctx, \
            tb.Context(local, ctx_options(tb, use_graph=0)) as ev_ctx, \
            tb.Context(local, ctx_options(tb, use_pdl=0)) as serial_ctx, \
            tb.Context(local, ctx_options(tb, warmup=0, use_graph=0)) as cold_ctx:
        nb = 4 * MiB
        plan = tb.rotation_plan(nb, 256 * MiB)
        src = torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda")
        ctx.fill_source(src, nb, tb.default_pattern(), 0)
        ctx.prepare_sources([src], nb, 256 * MiB)
        dst = torch.zeros(nb, dtype=torch.uint8, device="cuda")

        def med(c, iters=10):
            runs = [c.run_transfer([src], dst, nb, iters=iters, rotate_bytes=256 * MiB)
                    for _ in range(5)]
            return sorted(runs, key=lambda r: r["gbps"])[2]
        r, re, rs = med(ctx), med(ev_ctx), med(serial_ctx)
        # One full rotation (64 iterations): the event timer's ~2 us steps
        # blur a 10-iteration span, not a 64-iteration one.
        r64, rs64 = med(ctx, 64), med(serial_ctx, 64)
        print(json.dumps({"study": "single transfer 4 MiB, K=64 (median of 5 runs of 10)",
                          "gbps_graph": round(r["gbps"], 1),
                          "us_per_iteration_graph": round(r["mean_ms"] * 1e3, 2),
                          "gbps_graph_no_pdl": round(rs["gbps"], 1),
                          "us_per_iteration_graph_no_pdl": round(rs["mean_ms"] * 1e3, 2),
                          "gbps_events": round(re["gbps"], 1),
                          "us_per_iteration_events": round(re["mean_ms"] * 1e3, 2),
                          "gbps_graph_64": round(r64["gbps"], 1),
                          "us_per_iteration_graph_64": round(r64["mean_ms"] * 1e3, 3),
                          "gbps_graph_no_pdl_64": round(rs64["gbps"], 1),
                          "us_per_iteration_graph_no_pdl_64": round(rs64["mean_ms"] * 1e3, 3),
                          "K": r["K"], "alloc_bytes": r["alloc_bytes"]}), flush=True)
        del src
        pct = (40, 20, 0, 20, 20)
        for mib in (8, 16, 32, 64, 128, 256, 512):
            nb = mib * MiB
            row = {"study": "fillCompress sweep", "MiB": mib}
            for rot in (256 * MiB, 0):
                plan = tb.rotation_plan(nb, rot)
                src = torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda")
                ctx.fill_source(src, nb, tb.compress_pattern(pct, 0x5EED), 0)
                ctx.prepare_sources([src], nb, rot)
                dst = torch.zeros(nb, dtype=torch.uint8, device="cuda")
                cold, warm, graph = [], [], []
                for rep in range(3):
                    c = []
                    for _ in range(10):
                        flush.fill_(rep)
                        c.append(cold_ctx.run_transfer([src], dst, nb, iters=1,
                                                       rotate_bytes=rot)["total_ms"])
                    cold.append(2 * nb / (st.mean(c) / 1e3) / 1e9)
                    warm.append(ev_ctx.run_transfer([src], dst, nb, iters=20, rotate_bytes=rot)["gbps"])
                    graph.append(ctx.run_transfer([src], dst, nb, iters=20, rotate_bytes=rot)["gbps"])
                tag = "on" if rot else "off"
                row[f"{tag}_K"] = plan.K
                row[f"{tag}_cold_gbps"] = round(st.median(cold), 1)
                row[f"{tag}_warm_gbps"] = round(st.median(warm), 1)
                row[f"{tag}_w_over_c"] = round(st.median(warm) / st.median(cold), 3)
                row[f"{tag}_warm_graph_gbps"] = round(st.median(graph), 1)
                del src, dst
            row["off_over_on_warm_graph"] = round(row["off_warm_graph_gbps"] / row["on_warm_graph_gbps"], 3)
            print(json.dumps(row), flush=True)
    del flush
    print(json.dumps(study_validation(tb, torch, local)), flush=True)
    study_host_paths(tb, torch, local)
    study_tiny_batches(tb, torch, local)
    study_small_copies_under_compute(tb, torch, local)
    study_batch_configs(tb, torch, local)
    study_batch_phases(tb, torch, local)
    study_batch_routing(tb, torch, local)
    study_interference(tb, torch, local)
    study_grid_cap(tb, torch, local)


def study_batch_routing(tb, torch, local):
    """The 47,540 batch with its copies of at least 1 MiB (the 20 long ones)
    sent to the copy engines instead of the kernel: device time per call of
    10 back-to-back calls after 3 (upload + kernel + copy engines; the host
    packs the next call while the GPU works), median of 3 reps."""
    import statistics as st
    from copy_reduce_dst_gb300 import workloads
    layout = workloads.batch_head_sliced()
    src = torch.zeros(layout.src_pool_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(layout.dst_pool_bytes, dtype=torch.uint8, device="cuda")
    desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
    stream = torch.cuda.current_stream()
    for ce in (0, 1 << 20):
        with tb.Context(local, ctx_options(tb, ce_min_bytes=ce)) as ctx:
            ms = []
            for rep in range(4):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(10):
                    ctx.batch_copy(desc, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                if rep >= 1:
                    ms.append(e0.elapsed_time(e1) / 10)
            print(json.dumps({"study": "batch routing", "ce_min_bytes": ce,
                              "device_ms": round(st.median(ms), 4),
                              "gbps": round(2 * layout.total_bytes / (st.median(ms) / 1e3) / 1e9, 1)}),
                  flush=True)


def study_interference(tb, torch, local):
    """bf16 GEMM throughput (8192^3 torch.matmul on one stream) while the
    47,540 batch is copied on another stream at several rates (a batch every
    `gap` ms; 0 = back to back), the Mooncake RFC's interference measurement."""
    from copy_reduce_dst_gb300 import workloads
    n = 8192
    a = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    b = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    layout = workloads.batch_head_sliced()
    src = device_random_bytes(torch, layout.src_pool_bytes, 63)
    dst = device_random_bytes(torch, layout.dst_pool_bytes, 64)
    desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
    gemm_s = torch.cuda.Stream()
    copy_s = torch.cuda.Stream()
    flops = 2 * n ** 3

    def run(gap_ms, seconds=1.5):
        with tb.Context(local, ctx_options(tb)) as ctx:
            torch.cuda.synchronize()
            with torch.cuda.stream(gemm_s):
                for _ in range(3):
                    torch.matmul(a, b)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(gemm_s)
            with torch.cuda.stream(gemm_s):
                for _ in range(int(seconds * 1900e12 / flops)):
                    torch.matmul(a, b)
            e1.record(gemm_s)
            batches = 0
            t0 = time.perf_counter()
            while not e1.query():
                if gap_ms is not None:
                    ctx.batch_copy(desc, copy_s)
                    batches += 1
                    if gap_ms > 0:
                        time.sleep(gap_ms / 1e3)
                    else:
                        copy_s.synchronize()
                else:
                    time.sleep(0.01)
            wall = time.perf_counter() - t0
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            iters = int(seconds * 1900e12 / flops)
            return iters * flops / (ms / 1e3) / 1e12, 2 * layout.total_bytes * batches / wall / 1e9

    alone, _ = run(None)
    print(json.dumps({"study": "interference", "copy_gap_ms": None, "gemm_tflops": round(alone, 1),
                      "copy_gbps": 0.0}), flush=True)
    for gap in (20, 5, 1, 0):
        tf, gbps = run(gap)
        print(json.dumps({"study": "interference", "copy_gap_ms": gap, "gemm_tflops": round(tf, 1),
                          "copy_gbps": round(gbps, 1),
                          "gemm_loss_pct": round(100 * (1 - tf / alone), 2),
                          "loss_pct_per_100gbps": round(100 * (1 - tf / alone) / max(gbps, 1e-9) * 100, 3)}),
              flush=True)


def study_grid_cap(tb, torch, local):
    """The Mooncake RFC's open question 4 (a CU mask or rate limit for GPUs
    that also compute): an 8192^3 bf16 GEMM loop on one stream while the
    47,540 batch is copied back to back on another, with the batch kernel's
    grid capped at `batch_max_ctas` CTAs (none, 304, 152, 64, 32).  GEMM
    TFLOP/s, copy GB/s and the GEMM's loss per 100 GB/s of copies."""
    from copy_reduce_dst_gb300 import workloads
    n = 8192
    a = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    b = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
    flops = 2 * n ** 3
    reps = 900  # ~0.5 s of GEMMs alone
    layout = workloads.batch_head_sliced()
    src = device_random_bytes(torch, layout.src_pool_bytes, 61)
    dst = device_random_bytes(torch, layout.dst_pool_bytes, 62)
    desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
    gemm_s = torch.cuda.Stream()
    copy_s = torch.cuda.Stream()

    def loop():
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(gemm_s)
        with torch.cuda.stream(gemm_s):
            for _ in range(reps):
                torch.matmul(a, b, out=c)
        e1.record(gemm_s)
        return e0, e1

    with torch.cuda.stream(gemm_s):
        for _ in range(20):
            torch.matmul(a, b, out=c)
    torch.cuda.synchronize()
    e0, e1 = loop()
    torch.cuda.synchronize()
    alone = reps * flops / (e0.elapsed_time(e1) / 1e3) / 1e12
    print(json.dumps({"study": "grid cap", "cap": "no copies", "gemm_tflops": round(alone, 1)}),
          flush=True)
    for cap in (0, 304, 152, 64, 32):
        with tb.Context(local, ctx_options(tb, batch_max_ctas=cap)) as ctx:
            ctx.batch_copy(desc, copy_s)
            copy_s.synchronize()
            e0, e1 = loop()
            batches, t0 = 0, time.perf_counter()
            while not e1.query():
                ctx.batch_copy(desc, copy_s)
                copy_s.synchronize()
                batches += 1
            wall = time.perf_counter() - t0
            torch.cuda.synchronize()
        tf = reps * flops / (e0.elapsed_time(e1) / 1e3) / 1e12
        gbps = 2 * layout.total_bytes * batches / wall / 1e9
        loss = 100 * (1 - tf / alone)
        print(json.dumps({"study": "grid cap", "cap": cap or "none", "gemm_tflops": round(tf, 1),
                          "copy_gbps": round(gbps, 1), "gemm_loss_pct": round(loss, 2),
                          "loss_pct_per_100gbps": round(loss / max(gbps, 1e-9) * 100, 3)}),
              flush=True)
    del a, b, c, src, dst
    torch.cuda.empty_cache()


def study_small_copies_under_compute(tb, torch, local):
    """The 3840-page batch (3840 x 2112 B) copied while an 8192^3 bf16 GEMM
    loop keeps every SM busy on another stream, against the same copies on
    an idle GPU: tb_batch_copy, and one cudaMemcpyAsync per copy
    (tb_copy_each).  The Mooncake RFC saw per-copy memcpy collapse to
    0.03-0.04 GB/s under compute.  Wall time per batch (call + sync), median
    of the batches that ran while the GEMM loop was in flight."""
    import statistics as st
    from copy_reduce_dst_gb300 import workloads
    n = 8192
    a = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    b = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    layout = workloads.batch_index_pages()
    src = torch.zeros(layout.src_pool_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(layout.dst_pool_bytes, dtype=torch.uint8, device="cuda")
    desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
    gemm_s = torch.cuda.Stream()
    copy_s = torch.cuda.Stream()
    hi_s = torch.cuda.Stream(priority=-1)      # the caller's high-priority stream
    moved = 2 * layout.total_bytes
    out = {"study": "small copies under compute", "workload": layout.name}
    with tb.Context(local, ctx_options(tb)) as ctx:
        for name, fn, cs in (("batch", lambda: ctx.batch_copy(desc, copy_s), copy_s),
                             ("batch_high_priority", lambda: ctx.batch_copy(desc, hi_s), hi_s),
                             ("memcpy_each", lambda: ctx.copy_each(desc, copy_s), copy_s)):
            for busy in (False, True):
                torch.cuda.synchronize()
                end = None
                if busy:
                    with torch.cuda.stream(gemm_s):
                        for _ in range(3):
                            torch.matmul(a, b)
                    torch.cuda.synchronize()
                    end = torch.cuda.Event()
                    with torch.cuda.stream(gemm_s):
                        for _ in range(1500):         # ~1 s of GEMM
                            torch.matmul(a, b)
                    end.record(gemm_s)
                times = []
                limit = 3 if name == "memcpy_each" else 50
                while len(times) < limit and (end is None or not end.query()):
                    t0 = time.perf_counter()
                    fn()
                    cs.synchronize()
                    times.append(time.perf_counter() - t0)
                torch.cuda.synchronize()
                key = f"{name}_{'under_gemm' if busy else 'idle'}"
                if times:
                    w = st.median(times)
                    out[key + "_ms"] = round(w * 1e3, 3)
                    out[key + "_gbps"] = round(moved / w / 1e9, 2)
                out[key + "_samples"] = len(times)
    print(json.dumps(out), flush=True)
    del a, b, src, dst


def study_host_paths(tb, torch, local):
    """tb_reduce_copy_host on the bench workload (3 x 256 MiB): pinned host
    buffers (one kernel reads and writes them across the host link) against
    pageable ones (staged through device buffers in 32 MiB chunks on three
    streams); wall time per call with the stream synchronised, median of 5
    after 1, GB/s counting read + write bytes as the bench line does."""
    import statistics as st
    nb = 256 * MiB
    moved = 4 * nb
    dsrc = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(3)]
    ddst = torch.empty(nb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    out = {"study": "host paths", "workload": "3 x 256 MiB reduce-copy from host memory"}
    with tb.Context(local, ctx_options(tb)) as ctx:
        for kind in ("pinned", "pageable"):
            hs = [torch.full((nb // 4,), float(k + 1), dtype=torch.float32) for k in range(3)]
            hd = torch.empty(nb // 4, dtype=torch.float32)
            if kind == "pinned":
                hs = [h.pin_memory() for h in hs]
                hd = hd.pin_memory()
            t = []
            for i in range(6):
                t0 = time.perf_counter()
                ctx.reduce_copy_host(hs, hd, nb, dsrc, ddst, 0, stream)
                stream.synchronize()
                if i:
                    t.append(time.perf_counter() - t0)
            assert float(hd[12345]) == 6.0
            out[kind + "_ms"] = round(st.median(t) * 1e3, 2)
            out[kind + "_gbps"] = round(moved / st.median(t) / 1e9, 1)
            del hs, hd
    print(json.dumps(out), flush=True)


def study_tiny_batches(tb, torch, local):
    """Batches of 1 to 64 copies of 2112 B: wall time per call (call + sync,
    median of 200) through tb_batch_copy (one kernel) and through one
    cudaMemcpyAsync per copy - where a kernel launch stops paying off."""
    import statistics as st
    import numpy as np
    pool = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    base = pool.data_ptr()
    rows = []
    with tb.Context(local, ctx_options(tb)) as ctx:
        for k in (1, 2, 4, 8, 16, 32, 64):
            desc = np.array([[base + i * 4224, base + (32 << 20) + i * 4224, 2112]
                             for i in range(k)], dtype=np.uint64)
            row = {"copies": k}
            for name, fn in (("batch_us", lambda: ctx.batch_copy(desc, s)),
                             ("memcpy_each_us", lambda: ctx.copy_each(desc, s))):
                for _ in range(20):
                    fn()
                s.synchronize()
                t = []
                for _ in range(200):
                    t0 = time.perf_counter()
                    fn()
                    s.synchronize()
                    t.append(time.perf_counter() - t0)
                row[name] = round(st.median(t) * 1e6, 2)
            rows.append(row)
    print(json.dumps({"study": "tiny batches", "rows": rows}), flush=True)


def study_validation(tb, torch, local):
    """Validation of a 256 MiB destination (the bench line's dst): on the
    device (tb_validate_device, a compare kernel reading dst and an expected
    copy in HBM, first difference by atomicMin) against the host path
    (tb_validate: device-to-host copy in chunks and memcmp).  Wall time of
    each synchronous call, median of 5 after 2; and the 3-source transfer
    with validation after every iteration on the device."""
    import statistics as st
    nb = 256 * MiB
    n = nb // 4
    with tb.Context(local, ctx_options(tb)) as ctx:
        srcs = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(3)]
        for k, s_ in enumerate(srcs):
            ctx.fill_source(s_, nb, tb.default_pattern(), k)
        dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
        ctx.reduce_copy(srcs, dst, nb)
        exp_dev = dst.clone()
        exp_host = exp_dev.cpu().numpy()
        torch.cuda.synchronize()
        out = {"study": "validation", "MiB": 256}
        for name, fn in (("device", lambda: ctx.validate_device(dst, exp_dev, nb)),
                         ("host", lambda: ctx.validate(dst, exp_host, nb))):
            for _ in range(2):
                assert fn() is None
            t = []
            for _ in range(5):
                t0 = time.perf_counter()
                assert fn() is None
                t.append(time.perf_counter() - t0)
            ms = st.median(t) * 1e3
            out[name + "_ms"] = round(ms, 3)
            read = 2 * nb if name == "device" else nb
            out[name + "_gbps_read"] = round(read / (ms / 1e3) / 1e9, 1)
        with tb.Context(local, ctx_options(tb, always_validate=1)) as vctx:
            walls = {}
            for name, c, kw in (("end", ctx, {}), ("every_iteration", vctx,
                                                   {"expected_device": exp_dev})):
                c.run_transfer(srcs, dst, nb, 0, iters=10, rotate_bytes=0, **kw)
                t0 = time.perf_counter()
                c.run_transfer(srcs, dst, nb, 0, iters=10, rotate_bytes=0, **kw)
                walls[name] = (time.perf_counter() - t0) * 1e3 / (10 + 3)
            out["transfer_wall_ms_per_launch_no_validation"] = round(walls["end"], 4)
            out["transfer_wall_ms_per_launch_validating_each"] = round(walls["every_iteration"], 4)
        del srcs, dst, exp_dev
    torch.cuda.empty_cache()
    return out


def study_batch_configs(tb, torch, local):
    """The three batch workloads side by side: 3840 x 2112 B pages into a
    1 GiB pool, 7200 copies of 512 B-16 KiB, and the 47,540-descriptor batch.
    kernel_us = kernel-only events (median of 20); device_us = events around
    30 back-to-back calls (work-list upload + kernel); wall_us = one call
    with packing, upload, kernel and stream sync (median of 20); each_ms =
    one cudaMemcpyAsync per copy, wall-timed the same way (best of 2)."""
    import statistics as st
    from copy_reduce_dst_gb300 import workloads
    for layout in (workloads.batch_index_pages(), workloads.batch_block_pages(),
                   workloads.batch_head_sliced()):
        src = torch.zeros(layout.src_pool_bytes, dtype=torch.uint8, device="cuda")
        dst = torch.zeros(layout.dst_pool_bytes, dtype=torch.uint8, device="cuda")
        desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
        stream = torch.cuda.Stream()
        moved = 2 * int(layout.total_bytes)
        with tb.Context(local, ctx_options(tb, time_kernels=1)) as kctx, \
                tb.Context(local, ctx_options(tb)) as ctx:
            for _ in range(3):
                kctx.batch_copy(desc, stream)
            kern = []
            for _ in range(20):
                kctx.batch_copy(desc, stream)
                kern.append(kctx.last_batch_kernel_ms())
            for _ in range(3):
                ctx.batch_copy(desc, stream)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            a.record(stream)
            for _ in range(30):
                ctx.batch_copy(desc, stream)
            b.record(stream)
            b.synchronize()
            dev_ms = a.elapsed_time(b) / 30
            walls = []
            for _ in range(20):
                t0 = time.perf_counter()
                ctx.batch_copy(desc, stream)
                stream.synchronize()
                walls.append(time.perf_counter() - t0)
            each = []
            for _ in range(2):
                t0 = time.perf_counter()
                ctx.copy_each(desc, stream)
                stream.synchronize()
                each.append(time.perf_counter() - t0)
        k_ms = st.median(kern)
        wall = st.median(walls)
        print(json.dumps({
            "study": "batch configs", "workload": layout.name, "descriptors": layout.n,
            "bytes_copied": int(layout.total_bytes),
            "kernel_us": round(k_ms * 1e3, 2), "kernel_gbps": round(moved / (k_ms / 1e3) / 1e9, 1),
            "device_us": round(dev_ms * 1e3, 2), "device_gbps": round(moved / (dev_ms / 1e3) / 1e9, 1),
            "wall_us": round(wall * 1e6, 1), "copies_per_s_wall": round(layout.n / wall, 1),
            "copies_per_s_device": round(layout.n / (dev_ms / 1e3), 1),
            "each_ms": round(min(each) * 1e3, 3),
            "speedup_vs_memcpy_each": round(min(each) / wall, 1)}), flush=True)
        del src, dst


def study_batch_phases(tb, torch, local):
    """Kernel time of the 47,540 batch, of its bytes as one contiguous copy,
    and of its parts: the 20 long copies alone, the 47,520 short copies
    alone, the same short copies laid out back to back in both pools, their
    bytes as one contiguous copy, and one 1 GiB copy (median of 10 launches
    after 3, kernel-only events)."""
    import statistics as st
    import numpy as np
    from copy_reduce_dst_gb300 import workloads
    layout = workloads.batch_head_sliced()
    src = torch.zeros(layout.src_pool_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(layout.dst_pool_bytes, dtype=torch.uint8, device="cuda")
    desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
    long_ = desc[:, 2] > 16384
    short = desc[~long_]
    lens = short[:, 2]
    packed = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.uint64)
    back_to_back = np.stack([np.uint64(src.data_ptr()) + packed,
                             np.uint64(dst.data_ptr()) + packed, lens], axis=1)
    same_bytes = desc[:1].copy()
    same_bytes[0] = (src.data_ptr(), dst.data_ptr(), int(lens.sum()))
    all_bytes = desc[:1].copy()
    all_bytes[0] = (src.data_ptr(), dst.data_ptr(), int(desc[:, 2].sum()))
    one = desc[:1].copy()
    one[0] = (src.data_ptr(), dst.data_ptr(), GiB)
    with tb.Context(local, ctx_options(tb, time_kernels=1)) as ctx:
        for name, d in (("all 47,540", desc), ("all their bytes as one contiguous copy", all_bytes),
                        ("20 long copies", desc[long_]),
                        ("47,520 short copies", short),
                        ("47,520 short copies laid out back to back", back_to_back),
                        ("their bytes as one contiguous copy", same_bytes),
                        ("one 1 GiB copy", one)):
            for _ in range(3):
                ctx.batch_copy(d)
            ms = []
            for _ in range(10):
                ctx.batch_copy(d)
                ms.append(ctx.last_batch_kernel_ms())
            k = st.median(ms)
            moved = 2 * int(d[:, 2].sum())
            print(json.dumps({"study": "batch phases", "part": name, "kernel_us": round(k * 1e3, 1),
                              "gbps": round(moved / (k / 1e3) / 1e9, 1)}), flush=True)


# ---------------------------------------------------------------------------
# Profiling target: 3 warm-up + 3 launches of one kernel on the bench's own
# workload, nothing else (for ncu -k ... -s 3 -c 1..3).
# ---------------------------------------------------------------------------
def profile_target(kind, args, tb, torch, local):
    stream = torch.cuda.current_stream()
    if kind == "reduce":
        nb = 256 * MiB
        with tb.Context(local, ctx_options(tb)) as ctx:
            srcs = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(3)]
            for k, s in enumerate(srcs):
                ctx.fill_source(s, nb, tb.default_pattern(), k, stream)
            dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
            for _ in range(6):
                ctx.reduce_copy(srcs, dst, nb, 32, stream)
            torch.cuda.synchronize()
    elif kind == "rotation":
        # One fillCompress transfer of args.mib MiB with SRC_ROTATE_BYTES =
        # args.rotate_mib MiB: 4 timed iterations inside an NVTX range "timed"
        # (profile with --nvtx --nvtx-include timed/ --cache-control none).
        nb = args.mib * MiB
        rot = args.rotate_mib * MiB
        with tb.Context(local, ctx_options(tb, warmup=0)) as ctx:
            plan = tb.rotation_plan(nb, rot)
            src = torch.empty(plan.alloc_bytes, dtype=torch.uint8, device="cuda")
            ctx.fill_source(src, nb, tb.compress_pattern((40, 20, 0, 20, 20), 0x5EED), 0)
            ctx.prepare_sources([src], nb, rot)
            dst = torch.zeros(nb, dtype=torch.uint8, device="cuda")
            ctx.run_transfer([src], dst, nb, iters=4, rotate_bytes=rot)
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("timed")
            r = ctx.run_transfer([src], dst, nb, iters=4, rotate_bytes=rot)
            torch.cuda.nvtx.range_pop()
            print(json.dumps({"K": r["K"], "iter_ms": r["iter_ms"]}), flush=True)
    elif kind == "batch-small":
        # The 3840-page and 7200-page batches, 5 calls each; kernel times
        # from the library's events.
        from copy_reduce_dst_gb300 import workloads
        with tb.Context(local, ctx_options(tb, time_kernels=1)) as ctx:
            for name, lay in (("3840 index pages", workloads.batch_index_pages()),
                              ("7200 block pages", workloads.batch_block_pages())):
                src = device_random_bytes(torch, lay.src_pool_bytes, 31)
                dst = device_random_bytes(torch, lay.dst_pool_bytes, 32)
                desc = lay.descriptors(src.data_ptr(), dst.data_ptr())
                ms = []
                for _ in range(5):
                    ctx.batch_copy(desc)
                    ms.append(round(ctx.last_batch_kernel_ms() * 1e3, 2))
                print(json.dumps({"batch": name, "event_us": ms,
                                  "direct": ctx.last_batch_stats()["direct_launches"]}),
                      flush=True)
                del src, dst
        print("profile target batch-small: 10 launches done", flush=True)
        return 0
    else:
        from copy_reduce_dst_gb300 import workloads
        layout = workloads.batch_head_sliced(pool_bytes=args.pool_gib * GiB)
        src = device_random_bytes(torch, layout.src_pool_bytes, 41)
        dst = device_random_bytes(torch, layout.dst_pool_bytes, 42)
        desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
        if kind == "batch-short":  # its 47,520 short copies alone
            desc = desc[desc[:, 2] <= 16384]
        with tb.Context(local, ctx_options(tb)) as ctx:
            for _ in range(6):
                ctx.batch_copy(desc, stream)
            torch.cuda.synchronize()
    print(f"profile target {kind}: 6 launches done", flush=True)
    return 0


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-batch", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave out the single transfer, DMA executor, rotation sweep, small "
                         "batches and interference keys")
    ap.add_argument("--study", action="store_true")
    ap.add_argument("--profile", choices=["reduce", "batch", "batch-short", "batch-small",
                                          "rotation"])
    ap.add_argument("--mib", type=int, default=16, help="--profile rotation: transfer MiB")
    ap.add_argument("--rotate-mib", type=int, default=256,
                    help="--profile rotation: SRC_ROTATE_BYTES in MiB (0 = off)")
    ap.add_argument("--pool-gib", type=int, default=2,
                    help="--profile batch / batch-short: size of each pool of the 47,540 "
                         "layout in GiB (a smaller case for full ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    from copy_reduce_dst_gb300 import tb  # fails loudly if libtb.so is missing
    if args.study:
        return study(args, tb, torch, local)
    if args.profile:
        return profile_target(args.profile, args, tb, torch, local)
    ranks = Ranks(world, "nccl")
    red = run_reduce(args, tb, torch, ranks, local)
    batch = None if args.no_batch else run_batch(args, tb, torch, ranks, local)
    extra = {}
    if not args.no_extra:
        from copy_reduce_dst_gb300 import workloads
        extra["single_4mib_k64"] = run_single_transfer(tb, torch, local)
        extra["dma_executor_256mib"] = run_dma_large(tb, torch, local)
        extra["rotation_sweep"] = run_rotation_sweep(tb, torch, local)
        extra["index_pages_3840"] = run_small_batch(tb, torch, local, workloads.batch_index_pages,
                                                    31, 32)
        extra["block_pages_7200"] = run_small_batch(tb, torch, local, workloads.batch_block_pages,
                                                    33, 8)
        extra["multi_source_fill_compress"] = run_multi_source_compress(tb, torch, local)
        extra["validation_256mib"] = study_validation(tb, torch, local)
        # Last: its GEMM loops run the GPU at its power limit for seconds,
        # which would slow whatever ran next.
        extra["interference"] = run_interference(tb, torch, local)
    cpu = cpu_baseline(args.cpu_seconds) if (rank == 0 and world == 1) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(red["value"], 1), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(red["ms_per_step"], 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "num_subexec": red["subexec"],
                       "num_subexec_choice": "best of the sweep 1, 4, 16, 32",
                       "step": "one reduce-copy launch over 3 x 256 MiB -> 256 MiB "
                               "(1,073,741,824 B moved); the K timed steps run as one CUDA "
                               "graph replay",
                       "l2": "inputs larger than L2 (1 GiB per step vs 129 MB), no flush",
                       "parallelism": f"replicas x{world} (no data exchange)",
                       "subexec_sweep": red["subexec_sweep"],
                       "strict_one_cta_per_subexec": red["strict_one_cta_per_subexec"],
                       "pct_of_peak": round(red["value"] / world / read_peaks()[0] * 100, 1)},
            "roofline": red["roofline"], "cpu_baseline": cpu, "e2e": red["e2e"],
            "clocks": red["clocks"], "gpu_launches": red["gpu_launches"], "batch": batch,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    ranks.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())

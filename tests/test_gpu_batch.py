"""GPU parity of the batched descriptor copy (through the C ABI) against the
oracle's batch apply.  Bar: bit-exact over the whole destination pool, whose
untouched bytes keep a seeded random fill, so a stray write anywhere shows."""
import numpy as np
import pytest

import oracle
from copy_reduce_dst_gb300 import workloads
from gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu

MiB = 1 << 20


@pytest.fixture(scope="module")
def tb():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from copy_reduce_dst_gb300 import _build
    _build.build()
    from copy_reduce_dst_gb300 import tb as mod
    return mod


def run_layout(tb, ctx, layout, seed=1, stream=None, src_shift=0, dst_shift=0):
    """Random pools, one tb_batch_copy of the layout, whole-pool comparison.
    src_shift / dst_shift move every copy by a few bytes to vary alignment."""
    import torch
    src_h = workloads.random_bytes(layout.src_pool_bytes + 64, seed)
    dst_h = workloads.random_bytes(layout.dst_pool_bytes + 64, seed + 1000)
    src_d = to_dev(src_h)
    dst_d = to_dev(dst_h)
    so = layout.src_off + np.uint64(src_shift)
    do = layout.dst_off + np.uint64(dst_shift)
    desc = np.stack([np.uint64(src_d.data_ptr()) + so, np.uint64(dst_d.data_ptr()) + do,
                     layout.lens], axis=1)
    ctx.batch_copy(desc, stream)
    if stream is not None:
        stream.synchronize()
    got = to_host(dst_d)
    exp = dst_h.copy()
    oracle.apply_batch(exp, src_h, so, do, layout.lens)
    mm = oracle.first_mismatch(got, exp)
    assert mm == -1, f"first differing byte {mm}"
    return ctx.last_batch_stats()


@pytest.fixture(scope="module")
def ctx(tb):
    with tb.Context(0) as c:
        yield c


@pytest.mark.parametrize("seed", range(4))
def test_tiny_any_alignment(tb, ctx, seed):
    # lengths 0..300 B at any byte offset of src and dst
    layout = workloads.random_batch(seed, 2000, 300, 4 * MiB, align=1)
    st = run_layout(tb, ctx, layout, seed)
    assert st["descs"] == int((layout.lens > 0).sum())
    assert st["direct_launches"] == 1


@pytest.mark.parametrize("ss,ds", [(0, 0), (1, 0), (0, 1), (3, 7), (15, 1), (4, 12), (8, 8)])
def test_misalignment_pairs(tb, ctx, ss, ds):
    # every src/dst alignment pair over lengths that cross vector and tile edges
    layout = workloads.random_batch(ss * 16 + ds, 3000, 5000, 64 * MiB, align=16)
    run_layout(tb, ctx, layout, 7, src_shift=ss, dst_shift=ds)


@pytest.mark.parametrize("ss,ds", [(0, 0), (5, 5), (16, 16), (31, 31), (16, 0), (0, 16), (8, 24)])
def test_thirty_two_byte_classes(tb, ctx, ss, ds):
    # offsets on 32-byte boundaries, shifted: src and dst equal modulo 32 take
    # the 32-byte path after a head of up to 31 bytes; equal modulo 16 only,
    # the 16-byte path
    layout = workloads.random_batch(100 + ss + ds, 3000, 9000, 64 * MiB, align=32)
    run_layout(tb, ctx, layout, 9, src_shift=ss, dst_shift=ds)


@pytest.mark.parametrize("shift", [0, 1, 8, 15])
def test_ring_piece_boundaries(tb, ctx, shift):
    # Short copies whose src and dst agree modulo 16 go through each warp's
    # ring of shared-memory slots in pieces of 1-2 KiB: lengths at and
    # around every multiple of 1 KiB up to the 16 KiB short limit, with
    # heads and tails of 0-15 bytes (the shift moves src and dst alike).
    base = [1024 * k + d for k in range(17) for d in (-17, -16, -1, 0, 1, 15, 16, 17)]
    lens = np.array([x for x in base if 0 < x <= 16384] * 4, dtype=np.uint64)
    gen = workloads.rng(40 + shift)
    so = workloads.scatter_offsets(gen, lens, 0, 64 * MiB, 16)
    do = workloads.scatter_offsets(gen, lens, 0, 64 * MiB, 16)
    layout = workloads.BatchLayout("piece boundaries", so, do, lens, 64 * MiB, 64 * MiB)
    st = run_layout(tb, ctx, layout, 41 + shift, src_shift=shift, dst_shift=shift)
    assert st["warp_items"] == lens.size


@pytest.mark.parametrize("waves", [1, 2, 4, 5])
@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_short_counts_around_whole_waves(tb, ctx, waves, delta):
    # A launch of short copies only takes one copy per warp while a wave of
    # warps suffices, else whole waves whose warps take a second copy by
    # index (warp w: w, w + starters) before claiming from the counter.
    # Counts at and next to multiples of one copy per warp of a wave (three
    # 256-thread CTAs per SM on GB300) cross each of those rules.
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = sms * 3 * 8 * waves + delta
    lens = np.full(n, 2112, dtype=np.uint64)
    gen = workloads.rng(50 + waves)
    so = workloads.scatter_offsets(gen, lens, 0, 256 * MiB, 64)
    do = workloads.scatter_offsets(gen, lens, 0, 256 * MiB, 64)
    layout = workloads.BatchLayout("around waves", so, do, lens, 256 * MiB, 256 * MiB)
    st = run_layout(tb, ctx, layout, 60 + waves * 3 + delta)
    assert st["descs"] == n and st["launches"] == 1


@pytest.mark.parametrize("host_side", ["src", "dst"])
def test_pinned_host_pool(tb, ctx, host_side):
    # One pool in page-locked host memory (mapped into the device's address
    # space): the short copies' asynchronous copies and the long copies'
    # bulk copies cross the host link, byte-exact.
    import torch
    g = np.random.default_rng(31)
    lens = np.concatenate([g.integers(1, 16385, 400), g.integers(16385, 1 << 20, 6)]).astype(np.uint64)
    gen = workloads.rng(32)
    pool = 32 * MiB
    so = workloads.scatter_offsets(gen, lens, 0, pool, 1)
    do = workloads.scatter_offsets(gen, lens, 0, pool, 1)
    src_h = workloads.random_bytes(pool, 33)
    dst_h = workloads.random_bytes(pool, 34)
    if host_side == "src":
        src = torch.from_numpy(src_h.copy()).pin_memory()
        dst = to_dev(dst_h)
    else:
        src = to_dev(src_h)
        dst = torch.from_numpy(dst_h.copy()).pin_memory()
    desc = np.stack([np.uint64(src.data_ptr()) + so, np.uint64(dst.data_ptr()) + do, lens], axis=1)
    ctx.batch_copy(desc)
    torch.cuda.synchronize()
    got = dst.numpy() if host_side == "dst" else to_host(dst)
    exp = dst_h.copy()
    oracle.apply_batch(exp, src_h, so, do, lens)
    assert oracle.first_mismatch(got, exp) == -1
    st = ctx.last_batch_stats()
    assert st["warp_items"] == 400 and st["cta_items"] > 0


def test_lengths_one_byte_to_three_mib(tb, ctx):
    # Mooncake RFC "Correctness": lengths from 1 B to 3 MiB, unaligned ranges
    g = np.random.default_rng(11)
    lens = np.exp(g.uniform(0, np.log(3 * MiB), 600)).astype(np.uint64)
    lens = np.maximum(lens, 1)
    gen = workloads.rng(12)
    so = workloads.scatter_offsets(gen, lens, 0, 1024 * MiB, 1)
    do = workloads.scatter_offsets(gen, lens, 0, 1024 * MiB, 1)
    layout = workloads.BatchLayout("1B-3MiB", so, do, lens, 1024 * MiB, 1024 * MiB)
    st = run_layout(tb, ctx, layout, 13)
    assert st["cta_items"] > 0 and st["warp_items"] > 0


def test_more_launches_than_slots(tb):
    # 1024 items per slot and 2 slots: the batch needs many launches and every
    # slot is reused while earlier launches may still be running.
    with tb.Context(0, tb.options(slot_items=1024, num_slots=2)) as c:
        layout = workloads.random_batch(21, 9000, 20000, 512 * MiB, align=1)
        st = run_layout(tb, c, layout, 22)
        assert st["launches"] > 2 * 2
        for i in range(3):
            run_layout(tb, c, workloads.random_batch(30 + i, 3000, 4000, 64 * MiB), 40 + i)


@pytest.mark.parametrize("pdl", [1, 0])
@pytest.mark.parametrize("with_long", [0, 1])
def test_batch_chain_reads_previous_output(tb, pdl, with_long):
    """20 batches queued on one stream, batch i copying region i into
    region i + 1 (the next batch's sources): with programmatic dependent
    launch a batch may start while the one before drains and reads its work
    list early, yet every copy still sees the previous batch's output; the
    pool ends as the oracle's batches applied in order."""
    import torch
    steps, per, size, big = 20, 64, 2112, 65536
    region = per * 4224 + (big if with_long else 0)
    pool_h = workloads.random_bytes((steps + 1) * region, 93)
    pool_d = to_dev(pool_h)
    exp = pool_h.copy()
    inner = np.arange(per, dtype=np.uint64) * np.uint64(4224)
    lens = np.full(per, size, dtype=np.uint64)
    if with_long:
        inner = np.append(inner, np.uint64(per * 4224))
        lens = np.append(lens, np.uint64(big))
    with tb.Context(0, tb.options(use_pdl=pdl, num_slots=2)) as c:
        st = torch.cuda.Stream()
        for i in range(steps):
            so = np.uint64(i * region) + inner
            do = np.uint64((i + 1) * region) + inner
            base = np.uint64(pool_d.data_ptr())
            c.batch_copy(np.stack([base + so, base + do, lens], axis=1), st)
            oracle.apply_batch(exp, exp.copy(), so, do, lens)
        st.synchronize()
    assert oracle.first_mismatch(to_host(pool_d), exp) == -1


@pytest.mark.parametrize("with_long", [0, 1])
def test_one_slot_back_to_back(tb, with_long):
    """200 calls queued without a sync on one slot, call i copying its own
    source region into its own destination region (64 copies of 2112 B, plus
    one 64 KiB copy that makes the launch upload its work list): the slot is
    reused only after the launch before it has finished reading the work
    list, so every region ends equal to its source."""
    import torch
    calls, per, size, big = 200, 64, 2112, 65536
    region = per * 4224 + (big if with_long else 0)
    src_h = workloads.random_bytes(calls * region, 91)
    dst_h = workloads.random_bytes(calls * region, 92)
    src_d, dst_d = to_dev(src_h), to_dev(dst_h)
    exp = dst_h.copy()
    with tb.Context(0, tb.options(num_slots=1)) as c:
        st = torch.cuda.Stream()
        for i in range(calls):
            base = i * region
            off = np.uint64(base) + np.arange(per, dtype=np.uint64) * np.uint64(4224)
            lens = np.full(per, size, dtype=np.uint64)
            if with_long:
                off = np.append(off, np.uint64(base + per * 4224))
                lens = np.append(lens, np.uint64(big))
            desc = np.stack([np.uint64(src_d.data_ptr()) + off, np.uint64(dst_d.data_ptr()) + off,
                             lens], axis=1)
            c.batch_copy(desc, st)
            oracle.apply_batch(exp, src_h, off, off, lens)
        stats = c.last_batch_stats()
        st.synchronize()
    assert stats["direct_launches"] == (0 if with_long else 1)
    assert oracle.first_mismatch(to_host(dst_d), exp) == -1


@pytest.mark.parametrize("small", [1, 64, 1000, 16384, 1 << 20, 16 << 20])
def test_size_bins(tb, small):
    with tb.Context(0, tb.options(small_max_bytes=small)) as c:
        layout = workloads.random_batch(5, 1500, 100000, 512 * MiB, align=4)
        run_layout(tb, c, layout, 6, src_shift=1)


@pytest.mark.parametrize("ce_min", [1, 16384, 1 << 20])
def test_copy_engine_routing(tb, ce_min):
    """Descriptors of at least ce_min_bytes go to the copy engines on a
    forked stream, the rest to the kernel; the result is the same."""
    import torch
    with tb.Context(0, tb.options(ce_min_bytes=ce_min)) as c:
        layout = workloads.random_batch(77, 500, 2 << 20, 1024 * MiB, align=1)
        st = torch.cuda.Stream()
        stats = run_layout(tb, c, layout, 78, stream=st)
        routed = int(((layout.lens >= ce_min) & (layout.lens > 0)).sum())
        assert stats["ce_copies"] == routed and routed > 0
        assert stats["warp_items"] + routed <= stats["descs"]


def test_copy_engine_routing_head_sliced(tb):
    with tb.Context(0, tb.options(ce_min_bytes=1 << 20)) as c:
        stats = run_layout(tb, c, workloads.batch_head_sliced(), 104)
        assert stats["ce_copies"] == 20 and stats["warp_items"] == 47520


def test_two_contexts_on_two_threads(tb):
    """Two host threads, each with its own context and stream, submit
    batches (and reduce-copies) at the same time; every result is exact.
    Contexts share only the library's per-device launch caches."""
    import threading
    import torch
    layouts = [workloads.random_batch(80 + t, 3000, 40000, 128 * MiB, align=1) for t in range(2)]
    pools = []
    for t, lay in enumerate(layouts):
        src_h = workloads.random_bytes(lay.src_pool_bytes, 90 + t)
        pools.append((src_h, to_dev(src_h), torch.zeros(lay.dst_pool_bytes, dtype=torch.uint8,
                                                        device="cuda")))
    red = [(dev_bytes_f(1 << 22, 3.0), dev_bytes_f(1 << 22, 0.0)) for _ in range(2)]
    torch.cuda.synchronize()
    errors = []

    def work(t):
        try:
            with tb.Context(0) as c:
                st = torch.cuda.Stream()
                src_h, src_d, dst_d = pools[t]
                desc = layouts[t].descriptors(src_d.data_ptr(), dst_d.data_ptr())
                for _ in range(20):
                    c.batch_copy(desc, st)
                    c.reduce_copy([red[t][0], red[t][0]], red[t][1], 1 << 22, 0, st)
                st.synchronize()
        except Exception as e:  # reported in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t, lay in enumerate(layouts):
        src_h, _, dst_d = pools[t]
        exp = np.zeros(lay.dst_pool_bytes, dtype=np.uint8)
        oracle.apply_batch(exp, src_h, lay.src_off, lay.dst_off, lay.lens)
        assert oracle.first_mismatch(to_host(dst_d), exp) == -1
        assert np.all(to_host(red[t][1]).view(np.float32) == 6.0)


def dev_bytes_f(nbytes, value):
    import torch
    return torch.full((nbytes // 4,), value, dtype=torch.float32, device="cuda")


def test_user_stream_ordering(tb, ctx):
    """The copy runs after earlier work on the caller's stream: a fill queued
    just before on the same stream is what gets copied."""
    import torch
    st = torch.cuda.Stream()
    src = torch.zeros(8 * MiB, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(8 * MiB, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        big = torch.empty(256 * MiB, dtype=torch.uint8, device="cuda")
        for _ in range(4):
            big.fill_(1)               # keep the stream busy for a while
        src.fill_(0xAB)
    desc = np.array([[src.data_ptr(), dst.data_ptr(), 8 * MiB]], dtype=np.uint64)
    ctx.batch_copy(desc, st)
    st.synchronize()
    assert np.all(to_host(dst) == 0xAB)


def test_capturing_stream_is_refused(tb, ctx):
    """tb_batch_copy on a stream that is capturing a CUDA graph returns
    TB_ENOTSUP with nothing queued: the capture goes on, the graph replays
    what else was captured (here one cudaMemcpyAsync per copy, tb_copy_each),
    and the context copies the batch normally once capture is over."""
    import torch
    layout = workloads.random_batch(71, 200, 4096, 8 * MiB, align=1, min_len=1)
    src_h = workloads.random_bytes(layout.src_pool_bytes, 72)
    dst_h = workloads.random_bytes(layout.dst_pool_bytes, 73)
    src_d, dst_d = to_dev(src_h), to_dev(dst_h)
    desc = np.stack([np.uint64(src_d.data_ptr()) + layout.src_off,
                     np.uint64(dst_d.data_ptr()) + layout.dst_off, layout.lens], axis=1)
    exp = dst_h.copy()
    oracle.apply_batch(exp, src_h, layout.src_off, layout.dst_off, layout.lens)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        s = torch.cuda.current_stream()
        with pytest.raises(tb.TBError) as err:
            ctx.batch_copy(desc, s)
        assert err.value.code == tb.TB_ENOTSUP
        ctx.copy_each(desc, s)
    assert np.array_equal(to_host(dst_d), dst_h)     # capture ran nothing
    graph.replay()
    torch.cuda.synchronize()
    assert oracle.first_mismatch(to_host(dst_d), exp) == -1
    del graph
    dst_d.copy_(to_dev(dst_h))
    st = torch.cuda.Stream()
    ctx.batch_copy(desc, st)
    st.synchronize()
    assert oracle.first_mismatch(to_host(dst_d), exp) == -1


def test_bad_descriptors(tb, ctx):
    import torch
    d = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(tb.TBError) as e:
        ctx.batch_copy(np.array([[0, d.data_ptr(), 8]], dtype=np.uint64))
    assert e.value.code == tb.TB_EINVAL
    with pytest.raises(tb.TBError):
        ctx.batch_copy(np.array([[d.data_ptr(), 2**64 - 4, 8]], dtype=np.uint64))
    ctx.batch_copy(np.array([[0, 0, 0]], dtype=np.uint64))         # len 0 is a no-op
    ctx.batch_copy(np.zeros((0, 3), dtype=np.uint64))


@pytest.mark.parametrize("k", [1, 2, 3])
def test_batch_min_copies(tb, k):
    """batch_min_copies = 3 (the RFC's MC_HIP_BATCH_COPY_MIN): batches of 1
    or 2 copies go out as one cudaMemcpyAsync each, 3 or more as a kernel;
    the bytes are the same."""
    with tb.Context(0, tb.options(batch_min_copies=3)) as c:
        layout = workloads.random_batch(200 + k, k, 70000, 8 * MiB, align=1, min_len=1)
        st = run_layout(tb, c, layout, 210 + k)
        assert st["descs"] == k
        assert (st["launches"], st["ce_copies"]) == ((0, k) if k < 3 else (1, 0))


def test_check_overlap(tb):
    """check_overlap = 1: a batch whose copies overlap is rejected before
    any launch (the destination pool is untouched); a clean one copies."""
    import torch
    with tb.Context(0, tb.options(check_overlap=1)) as c:
        run_layout(tb, c, workloads.random_batch(71, 2000, 5000, 64 * MiB, align=1), 72)
        src = torch.arange(256, dtype=torch.uint8, device="cuda").repeat(4096)
        dst = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        s0, d0 = src.data_ptr(), dst.data_ptr()
        for rows in ([[s0, d0, 4096], [s0 + 8192, d0 + 4000, 4096]],      # dst over dst
                     [[s0, d0, 4096], [d0 + 100, d0 + 8192, 64]]):        # dst over a source
            with pytest.raises(tb.TBError) as e:
                c.batch_copy(np.array(rows, dtype=np.uint64))
            assert e.value.code == tb.TB_EINVAL and "overlap" in str(e.value)
        assert int(dst.count_nonzero().item()) == 0


def test_slot_wait_deadline(tb):
    """With one slot, a second batch waits for the first launch; a 1 ns limit
    expires first and the call returns TB_ETIMEOUT instead of blocking."""
    import torch
    with tb.Context(0, tb.options(num_slots=1, wait_timeout_ns=1)) as c:
        layout = workloads.random_batch(3, 40000, 16384, 1024 * MiB, align=64)
        src = torch.empty(1024 * MiB, dtype=torch.uint8, device="cuda")
        dst = torch.empty(1024 * MiB, dtype=torch.uint8, device="cuda")
        desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            for _ in range(8):
                src.fill_(3)           # the launch queues behind these
        c.batch_copy(desc, st)
        with pytest.raises(tb.TBError) as e:
            c.batch_copy(desc, st)
        assert e.value.code == tb.TB_ETIMEOUT
        st.synchronize()
        c.batch_copy(desc, st)         # the slot is free again
        st.synchronize()


def test_failed_slot_wait_mid_batch_keeps_stream_order(tb):
    """A batch of two slots' worth (slot_items = 1024, one slot) whose wait
    for the second slot expires behind a busy stream: TB_ETIMEOUT; the first
    slot's launch and its copy-engine copy stay queued and copy their part,
    work queued on the stream after the failed call sees that copy-engine
    copy done, and the second part is not copied."""
    import torch
    n = 2048
    lens = np.full(n, 512, dtype=np.uint64)
    lens[5] = lens[1500] = 2 * MiB                     # routed to the copy engines
    off = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.uint64)
    pool = int(lens.sum())
    src_h = workloads.random_bytes(pool, 81)
    dst_h = workloads.random_bytes(pool, 82)
    src_d, dst_d = to_dev(src_h), to_dev(dst_h)
    desc = np.stack([np.uint64(src_d.data_ptr()) + off, np.uint64(dst_d.data_ptr()) + off, lens],
                    axis=1)
    busy = torch.empty(256 * MiB, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with tb.Context(0, tb.options(num_slots=1, slot_items=1024, wait_timeout_ns=1,
                                  ce_min_bytes=1 * MiB)) as c:
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            for _ in range(8):
                busy.fill_(3)                          # the first launch queues behind these
        with pytest.raises(tb.TBError) as e:
            c.batch_copy(desc, st)
        assert e.value.code == tb.TB_ETIMEOUT
        with torch.cuda.stream(st):
            probe = dst_d[int(off[5]):int(off[5]) + 2 * MiB].clone()
        st.synchronize()
    assert np.array_equal(to_host(probe), src_h[int(off[5]):int(off[5]) + 2 * MiB])
    exp = dst_h.copy()
    oracle.apply_batch(exp, src_h, off[:1024], off[:1024], lens[:1024])
    assert oracle.first_mismatch(to_host(dst_d), exp) == -1


def test_pipeline_wait_expiry_is_reported(tb):
    """kernel_wait_ns = 0: the bulk pipeline of the long copies cannot meet
    its first wait; the kernel records it in the slot's status word and
    stops its pipeline after the issued loads land.  The failure comes back
    as TB_ETIMEOUT from tb_last_batch_kernel_ms and from the next call that
    reuses the slot; a context with the default limit then copies the same
    batch bit-exactly."""
    import torch
    with tb.Context(0, tb.options(kernel_wait_ns=0, time_kernels=1, num_slots=1)) as c:
        layout = workloads.random_batch(61, 40, 4 * MiB, 256 * MiB, align=64, min_len=1 * MiB)
        src = torch.zeros(256 * MiB, dtype=torch.uint8, device="cuda")
        dst = torch.zeros(256 * MiB, dtype=torch.uint8, device="cuda")
        desc = layout.descriptors(src.data_ptr(), dst.data_ptr())
        c.batch_copy(desc)
        with pytest.raises(tb.TBError) as e:
            c.last_batch_kernel_ms()
        assert e.value.code == tb.TB_ETIMEOUT
        with pytest.raises(tb.TBError) as e:
            c.batch_copy(desc)                   # the slot reports it once
        assert e.value.code == tb.TB_ETIMEOUT
    with tb.Context(0) as c:
        run_layout(tb, c, layout, 62)


@pytest.mark.parametrize("shape", [1, 2])
@pytest.mark.parametrize("seed", range(3))
def test_short_only_shapes(tb, shape, seed):
    """Each k_short shape forced on batches of short copies only: any byte
    alignment (src and dst equal modulo 16 go through the warp's ring, other
    pairs through the shifted path), 0 to 16 KiB, and the 3840-page shape;
    whole pools byte-exact against the oracle."""
    with tb.Context(0, tb.options(batch_short_shape=shape)) as c:
        run_layout(tb, c, workloads.random_batch(700 + seed, 5000, 16384, 64 * MiB, align=1), seed)
        run_layout(tb, c, workloads.random_batch(710 + seed, 3000, 4096, 16 * MiB, align=16),
                   seed + 5, src_shift=seed, dst_shift=seed)
        st = run_layout(tb, c, workloads.batch_index_pages(seed), seed + 9)
        assert st["warp_items"] == 3840


@pytest.mark.parametrize("shape,n", [(2, 20000), (1, 500), (2, 1)])
def test_short_only_shapes_claims_and_few_copies(tb, shape, n):
    """A forced shape past the copies its warps take by index (shape 2 with
    20,000 copies: the rest claimed from the counter), with fewer copies
    than warps (shape 1, 500 copies), and a single copy."""
    with tb.Context(0, tb.options(batch_short_shape=shape)) as c:
        layout = workloads.random_batch(720 + n, n, 4096, 96 * MiB, align=1, min_len=1)
        st = run_layout(tb, c, layout, n)
        assert st["warp_items"] == n


# ---------------------------------------------------------------------------
# Beside compute (Mooncake RFC, "Design of #5040", interference with compute
# on the sending GPU; "Motivation", small copies under a bf16 GEMM)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("priority", [0, -1])
def test_batches_exact_beside_a_gemm_loop(tb, ctx, priority):
    """The 3840-page batch and the 47,540-descriptor batch (its layout in
    1 GiB pools) copied on a normal- or high-priority stream while a bf16
    GEMM loop runs on another stream: both whole pools byte-exact against
    the oracle, and the GEMM loop still running when the batches were
    enqueued."""
    import torch
    layouts = [workloads.batch_index_pages(), workloads.batch_head_sliced(pool_bytes=1 << 30)]
    pools = []
    for j, lay in enumerate(layouts):
        src_h = workloads.random_bytes(lay.src_pool_bytes, 300 + 2 * j)
        dst_h = workloads.random_bytes(lay.dst_pool_bytes, 301 + 2 * j)
        pools.append((src_h, dst_h, to_dev(src_h), to_dev(dst_h)))
    n = 4096
    a = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    b = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
    gemm_s = torch.cuda.Stream()
    copy_s = torch.cuda.Stream(priority=priority)
    torch.cuda.synchronize()
    done = torch.cuda.Event()
    with torch.cuda.stream(gemm_s):
        for _ in range(600):
            torch.matmul(a, b, out=c)
    done.record(gemm_s)
    for lay, (_, _, src_d, dst_d) in zip(layouts, pools):
        ctx.batch_copy(lay.descriptors(src_d.data_ptr(), dst_d.data_ptr()), copy_s)
    running = not done.query()
    copy_s.synchronize()
    torch.cuda.synchronize()
    assert running
    for lay, (src_h, dst_h, _, dst_d) in zip(layouts, pools):
        exp = dst_h.copy()
        oracle.apply_batch(exp, src_h, lay.src_off, lay.dst_off, lay.lens)
        mm = oracle.first_mismatch(to_host(dst_d), exp)
        assert mm == -1, f"{lay.name}: first differing byte {mm}"


# ---------------------------------------------------------------------------
# Full-size layouts, in the launch configuration the bench times
# ---------------------------------------------------------------------------
def test_index_pages_full(tb, ctx):
    st = run_layout(tb, ctx, workloads.batch_index_pages(), 101)
    assert st["descs"] == 3840 and st["warp_items"] == 3840
    assert st["direct_launches"] == 1        # work list read in place from pinned memory


def test_block_pages_full(tb, ctx):
    st = run_layout(tb, ctx, workloads.batch_block_pages(), 102)
    assert st["descs"] == 7200


def test_head_sliced_full(tb, ctx):
    layout = workloads.batch_head_sliced()
    st = run_layout(tb, ctx, layout, 103)
    assert st["descs"] == 47540 and st["warp_items"] == 47520
    assert st["cta_items"] > 0                     # chunks of the 20 long copies
    assert st["launches"] == 1 and st["direct_launches"] == 0

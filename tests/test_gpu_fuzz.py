"""Seeded random cases over the option space, each compared with the oracle.

Reduce-copy: 0-16 sources, 0-300,000 elements, byte offsets of any 4-byte
class, engine, vector width, block size, unroll, sub-executor layout and
programmatic launch drawn at random; a combination the library does not
support must be refused with TB_ENOTSUP, everything else must be bit-exact
with dstReference and leave the guard bytes around dst untouched.
Batched copy: 0-3000 copies of 0 B - 256 KiB at any byte alignment, with the
short/long threshold, slot size and count, copy-count and copy-engine
routing, the short-only kernel shape and a cap on the CTAs drawn at random;
the whole destination pool must equal the oracle's apply of the batch.
DMA executor: one source of 1-300,000 elements in K = 1-9 rotation slices
filled with different patterns, byte offset, warm-up, iterations, graph or
gate drawn at random; dst must equal the slice of the last iteration.
Kernel executor with rotation: the same over 1-16 sources, with the engine,
programmatic launch and sub-executors drawn too; dst must equal
dstReference of the last iteration's slices.
The seeds are fixed, so a failure names its case."""
import numpy as np
import pytest

import oracle
from copy_reduce_dst_gb300 import workloads
from gpu_helpers import dev_bytes, finite_floats, to_dev, to_host

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


def _reduce_case(seed):
    g = np.random.default_rng(1000 + seed)
    n_src = int(g.choice([0, 1, 1, 2, 3, 3, 4, 5, 8, 9, 16]))
    n = int(g.choice([0, 1, 3, 1000, int(g.integers(1, 300000))]))
    common = int(g.choice([0, 4, 8, 16, 32, 48]))
    offs = [common if g.random() < 0.8 else int(g.integers(0, 16)) * 4 for _ in range(n_src)]
    dst_off = common if g.random() < 0.8 else int(g.integers(0, 16)) * 4
    opts = dict(reduce_engine=int(g.choice([0, 0, 1, 2])),
                vec_bytes=int(g.choice([0, 0, 4, 16, 32])),
                block_threads=int(g.choice([0, 128, 256, 512])),
                unroll=int(g.choice([0, 1, 2, 4])),
                ctas_per_subexec=int(g.choice([0, 0, 1, 2])),
                use_pdl=int(g.choice([0, 1])))
    subexec = int(g.choice([0, 0, 1, 4, 7, 32, 200]))
    return g, n_src, n, offs, dst_off, opts, subexec


@pytest.mark.parametrize("seed", range(200))
def test_reduce_fuzz(tb, seed):
    g, n_src, n, offs, dst_off, opts, subexec = _reduce_case(seed)
    srcs = [finite_floats(g, n) for _ in range(n_src)]
    nbytes = 4 * n
    pad = 256
    bufs = []
    for a, off in zip(srcs, offs):
        b = dev_bytes(nbytes + off + pad, fill=0x5A)
        if nbytes:
            b[off:off + nbytes].copy_(to_dev(a))
        bufs.append((b, off))
    dst = dev_bytes(nbytes + dst_off + pad, fill=0xC3)
    with tb.Context(0, tb.options(**opts)) as c:
        try:
            c.reduce_copy([b.data_ptr() + off for b, off in bufs], dst.data_ptr() + dst_off,
                          nbytes, subexec)
        except tb.TBError as e:
            # only a combination the library cannot serve may be refused
            assert e.code == tb.TB_ENOTSUP, (seed, opts, e)
            assert opts["reduce_engine"] == 2 or opts["vec_bytes"] in (16, 32)
            return
    got = to_host(dst)
    exp = oracle.dst_reference(srcs, n=n)
    body = got[dst_off:dst_off + nbytes]
    if nbytes:
        mm = oracle.first_mismatch(body.view(np.uint32), exp.view(np.uint32))
        assert mm == -1, f"seed {seed} {opts} subexec {subexec}: first mismatch at {mm}"
    assert np.all(got[:dst_off] == 0xC3) and np.all(got[dst_off + nbytes:] == 0xC3)


@pytest.mark.parametrize("seed", range(100))
def test_batch_fuzz(tb, seed):
    import torch
    g = np.random.default_rng(5000 + seed)
    n = int(g.choice([0, 1, 2, 17, int(g.integers(1, 3000))]))
    long_frac = float(g.choice([0.0, 0.01, 0.2]))
    lens = np.where(g.random(n) < long_frac, g.integers(16385, 1 << 18, n),
                    g.integers(0, 16385, n)).astype(np.uint64)
    pool = int(lens.sum()) * 2 + (4 << 20)
    gen = workloads.rng(6000 + seed)
    so = workloads.scatter_offsets(gen, lens, 0, pool, 1)
    do = workloads.scatter_offsets(gen, lens, 0, pool, 1)
    opts = dict(small_max_bytes=int(g.choice([64, 4096, 16384, 1 << 20])),
                slot_items=int(g.choice([1024, 4096, 65536])),
                num_slots=int(g.choice([1, 2, 4])),
                batch_min_copies=int(g.choice([0, 0, 3])),
                ce_min_bytes=int(g.choice([0, 0, 0, 1 << 17])),
                # own generator, so the cases above stay as they were
                batch_short_shape=int(np.random.default_rng(9000 + seed).choice([0, 0, 1, 2])),
                batch_max_ctas=int(np.random.default_rng(9500 + seed).choice([0, 0, 0, 1, 7, 64])))
    src_h = workloads.random_bytes(pool, 7000 + seed)
    dst_h = workloads.random_bytes(pool, 8000 + seed)
    src_d, dst_d = to_dev(src_h), to_dev(dst_h)
    desc = np.stack([np.uint64(src_d.data_ptr()) + so, np.uint64(dst_d.data_ptr()) + do, lens],
                    axis=1) if n else np.zeros((0, 3), np.uint64)
    with tb.Context(0, tb.options(**opts)) as c:
        st = torch.cuda.Stream()
        c.batch_copy(desc, st)
        st.synchronize()
        stats = c.last_batch_stats()
    assert stats["descs"] == int((lens > 0).sum())
    exp = dst_h.copy()
    oracle.apply_batch(exp, src_h, so, do, lens)
    mm = oracle.first_mismatch(to_host(dst_d), exp)
    assert mm == -1, f"seed {seed} {opts} n {n}: first differing byte {mm}"


@pytest.mark.parametrize("seed", range(30))
def test_dma_executor_fuzz(tb, seed):
    g = np.random.default_rng(11000 + seed)
    n = int(g.choice([1, 3, 64, int(g.integers(1, 300000))]))
    nb = 4 * n
    K = int(g.integers(1, 10))
    iters = int(g.integers(1, 12))
    off = int(g.choice([0, 0, 4, 20, 256]))
    opts = dict(byte_offset=off, warmup=int(g.integers(0, 4)), use_graph=int(g.choice([0, 1])),
                use_gate=int(g.choice([0, 1])))
    plan = tb.rotation_plan(nb, K * nb if K > 1 else 0, off)
    assert plan.K == K
    src = dev_bytes(plan.alloc_bytes, fill=0x11)
    slices = [finite_floats(g, n) for _ in range(K)]
    for j, a in enumerate(slices):
        start = off + j * plan.slice_stride
        src[start:start + nb].copy_(to_dev(a))
    dst = dev_bytes(nb + off + 128, fill=0xC3)
    last = oracle.slice_for_iteration(iters - 1, K)
    with tb.Context(0, tb.options(**opts)) as c:
        r = c.run_transfer([src], dst, nb, iters=iters, rotate_bytes=K * nb if K > 1 else 0,
                           expected=slices[last], executor=tb.TB_EXEC_DMA)
    assert r["mismatch_index"] == -1 and r["executor"] == tb.TB_EXEC_DMA, (seed, opts)
    got = to_host(dst)
    assert np.array_equal(got[off:off + nb].view(np.uint32), slices[last].view(np.uint32))
    assert np.all(got[:off] == 0xC3) and np.all(got[off + nb:] == 0xC3)


@pytest.mark.parametrize("seed", range(40))
def test_rotation_fuzz(tb, seed):
    """The kernel executor with rotation: 1-16 sources, each a K-slice
    allocation (K = 1-6) whose slices hold different random floats; byte
    offset, warm-up, iterations, graph, gate, programmatic launch, engine and
    sub-executors drawn at random.  dst must equal dstReference of every
    source's slice (iters - 1) mod K, guard bytes untouched."""
    g = np.random.default_rng(13000 + seed)
    n_src = int(g.choice([1, 2, 3, 3, 4, 5, 8, 16]))
    n = int(g.choice([1, 3, 64, 1000, int(g.integers(1, 200000))]))
    nb = 4 * n
    K = int(g.integers(1, 7))
    iters = int(g.integers(1, 9))
    off = int(g.choice([0, 0, 4, 20, 256]))
    opts = dict(byte_offset=off, warmup=int(g.integers(0, 4)), use_graph=int(g.choice([0, 1])),
                use_gate=int(g.choice([0, 1])), use_pdl=int(g.choice([0, 1])),
                reduce_engine=int(g.choice([0, 0, 1, 2])),
                ctas_per_subexec=int(g.choice([0, 0, 1])))
    subexec = int(g.choice([0, 0, 1, 4]))
    rotate = K * nb if K > 1 else 0
    plan = tb.rotation_plan(nb, rotate, off)
    assert plan.K == K
    slices = [[finite_floats(g, n) for _ in range(K)] for _ in range(n_src)]
    srcs = []
    for per_src in slices:
        b = dev_bytes(plan.alloc_bytes, fill=0x11)
        for j, a in enumerate(per_src):
            start = off + j * plan.slice_stride
            b[start:start + nb].copy_(to_dev(a))
        srcs.append(b)
    dst = dev_bytes(nb + off + 128, fill=0xC3)
    last = oracle.slice_for_iteration(iters - 1, K)
    exp = oracle.dst_reference([s[last] for s in slices])
    with tb.Context(0, tb.options(**opts)) as c:
        try:
            r = c.run_transfer(srcs, dst, nb, num_subexec=subexec, iters=iters,
                               rotate_bytes=rotate, expected=exp)
        except tb.TBError as e:
            # every case here shares one alignment, so nothing may be refused
            raise AssertionError((seed, opts, e)) from e
    assert r["mismatch_index"] == -1 and r["K"] == K and r["iters"] == iters, (seed, opts)
    got = to_host(dst)
    mm = oracle.first_mismatch(got[off:off + nb].view(np.uint32), exp.view(np.uint32))
    assert mm == -1, f"seed {seed} {opts} subexec {subexec}: first mismatch at {mm}"
    assert np.all(got[:off] == 0xC3) and np.all(got[off + nb:] == 0xC3)

"""GPU parity of the reduce-copy path (through the C ABI) against the oracle.

Bar: bit-exact.  Every float add on both sides is one IEEE binary32
round-to-nearest-even add taken left to right, so dst must equal
dstReference[nSrc] byte for byte (inputs are finite and NaN-free; a NaN's
payload after an add is not fixed by IEEE 754 and is not compared here).
"""
import numpy as np
import pytest

import oracle
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


@pytest.fixture(scope="module")
def ctx(tb):
    with tb.Context(0) as c:
        yield c


def reduce_and_compare(tb, ctx, srcs_host, byte_offsets=None, dst_offset=0, num_subexec=0,
                       memset_byte=0):
    """Uploads the sources at the given byte offsets inside padded buffers,
    runs one tb_reduce_copy, and compares dst (and the guard bytes around it)
    with the oracle."""
    n = srcs_host[0].size if srcs_host else 0
    nbytes = 4 * n
    offs = byte_offsets or [0] * len(srcs_host)
    pad = 256
    bufs = []
    for a, off in zip(srcs_host, offs):
        b = dev_bytes(nbytes + off + pad, fill=0x5A)
        b[off:off + nbytes].copy_(to_dev(a)[:nbytes]) if nbytes else None
        bufs.append((b, off))
    dst = dev_bytes(nbytes + dst_offset + pad, fill=0xC3)
    ctx.reduce_copy([b.data_ptr() + off for b, off in bufs], dst.data_ptr() + dst_offset, nbytes,
                    num_subexec)
    got = to_host(dst)
    exp = oracle.dst_reference(srcs_host, n=n, memset_byte=memset_byte)
    body = got[dst_offset:dst_offset + nbytes]
    mm = oracle.first_mismatch(body.view(np.uint32) if nbytes else body, exp.view(np.uint32))
    assert mm == -1, f"first mismatch at element {mm}"
    assert np.all(got[:dst_offset] == 0xC3) and np.all(got[dst_offset + nbytes:] == 0xC3), \
        "write outside dst"


@pytest.mark.parametrize("nsrc", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16])
def test_reduce_parity_source_counts(tb, ctx, nsrc):
    g = np.random.default_rng(100 + nsrc)
    n = 3 * 512 * 4 * 8 + 13          # several tiles plus a ragged tail
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    reduce_and_compare(tb, ctx, srcs)


@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 7, 8, 9, 31, 32, 33, 1000, 4097, 65536 + 3])
def test_reduce_parity_sizes(tb, ctx, n):
    g = np.random.default_rng(n)
    srcs = [finite_floats(g, n) for _ in range(3)]
    if n == 0:
        dst = dev_bytes(64, fill=0xC3)
        ctx.reduce_copy([dev_bytes(16).data_ptr()] * 3, dst.data_ptr(), 0)
        assert np.all(to_host(dst) == 0xC3)
        return
    reduce_and_compare(tb, ctx, srcs)


@pytest.mark.parametrize("offs,doff", [
    ([4, 4, 4], 4),          # co-aligned, head of 7 elements to 32 B
    ([20, 20, 20], 20),      # co-aligned mod 32 with a 3-element head
    ([16, 16, 16], 16),      # co-aligned mod 16, not mod 32
    ([48, 16, 80], 16),      # co-aligned mod 16 only, different mod 32
    ([0, 4, 8], 12),         # no common alignment: scalar path
    ([0, 0, 0], 4),          # dst misaligned against the sources
])
def test_reduce_parity_alignment(tb, ctx, offs, doff):
    g = np.random.default_rng(sum(offs) + doff)
    n = 100003
    srcs = [finite_floats(g, n) for _ in range(3)]
    reduce_and_compare(tb, ctx, srcs, byte_offsets=offs, dst_offset=doff)


@pytest.mark.parametrize("nsrc", [1, 2, 9])
def test_reduce_parity_alignment_many(tb, ctx, nsrc):
    g = np.random.default_rng(7 * nsrc)
    n = 50001
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    reduce_and_compare(tb, ctx, srcs, byte_offsets=[4 * (k % 3) for k in range(nsrc)],
                       dst_offset=8)
    reduce_and_compare(tb, ctx, srcs, byte_offsets=[12] * nsrc, dst_offset=12)


@pytest.mark.parametrize("subexec", [1, 3, 4, 16, 32, 1000, 0])
@pytest.mark.parametrize("ctas", [0, 1, 3])
def test_reduce_parity_subexecutors(tb, subexec, ctas):
    g = np.random.default_rng(subexec * 10 + ctas)
    n = 262144 + 5
    srcs = [finite_floats(g, n) for _ in range(3)]
    with tb.Context(0, tb.options(ctas_per_subexec=ctas)) as c:
        reduce_and_compare(tb, c, srcs, num_subexec=subexec)


@pytest.mark.parametrize("vec,unroll,threads", [(4, 0, 0), (16, 1, 256), (16, 2, 0), (16, 4, 512),
                                               (32, 1, 128), (32, 2, 512), (32, 4, 0), (0, 0, 64)])
@pytest.mark.parametrize("nsrc", [1, 3, 8])
def test_reduce_parity_kernel_shapes(tb, vec, unroll, threads, nsrc):
    g = np.random.default_rng(vec + unroll + threads + nsrc)
    n = 131072 + 9
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    with tb.Context(0, tb.options(vec_bytes=vec, unroll=unroll, block_threads=threads)) as c:
        reduce_and_compare(tb, c, srcs, num_subexec=7)


@pytest.mark.parametrize("nsrc", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 16])
@pytest.mark.parametrize("n,offs,subexec", [
    (5, 0, 0), (2048, 0, 1), (2048 * 7 + 3, 4, 3), (1000003, 20, 0), (262144 * 3 + 17, 16, 32),
    (65536, 12, 1000)])
def test_reduce_parity_bulk_engine(tb, nsrc, n, offs, subexec):
    """The bulk engine (shared-memory stages filled and drained by bulk
    copies) against the oracle: heads, ragged tails, tile edges and
    sub-executor splits."""
    g = np.random.default_rng(nsrc * 1000 + n % 1000 + offs)
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    with tb.Context(0, tb.options(reduce_engine=2)) as c:
        reduce_and_compare(tb, c, srcs, byte_offsets=[offs] * nsrc, dst_offset=offs,
                           num_subexec=subexec)


@pytest.mark.parametrize("nsrc", [2, 3, 4, 5, 6, 7, 8, 12])
def test_bulk_several_waves(tb, nsrc):
    """The bulk form's own grid at 32 MiB per source (plus a 12-byte tail,
    pointers 4 bytes past alignment): whole waves of short-lived CTAs (two
    or three waves from three sources on; one for two), each over about 4
    tiles (8 from six sources), the tile size its source count's; bit-exact
    against the oracle, guard bytes untouched."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = (32 << 20) // 4 + 3
    g = np.random.default_rng(700 + nsrc)
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    with tb.Context(0) as c:
        d = dev_bytes(1 << 20)
        far = d.data_ptr() + (1 << 36) + 4       # planning only: never accessed
        info = c.reduce_plan([d.data_ptr() + 4] * nsrc, far, 4 * n)
        tile = {2: 4096, 3: 3072, 4: 2048, 5: 2048, 6: 2048, 7: 2048, 8: 3072, 12: 2048}[nsrc]
        assert info["engine"] == 2 and info["tile_bytes"] == tile
        assert info["grid"] % sms == 0                                 # whole waves
        reduce_and_compare(tb, c, srcs, byte_offsets=[4] * nsrc, dst_offset=4)


@pytest.mark.parametrize("nsrc", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("subexec", [1, 4, 32, 152])
def test_bulk_deep_pipeline(tb, nsrc, subexec):
    """One CTA per sub-executor and no more CTAs than SMs: each CTA runs the
    bulk pipeline with the deep tiles (16 KiB per source for 2 to 4 sources,
    8 KiB for 5 to 8, 32 KiB for one source) and every stage its shared
    memory holds (3 to 7).  Enough tiles per CTA that the stage ring wraps
    many times, a head and a ragged tail; bit-exact against the oracle."""
    import torch
    if subexec > torch.cuda.get_device_properties(0).multi_processor_count:
        pytest.skip("fewer SMs than sub-executors")
    n = 786432 * 2 + 5
    g = np.random.default_rng(50 + nsrc * 7 + subexec)
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    with tb.Context(0, tb.options(reduce_engine=2, ctas_per_subexec=1)) as c:
        d = dev_bytes(4 * n + 64)
        far = d.data_ptr() + (1 << 36) + 4       # planning only: never accessed
        info = c.reduce_plan([d.data_ptr() + 4] * nsrc, far, 4 * n, subexec)
        tile = 32768 if nsrc == 1 else 16384 if nsrc <= 4 else 8192
        assert info["tile_bytes"] == tile
        stages = info["stages"]
        assert info["smem_bytes"] == 128 + stages * nsrc * tile
        assert info["grid"] == subexec
        assert stages == min(16, (232448 - 128) // (nsrc * tile)) and stages >= 3
        reduce_and_compare(tb, c, srcs, byte_offsets=[4] * nsrc, dst_offset=4,
                           num_subexec=subexec)


@pytest.mark.parametrize("nsrc", [2, 3, 4])
@pytest.mark.parametrize("subexec,n,off", [(1, 262144 * 5 + 7, 4), (5, 1000003, 20),
                                           (32, 65536 * 3 + 1, 0), (152, 4099, 12)])
def test_reduce_parity_wide_ctas(tb, nsrc, subexec, n, off):
    """1024-thread CTAs (one CTA per sub-executor, no more than one per SM)
    against the oracle: heads, ragged tails, several rounds per CTA."""
    import torch
    if subexec > torch.cuda.get_device_properties(0).multi_processor_count:
        pytest.skip("fewer SMs than sub-executors")
    g = np.random.default_rng(700 + nsrc * 10 + subexec)
    srcs = [finite_floats(g, n) for _ in range(nsrc)]
    with tb.Context(0, tb.options(ctas_per_subexec=1)) as c:
        d = dev_bytes(64)
        info = c.reduce_plan([d.data_ptr() + off] * nsrc, d.data_ptr() + off + (1 << 36), 4 * n,
                             subexec)
        assert info["block_threads"] == 1024 and info["grid"] == subexec
        reduce_and_compare(tb, c, srcs, byte_offsets=[off] * nsrc, dst_offset=off,
                           num_subexec=subexec)


def test_plan_fixed_ctas_with_automatic_subexecutors(tb):
    """ctas_per_subexec fixed and numSubExec 0: one sub-executor per CTA of
    the library's grid, for both forms (not a single CTA)."""
    d = dev_bytes(64)
    p = d.data_ptr()
    far = p + (1 << 36)            # planning only: never accessed
    for engine in (1, 2):
        with tb.Context(0, tb.options(reduce_engine=engine, ctas_per_subexec=1)) as c:
            info = c.reduce_plan([p] * 3, far, 256 << 20, 0)
            assert info["engine"] == engine
            assert info["grid"] == info["num_subexec"] and info["grid"] >= 152


def test_reduce_plan_engine_choice(tb, ctx):
    # planning only: the addresses are never accessed; dst lies far away
    d = dev_bytes(1 << 20)
    p = d.data_ptr()
    far = p + (1 << 36)
    big = 32 << 20
    MB = 1 << 20
    three = [p, p + 4096, p + 8192]
    info = ctx.reduce_plan(three, far, 2 * big)
    assert info["engine"] == 2 and info["vec_bytes"] == 16       # bulk where it applies
    assert (info["tile_bytes"], info["stages"]) == (3072, 3)      # short tiles, CTAs share SMs
    assert info["smem_bytes"] == 128 + 3 * 3 * 3072
    assert [ctx.reduce_plan([p] * n, far, 2 * big)["tile_bytes"] for n in range(2, 9)] \
        == [4096, 3072, 2048, 2048, 2048, 2048, 3072]
    relay = ctx.reduce_plan([p], far, 2 * big)
    assert (relay["tile_bytes"], relay["stages"]) == (32768, 3)
    vec = ctx.reduce_plan([p] * 16, far, 2 * big)
    assert vec["engine"] == 1 and (vec["tile_bytes"], vec["stages"]) == (0, 0)
    assert [ctx.reduce_plan([p] * n, far, m)["engine"]            # nine to sixteen
            for n in (9, 12, 14, 15, 16) for m in (MB - 256, MB, 32 * MB - 256, 32 * MB)] \
        == [1, 2, 2, 2] * 3 + [1, 2, 2, 1] * 2
    assert [ctx.reduce_plan([p] * n, far, 8 * MB)["tile_bytes"] for n in (12, 13, 16)] \
        == [2048, 1024, 1024]
    assert [ctx.reduce_plan([p] * 5, far, m)["engine"]            # five: from 4 MiB
            for m in (4 * MB - 256, 4 * MB, 256 * MB)] == [1, 2, 2]
    assert [ctx.reduce_plan([p] * n, far, m)["engine"]            # six to eight: from 3 MiB
            for n in (6, 8) for m in (3 * MB - 256, 3 * MB, 256 * MB)] == [1, 2, 2] * 2
    assert ctx.reduce_plan(three, far, 8 * MB)["engine"] == 2     # three: from 8 MiB
    assert ctx.reduce_plan(three, far, 8 * MB - 256)["engine"] == 1
    two = three[:2]                                               # two: from 12 MiB
    assert [ctx.reduce_plan(two, far, m)["engine"]
            for m in (8 * MB, 12 * MB - 256, 12 * MB, 40 * MB, 256 * MB)] == [1, 1, 2, 2, 2]
    one = 12 << 20
    assert ctx.reduce_plan([p], far, one)["engine"] == 2          # one source: from 12 MiB
    assert ctx.reduce_plan([p], far, one - 256)["engine"] == 1
    four = three + [p + 12288]                                    # four: from 6 MiB
    assert [ctx.reduce_plan(four, far, m)["engine"]
            for m in (4 * MB, 6 * MB - 256, 6 * MB, 32 * MB, 48 * MB, 256 * MB)] \
        == [1, 1, 2, 2, 2, 2]
    info = ctx.reduce_plan([p] * 5, far, 4096)
    assert info["engine"] == 1 and info["vec_bytes"] == 32       # more than 4 sources
    info = ctx.reduce_plan([p + 4, p + 8], far, 4096)
    assert info["engine"] == 1 and info["vec_bytes"] == 4        # no common alignment
    info = ctx.reduce_plan([p + 4, p + 4100], far + 4, big)
    assert info["engine"] == 2 and info["head_elems"] == 3       # head to 16 bytes
    assert info["head_elems"] + 4 * info["body_vectors"] + info["tail_elems"] == big // 4
    with tb.Context(0, tb.options(vec_bytes=32)) as c:
        info = c.reduce_plan([p], far, 4096)
        assert info["engine"] == 1 and info["vec_bytes"] == 32


def test_engine_choice_one_cta_per_subexecutor(tb):
    """With one CTA per sub-executor and no more CTAs than SMs, large
    transfers of 2 to 4 sources take the vector form in 1024-thread CTAs
    with 32-byte vectors (two per source in flight, one for 4 sources); one
    source keeps the bulk form with its deep pipeline."""
    d = dev_bytes(1 << 20)
    p = d.data_ptr()
    far = p + (1 << 36)            # planning only: never accessed
    big = 64 << 20
    with tb.Context(0, tb.options(ctas_per_subexec=1)) as c:
        for n, engine in ((1, 2), (2, 1), (3, 1), (4, 1)):
            info = c.reduce_plan([p] * n, far, big, 32)
            assert info["engine"] == engine and info["grid"] == 32
            if engine == 1:
                assert info["vec_bytes"] == 32 and info["block_threads"] == 1024
                assert info["unroll"] == (2 if n <= 3 else 1)
            else:
                assert info["smem_bytes"] > 128 + 3 * n * (32768 if n == 1 else 8192)
        assert c.reduce_plan([p] * 3, far, big, 1000)["engine"] == 2  # CTAs share SMs
    with tb.Context(0) as c:
        assert c.reduce_plan([p] * 3, far, big, 32)["engine"] == 2    # the grid shared


def test_vector_grid_follows_the_work(tb, ctx):
    """The vector form launches one CTA per round of work (block_threads x
    unroll vectors), at least one per SM and at most one full wave; a small
    transfer gives every CTA its own range, a large one deals whole rounds
    over one range; its block size keeps the most threads resident; fixed
    sub-executor counts keep their grids."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d = dev_bytes(64 << 20)
    p = d.data_ptr()
    with tb.Context(0, tb.options(reduce_engine=1)) as vec:
        infos = [vec.reduce_plan([p], p + (32 << 20), nb)
                 for nb in (4096, 4 << 20, 16 << 20, 24 << 20)]
    for info in infos:
        assert info["engine"] == 1
        rounds = -(-info["body_vectors"] // (info["block_threads"] * info["unroll"]))
        assert info["grid"] >= sms and (info["grid"] == sms or info["grid"] <= rounds)
    small = ctx.reduce_plan([p], p + (32 << 20), 4 << 20)
    assert small["grid"] == sms and small["num_subexec"] == sms    # every CTA takes a part
    assert ctx.reduce_plan([p], p + (32 << 20), 4 << 20, 1000)["grid"] == 1000
    with tb.Context(0, tb.options(reduce_engine=1)) as c:
        far = p + (1 << 36)                                          # planning only
        big = c.reduce_plan([p] * 3, far, 128 << 20)
        assert big["num_subexec"] == 1 and big["grid"] >= sms        # one range, whole rounds
        five = c.reduce_plan([p] * 5, far, 128 << 20)
        assert five["block_threads"] == 256                           # more threads resident


def test_bulk_engine_limits(tb):
    d = dev_bytes(1 << 16)
    with tb.Context(0, tb.options(reduce_engine=2)) as c:
        with pytest.raises(tb.TBError) as e:
            c.reduce_copy([d.data_ptr()] * 17, d.data_ptr() + 8192, 256)   # 17 sources
        assert e.value.code == tb.TB_EINVAL
        with pytest.raises(tb.TBError) as e:
            c.reduce_copy([d.data_ptr() + 4], d.data_ptr() + 8192, 256)   # no common 16 B
        assert e.value.code == tb.TB_ENOTSUP


@pytest.mark.parametrize("byte", [0x00, 0xA5])
def test_zero_sources_is_memset(tb, byte):
    with tb.Context(0, tb.options(memset_byte=byte)) as c:
        for n, doff in ((1, 0), (77777, 4), (4096, 20)):
            dst = dev_bytes(4 * n + doff + 64, fill=0x11)
            c.reduce_copy([], dst.data_ptr() + doff, 4 * n)
            got = to_host(dst)
            assert np.all(got[doff:doff + 4 * n] == byte)
            assert np.all(got[:doff] == 0x11) and np.all(got[doff + 4 * n:] == 0x11)


def test_one_source_copies_bits(tb, ctx):
    bits = np.array([0x80000000, 0x7FC00001, 0xFF800001, 0x7FA00000, 0x00000001, 0x807FFFFF,
                     0x7F800000, 0xFF800000] * 5001, dtype=np.uint32)
    reduce_and_compare(tb, ctx, [bits.view(np.float32)])
    reduce_and_compare(tb, ctx, [bits.view(np.float32)], byte_offsets=[4], dst_offset=12)


def test_left_to_right_association(tb, ctx):
    one = np.ones(1000, np.float32)
    eps = np.full(1000, 2.0**-24, np.float32)
    reduce_and_compare(tb, ctx, [one, eps, eps])
    reduce_and_compare(tb, ctx, [eps, eps, one])


def test_bad_arguments(tb, ctx):
    d = dev_bytes(64)
    with pytest.raises(tb.TBError) as e:
        ctx.reduce_copy([d.data_ptr()], d.data_ptr() + 32, 6)          # not a multiple of 4
    assert e.value.code == tb.TB_EINVAL
    with pytest.raises(tb.TBError):
        ctx.reduce_copy([d.data_ptr() + 2], d.data_ptr() + 32, 8)      # misaligned
    with pytest.raises(tb.TBError):
        ctx.reduce_copy([d.data_ptr()] * 17, d.data_ptr(), 8)          # too many sources
    with pytest.raises(tb.TBError):
        ctx.reduce_copy([0], d.data_ptr(), 8)                          # null source
    for src_off, dst_off in ((0, 0), (16, 0), (0, 16), (0, 28)):         # dst overlaps a source
        with pytest.raises(tb.TBError) as e:
            ctx.reduce_copy([d.data_ptr() + 32, d.data_ptr() + src_off], d.data_ptr() + dst_off, 32)
        assert e.value.code == tb.TB_EINVAL
    ctx.reduce_copy([d.data_ptr(), d.data_ptr()], d.data_ptr() + 32, 32)  # sources may alias


# ---------------------------------------------------------------------------
# Source patterns written by the library's fill kernels
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("k", [0, 1, 2, 15])
def test_fill_default_pattern(tb, ctx, k):
    n = 383 * 1000 + 77
    d = dev_bytes(4 * n + 4)
    ctx.fill_source(d.data_ptr() + 4, 4 * n, tb.default_pattern(), k)
    got = to_host(d, 4 * n, 4).view(np.float32)
    assert oracle.first_mismatch(got, oracle.prepare_reference(n, k)) == -1


@pytest.mark.parametrize("pct,k,n", [((40, 20, 0, 20, 20), 0, 16 * 20000),
                                     ((40, 20, 0, 20, 20), 1, 16 * 3000 + 7),
                                     ((0, 25, 25, 25, 25), 2, 16 * 999 + 15),
                                     ((100, 0, 0, 0, 0), 0, 33)])
def test_fill_compress_pattern(tb, ctx, pct, k, n):
    d = dev_bytes(4 * n)
    ctx.fill_source(d, 4 * n, tb.compress_pattern(pct, 0x5EED), k)
    got = to_host(d, 4 * n).view(np.uint32)
    exp = oracle.fill_compress(n, pct, 0x5EED, k).view(np.uint32)
    assert oracle.first_mismatch(got, exp) == -1


def test_fill_repeat_pattern(tb, ctx):
    vals = [1.5, -2.0, 0.25, 7.0, -0.0]
    pat, keep = tb.repeat_pattern(vals)
    n = 100001
    d = dev_bytes(4 * n)
    ctx.fill_source(d, 4 * n, pat, 0)
    got = to_host(d).view(np.float32)
    assert oracle.first_mismatch(got, oracle.fill_pattern(n, np.array(vals, np.float32))) == -1


def test_fill_rejects_bad_patterns(tb, ctx):
    d = dev_bytes(64)
    with pytest.raises(tb.TBError):
        ctx.fill_source(d, 64, tb.compress_pattern((50, 0, 0, 0, 0), 1), 0)
    with pytest.raises(tb.TBError):
        ctx.fill_source(d, 62, tb.default_pattern(), 0)


@pytest.mark.parametrize("engine,nsrc", [(1, 2), (1, 3), (1, 4), (1, 5), (1, 8),
                                         (2, 2), (2, 3), (2, 4), (2, 5),
                                         (2, 8)])    # bulk: 1 to 8 sources
def test_multi_source_fill_compress(tb, nsrc, engine):
    """Sources k = 0..N-1 of the fillCompress pattern (every mode, 2B0
    included), written by the library's fill kernel and summed on the GPU,
    against the oracle's patterns and dstReference.  Masks that zero a
    float's exponent byte make tiny and subnormal values, so the sums test
    the left-to-right order and the absence of flush-to-zero."""
    n = 16 * 40000 + 9
    pct = (20, 20, 20, 20, 20)
    refs = [oracle.fill_compress(n, pct, 0xC0FFEE, k) for k in range(nsrc)]
    sub = sum(int(np.count_nonzero((r != 0) & (np.abs(r) < np.float32(1.1754944e-38))))
              for r in refs)
    assert sub > 1000                                   # subnormal inputs present
    exp = oracle.dst_reference(refs)
    with tb.Context(0, tb.options(reduce_engine=engine)) as c:
        srcs = [dev_bytes(4 * n) for _ in range(nsrc)]
        for k, d in enumerate(srcs):
            c.fill_source(d, 4 * n, tb.compress_pattern(pct, 0xC0FFEE), k)
        dst = dev_bytes(4 * n)
        c.reduce_copy(srcs, dst, 4 * n)
        got = to_host(dst).view(np.float32)
        assert oracle.first_mismatch(got, exp) == -1
        # with rotation: 4 slices each, validated after every iteration
        plan = tb.rotation_plan(4 * n, 4 * 4 * n)
        with tb.Context(0, tb.options(reduce_engine=engine, always_validate=1)) as cv:
            rot = [dev_bytes(plan.alloc_bytes) for _ in range(nsrc)]
            for k, d in enumerate(rot):
                cv.fill_source(d, 4 * n, tb.compress_pattern(pct, 0xC0FFEE), k)
            cv.prepare_sources(rot, 4 * n, 4 * 4 * n)
            r = cv.run_transfer(rot, dst, 4 * n, iters=6, rotate_bytes=4 * 4 * n, expected=exp)
            assert r["K"] == 4 and r["mismatch_index"] == -1 and r["engine"] == engine


# ---------------------------------------------------------------------------
# Rotation, timed loop and validation (tb_run_transfer)
# ---------------------------------------------------------------------------
def test_single_transfer_mechanism(tb):
    """PR #365's mechanism check: a 4 MiB transfer at the 256 MiB default
    allocates 268,435,456 B (K = 64) while the prep host-to-device copy stays
    4 MiB; every slice holds slice 0's data; validation passes with rotation
    on, once at the end and after every iteration."""
    nb = 4 * MiB
    n = nb // 4
    plan = tb.rotation_plan(nb, 256 * MiB)
    assert (plan.K, plan.alloc_bytes) == (64, 268435456)
    ref = oracle.prepare_reference(n, 0)
    for always in (0, 1):
        with tb.Context(0, tb.options(always_validate=always)) as c:
            src = dev_bytes(plan.alloc_bytes)
            dst = dev_bytes(nb, fill=0)
            c.upload_sources([src], [ref], nb)
            assert c.prep_h2d_bytes == nb
            c.prepare_sources([src], nb, 256 * MiB)
            assert c.prep_h2d_bytes == nb
            whole = to_host(src).view(np.float32).reshape(64, n)
            for j in range(64):
                assert oracle.first_mismatch(whole[j], ref) == -1, f"slice {j}"
            r = c.run_transfer([src], dst, nb, iters=10, rotate_bytes=256 * MiB, expected=ref)
            assert r["K"] == 64 and r["alloc_bytes"] == 268435456 and r["prep_h2d_bytes"] == nb
            assert r["iters"] == 10 and r["validated"] == 1 and r["mismatch_index"] == -1
            assert len(r["iter_ms"]) == 10 and all(t > 0 for t in r["iter_ms"])
            assert r["graphed"] == (0 if always else 1) and r["gated"] == 0
            assert abs(sum(r["iter_ms"]) - r["total_ms"]) < 1e-3 * r["total_ms"] + 1e-6


@pytest.mark.parametrize("pdl", [1, 0])
@pytest.mark.parametrize("engine,nsrc", [(1, 2), (2, 2), (2, 4), (1, 10)])
def test_back_to_back_launches_read_previous_output(tb, engine, nsrc, pdl):
    """A chain of launches on one stream with no host synchronisation, each
    reading what the launch before it wrote (x_{j+1} = x_j + c_1 + ...).
    With programmatic dependent launch a kernel is scheduled while its
    predecessor drains; its CTAs must still see every byte the predecessor
    wrote, so the chain ends bit-exact with the oracle's."""
    import torch
    n = (24 << 20) // 4 + 7                     # 24 MiB + a ragged tail
    g = np.random.default_rng(300 + 10 * engine + nsrc)
    x0 = finite_floats(g, n, max_exp=120)
    consts = [finite_floats(g, n, max_exp=120) for _ in range(nsrc - 1)]
    with tb.Context(0, tb.options(reduce_engine=engine, use_pdl=pdl)) as c:
        bufs = [to_dev(x0), dev_bytes(4 * n)]
        cd = [to_dev(k) for k in consts]
        st = torch.cuda.Stream()
        torch.cuda.synchronize()
        steps = 9
        for j in range(steps):
            cur, nxt = bufs[j % 2], bufs[(j + 1) % 2]
            c.reduce_copy([cur.data_ptr()] + [k.data_ptr() for k in cd], nxt.data_ptr(), 4 * n,
                          0, st)
        st.synchronize()
        got = to_host(bufs[steps % 2]).view(np.float32)
    exp = x0
    for _ in range(steps):
        exp = oracle.dst_reference([exp] + consts)
    mm = oracle.first_mismatch(got.view(np.uint32), exp.view(np.uint32))
    assert mm == -1, f"first mismatch at element {mm}"


@pytest.mark.parametrize("engine", [1, 2])
def test_captured_chain_reads_previous_output(tb, engine):
    """The same chain captured into one CUDA graph through the caller's
    stream (as the bench's timed loop is): consecutive kernel nodes get
    programmatic edges, and the result is still the serial one."""
    import torch
    n = (16 << 20) // 4 + 3
    g = np.random.default_rng(400 + engine)
    x0 = finite_floats(g, n, max_exp=120)
    c1 = finite_floats(g, n, max_exp=120)
    with tb.Context(0, tb.options(reduce_engine=engine)) as c:
        bufs = [to_dev(x0), dev_bytes(4 * n)]
        cd = to_dev(c1)
        st = torch.cuda.Stream()
        torch.cuda.synchronize()
        steps = 6
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            for j in range(steps):
                c.reduce_copy([bufs[j % 2].data_ptr(), cd.data_ptr()],
                              bufs[(j + 1) % 2].data_ptr(), 4 * n, 0, st)
        bufs[0].copy_(to_dev(x0))             # capture does not run the kernels
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got = to_host(bufs[steps % 2]).view(np.float32)
        del graph
    exp = x0
    for _ in range(steps):
        exp = oracle.dst_reference([exp, c1])
    mm = oracle.first_mismatch(got.view(np.uint32), exp.view(np.uint32))
    assert mm == -1, f"first mismatch at element {mm}"


@pytest.mark.parametrize("graph", [1, 0])
@pytest.mark.parametrize("nsrc,n", [(3, 3 * (1 << 20) + 5), (3, 40000 + 3), (6, 1 << 20)])
def test_early_reads_over_unwritten_slices(tb, graph, nsrc, n):
    """early_reads = 1: successive tb_reduce_copy launches over rotation
    slices that nothing writes, each free to read its sources before the
    launch ahead has finished (the bulk form at 12 MiB, the vector form at
    160 KB): dst holds the sum of the last launch's slices, bit for bit, as
    one captured CUDA graph and as stream launches; with 0 the same."""
    import torch
    K, launches = 5, 12
    nb = 4 * n
    plan = tb.rotation_plan(nb, K * nb)
    g = np.random.default_rng(600 + nsrc + n % 97 + graph)
    slices = [[finite_floats(g, n) for _ in range(K)] for _ in range(nsrc)]
    bufs = []
    for per_src in slices:
        b = dev_bytes(plan.alloc_bytes)
        for j, a in enumerate(per_src):
            b[j * plan.slice_stride:j * plan.slice_stride + nb].copy_(to_dev(a))
        bufs.append(b)
    last = (launches - 1) % K
    exp = oracle.dst_reference([per_src[last] for per_src in slices])
    for early in (1, 0):
        dst = dev_bytes(nb, fill=0)
        with tb.Context(0, tb.options(early_reads=early)) as c:
            def chain(stream):
                for i in range(launches):
                    off = (i % K) * plan.slice_stride
                    c.reduce_copy([b.data_ptr() + off for b in bufs], dst, nb, 0, stream)
            torch.cuda.synchronize()
            if graph:
                cap = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream()
                with torch.cuda.graph(cap, stream=s):
                    chain(s)
                cap.replay()
                torch.cuda.synchronize()
                del cap
            else:
                s = torch.cuda.Stream()
                chain(s)
                s.synchronize()
        mm = oracle.first_mismatch(to_host(dst).view(np.uint32), exp.view(np.uint32))
        assert mm == -1, f"early_reads={early}: first mismatch at element {mm}"


@pytest.mark.parametrize("graph", [1, 0])
@pytest.mark.parametrize("iters,warmup,K", [(5, 3, 8), (1, 3, 8), (8, 0, 8), (3, 5, 4), (7, 2, 1)])
def test_rotation_reads_slice_i_mod_k(tb, iters, warmup, K, graph):
    """Slices filled with different patterns: after the loop dst holds the
    last iteration's slice, (iters - 1) % K - whether the loop runs as one
    CUDA graph or as stream launches."""
    nb = 64 * 1024
    n = nb // 4
    with tb.Context(0, tb.options(warmup=warmup, use_graph=graph)) as c:
        plan = tb.rotation_plan(nb, K * nb)
        assert plan.K == K
        src = dev_bytes(plan.alloc_bytes)
        for j in range(K):
            c.fill_source(src.data_ptr() + j * plan.slice_stride, nb, tb.default_pattern(), j)
        dst = dev_bytes(nb, fill=0)
        last = oracle.slice_for_iteration(iters - 1, K)
        expect = oracle.prepare_reference(n, last)
        r = c.run_transfer([src], dst, nb, iters=iters, rotate_bytes=K * nb, expected=expect)
        assert r["mismatch_index"] == -1 and r["graphed"] == graph
        assert len(r["iter_ms"]) == iters and all(t > 0 for t in r["iter_ms"])


@pytest.mark.parametrize("graph,gate", [(1, 0), (0, 1), (0, 0)])
@pytest.mark.parametrize("iters,warmup,K", [(10, 3, 4), (7, 2, 5), (1, 0, 3)])
def test_dma_executor_reads_slice_i_mod_k(tb, iters, warmup, K, graph, gate):
    """The DMA (copy-engine) executor of PR #365's "Technical Details" rotates
    inline: slices filled with different patterns, dst ends as the slice of
    the last iteration, (iters - 1) % K, in graph and stream loops."""
    nb = 64 * 1024 + 12
    n = nb // 4
    with tb.Context(0, tb.options(warmup=warmup, use_graph=graph, use_gate=gate)) as c:
        plan = tb.rotation_plan(nb, K * nb)
        assert plan.K == K
        src = dev_bytes(plan.alloc_bytes)
        for j in range(K):
            c.fill_source(src.data_ptr() + j * plan.slice_stride, nb, tb.default_pattern(), j)
        dst = dev_bytes(nb + 64, fill=0x5A)
        expect = oracle.prepare_reference(n, oracle.slice_for_iteration(iters - 1, K))
        r = c.run_transfer([src], dst, nb, iters=iters, rotate_bytes=K * nb, expected=expect,
                           executor=tb.TB_EXEC_DMA)
        assert r["mismatch_index"] == -1 and r["validated"] == 1
        assert r["executor"] == tb.TB_EXEC_DMA and r["ctas"] == 0 and r["engine"] == 0
        assert r["graphed"] == graph and len(r["iter_ms"]) == iters
        assert np.all(to_host(dst, 64, nb) == 0x5A)


def test_dma_executor_single_transfer_4mib(tb):
    """The 4 MiB single transfer (K = 64 at 256 MiB of rotation, a
    268,435,456 B allocation) on the copy engines: dst == src0 bit for bit,
    checked on the device and against the oracle's PrepSrcValue."""
    nb = 4 * MiB
    with tb.Context(0) as c:
        plan = tb.rotation_plan(nb, 256 * MiB)
        assert plan.K == 64 and plan.alloc_bytes == 268435456
        src = dev_bytes(plan.alloc_bytes)
        c.fill_source(src, nb, tb.default_pattern(), 0)
        c.prepare_sources([src], nb, 256 * MiB)
        dst = dev_bytes(nb, fill=0)
        r = c.run_transfer([src], dst, nb, iters=10, rotate_bytes=256 * MiB,
                           expected_device=src, executor=tb.TB_EXEC_DMA)
        assert r["K"] == 64 and r["validated"] == 1 and r["gbps"] > 0
        assert np.array_equal(to_host(dst).view(np.float32), oracle.prepare_reference(nb // 4, 0))


def test_dma_executor_rejects_other_source_counts(tb):
    with tb.Context(0) as c:
        a, b, d = dev_bytes(4096), dev_bytes(4096), dev_bytes(4096, fill=3)
        for srcs in ([], [a, b]):
            with pytest.raises(tb.TBError) as e:
                c.run_transfer(srcs, d, 4096, iters=1, rotate_bytes=0, executor=tb.TB_EXEC_DMA)
            assert e.value.code == tb.TB_ENOTSUP
        with pytest.raises(tb.TBError) as e:
            c.run_transfer([a], d, 4096, iters=1, rotate_bytes=0, executor=7)
        assert e.value.code == tb.TB_EINVAL
        assert np.all(to_host(d) == 3)


def test_byte_offset(tb):
    nb = 1 * MiB + 64
    n = nb // 4
    with tb.Context(0, tb.options(byte_offset=20)) as c:
        plan = tb.rotation_plan(nb, 4 * MiB, 20)
        srcs = [dev_bytes(plan.alloc_bytes) for _ in range(2)]
        refs = [oracle.prepare_reference(n, k) for k in range(2)]
        c.upload_sources(srcs, refs, nb)
        c.prepare_sources(srcs, nb, 4 * MiB)
        dst = dev_bytes(nb + 20, fill=0x77)
        r = c.run_transfer(srcs, dst, nb, iters=6, rotate_bytes=4 * MiB,
                           expected=oracle.dst_reference(refs))
        assert r["K"] == plan.K == 4 and r["mismatch_index"] == -1
        assert np.all(to_host(dst, 20) == 0x77)


@pytest.mark.parametrize("always", [0, 1])
@pytest.mark.parametrize("direct", [0, 1])
def test_validation_reports_first_mismatch(tb, always, direct):
    """validateDirect = 1 compares on the GPU against a device copy of the
    host expected values; the reported mismatch is the same either way."""
    nb = 256 * 1024
    n = nb // 4
    with tb.Context(0, tb.options(always_validate=always, validate_direct=direct)) as c:
        src = dev_bytes(nb)
        c.fill_source(src, nb, tb.default_pattern(), 0)
        dst = dev_bytes(nb)
        wrong = oracle.prepare_reference(n, 0)
        wrong[12345] = 1.0        # a planted error in the expected copy
        with pytest.raises(tb.TBError) as e:
            c.run_transfer([src], dst, nb, iters=3, rotate_bytes=0, expected=wrong)
        assert e.value.code == tb.TB_EVALIDATE
        r = e.value.result
        assert r["mismatch_index"] == 12345
        assert r["mismatch_expected"] == np.float32(1.0).view(np.uint32)
        assert r["mismatch_actual"] == np.float32(oracle.prep_src_value(0, 12345)).view(np.uint32)
        if always:
            assert r["iters"] == 1       # stopped at the first iteration
        assert c.validate(dst, wrong, nb) == (12345, int(r["mismatch_expected"]),
                                              int(r["mismatch_actual"]))
        assert c.validate(dst, oracle.prepare_reference(n, 0), nb) is None


def test_validate_source_checks_uploads_and_slices(tb):
    """validateSource = 1: tb_upload_sources compares every device source
    with its host copy and tb_prepare_sources every one of the 64 slices of
    a 4 MiB source with slice 0; both pass on correct data, and the transfer
    afterwards validates."""
    nb = 4 * MiB
    n = nb // 4
    plan = tb.rotation_plan(nb, 256 * MiB)
    refs = [oracle.prepare_reference(n, k) for k in range(2)]
    with tb.Context(0, tb.options(validate_source=1, byte_offset=12)) as c:
        srcs = [dev_bytes(plan.alloc_bytes + 12) for _ in range(2)]
        c.upload_sources(srcs, refs, nb)
        c.prepare_sources(srcs, nb, 256 * MiB)
        whole = to_host(srcs[1])[12:12 + 64 * plan.slice_stride].reshape(64, -1)
        assert all(np.array_equal(whole[j][:nb], refs[1].view(np.uint8)) for j in (0, 37, 63))
        dst = dev_bytes(nb + 12, fill=0)
        r = c.run_transfer(srcs, dst, nb, iters=4, rotate_bytes=256 * MiB,
                           expected=oracle.dst_reference(refs))
        assert r["mismatch_index"] == -1 and r["K"] == 64


@pytest.mark.parametrize("da,db", [(0, 0), (4, 4), (3, 3), (0, 5), (7, 1)])
def test_validate_device_first_mismatch(tb, ctx, da, db):
    """validateDirect on the GPU: the first differing byte, wherever it sits
    (byte head, vector body, tail), for co-aligned and misaligned buffers."""
    g = np.random.default_rng(da * 16 + db)
    n = 3 * (1 << 20) + 13
    data = g.integers(0, 256, n, dtype=np.uint8)
    a = dev_bytes(n + 16)
    b = dev_bytes(n + 16)
    a[da:da + n].copy_(to_dev(data))
    b[db:db + n].copy_(to_dev(data))
    pa, pb = a.data_ptr() + da, b.data_ptr() + db
    assert ctx.validate_device(pa, pb, n, 1) is None
    for pos in (0, 1, 15, 16, 4097, n // 2, n - 1):
        for extra in (None, pos + 1000):
            bad = data.copy()
            bad[pos] ^= 0x5A
            if extra is not None and extra < n:
                bad[extra] ^= 0x01
            b[db:db + n].copy_(to_dev(bad))
            got = ctx.validate_device(pa, pb, n, 1)
            assert got is not None and got[0] == pos
            assert got[1] == bad[pos] and got[2] == data[pos]
    b[db:db + n].copy_(to_dev(data))
    assert ctx.validate_device(pa, pb, n - n % 4, 4) is None


def test_run_transfer_validates_on_the_device(tb):
    nb = 64 * MiB
    n = nb // 4
    refs = [oracle.prepare_reference(n, k) for k in range(3)]
    exp_dev = to_dev(oracle.dst_reference(refs))
    with tb.Context(0, tb.options(always_validate=1)) as c:
        srcs = [dev_bytes(nb) for _ in range(3)]
        for k, s in enumerate(srcs):
            c.fill_source(s, nb, tb.default_pattern(), k)
        dst = dev_bytes(nb)
        r = c.run_transfer(srcs, dst, nb, iters=5, rotate_bytes=0, expected_device=exp_dev)
        assert r["validated"] == 1 and r["mismatch_index"] == -1 and r["iters"] == 5
        wrong = oracle.dst_reference(refs)
        wrong[777777] = 0.5
        with pytest.raises(tb.TBError) as e:
            c.run_transfer(srcs, dst, nb, iters=5, rotate_bytes=0, expected_device=to_dev(wrong))
        assert e.value.code == tb.TB_EVALIDATE and e.value.result["mismatch_index"] == 777777
        assert e.value.result["iters"] == 1


def test_gate_deadline_returns_timeout(tb):
    """A gate whose deadline (1 microsecond) passes before the host releases
    it returns on its own; the call reports TB_ETIMEOUT and the context stays
    usable."""
    nb = 1 * MiB
    with tb.Context(0, tb.options(wait_timeout_ns=1000, warmup=3, use_graph=0)) as c:
        src = dev_bytes(nb)
        c.fill_source(src, nb, tb.default_pattern(), 0)
        dst = dev_bytes(nb)
        with pytest.raises(tb.TBError) as e:
            c.run_transfer([src], dst, nb, iters=200, rotate_bytes=0)
        assert e.value.code == tb.TB_ETIMEOUT
        ref = oracle.prepare_reference(nb // 4, 0)
        assert c.validate(dst, ref, nb) is None
        c2 = tb.options(use_gate=0, use_graph=0)
    with tb.Context(0, c2) as c:
        src = dev_bytes(nb)
        c.fill_source(src, nb, tb.default_pattern(), 0)
        dst = dev_bytes(nb)
        r = c.run_transfer([src], dst, nb, iters=4, rotate_bytes=0, expected=ref)
        assert r["gated"] == 0 and r["graphed"] == 0


@pytest.mark.parametrize("nsrc,graph", [(3, 1), (3, 0), (1, 1)])
def test_pipeline_wait_expiry_is_reported(tb, nsrc, graph):
    """kernel_wait_ns = 0: the bulk pipeline's wait for the first tile's loads
    cannot be met (they were issued a few instructions earlier), so the
    kernel records the failure, lets the loads it issued land and stops.
    tb_run_transfer reports TB_ETIMEOUT; the context and the device stay
    usable, and a normal transfer afterwards is bit-exact."""
    nb = 64 * MiB
    n = nb // 4
    srcs = [dev_bytes(nb) for _ in range(nsrc)]
    dst = dev_bytes(nb, fill=0)
    with tb.Context(0, tb.options(reduce_engine=2, kernel_wait_ns=0, use_graph=graph)) as c:
        for k, s_ in enumerate(srcs):
            c.fill_source(s_, nb, tb.default_pattern(), k)
        with pytest.raises(tb.TBError) as e:
            c.run_transfer(srcs, dst, nb, iters=2, rotate_bytes=0)
        assert e.value.code == tb.TB_ETIMEOUT
        assert "expired" in str(e.value)
    with tb.Context(0, tb.options(reduce_engine=2)) as c:
        expect = oracle.dst_reference([oracle.prepare_reference(n, k) for k in range(nsrc)])
        r = c.run_transfer(srcs, dst, nb, iters=2, rotate_bytes=0, expected=expect)
        assert r["mismatch_index"] == -1


def test_async_reduce_copy_reports_an_earlier_expiry(tb):
    """tb_reduce_copy is asynchronous; an expired wait in one launch is
    reported by the context's next tb_reduce_copy, which launches nothing."""
    import torch
    nb = 64 * MiB
    srcs = [dev_bytes(nb, fill=0) for _ in range(3)]
    dst = dev_bytes(nb, fill=0)
    with tb.Context(0, tb.options(reduce_engine=2, kernel_wait_ns=0)) as c:
        c.reduce_copy(srcs, dst, nb)
        torch.cuda.synchronize()
        with pytest.raises(tb.TBError) as e:
            c.reduce_copy(srcs, dst, nb)
        assert e.value.code == tb.TB_ETIMEOUT
        torch.cuda.synchronize()


@pytest.mark.parametrize("n", [1, 1000003, (96 << 20) // 4 + 5])
def test_reduce_copy_host_staged(tb, ctx, n):
    """Pageable host memory: the bytes are staged through device buffers in
    32 MiB chunks on three streams."""
    import torch
    g = np.random.default_rng(n)
    srcs = [finite_floats(g, n) for _ in range(3)]
    hd = np.zeros(n, np.float32)
    ds = [dev_bytes(4 * n) for _ in range(3)]
    dd = dev_bytes(4 * n)
    st = torch.cuda.Stream()
    ctx.reduce_copy_host(srcs, hd, 4 * n, ds, dd, 0, st)
    st.synchronize()
    assert oracle.first_mismatch(hd, oracle.dst_reference(srcs)) == -1
    with pytest.raises(tb.TBError):
        ctx.reduce_copy_host(srcs, hd, 4 * n, [None] * 3, None, 0, st)


def test_reduce_copy_host_rejects_before_queuing(tb, ctx):
    """A staged call whose length is not whole float32 elements (here past
    the first 32 MiB chunk) or whose device buffers are misaligned is
    rejected before any copy is queued; the next call on the stream works."""
    import torch
    n = (40 << 20) // 4
    srcs = [np.full(n, 1.5, np.float32) for _ in range(2)]
    hd = np.zeros(n, np.float32)
    ds = [dev_bytes(4 * n + 64) for _ in range(2)]
    dd = dev_bytes(4 * n + 64, fill=0x7F)
    st = torch.cuda.Stream()
    with pytest.raises(tb.TBError) as e:
        ctx.reduce_copy_host(srcs, hd, 4 * n - 2, ds, dd, 0, st)
    assert e.value.code == tb.TB_EINVAL
    with pytest.raises(tb.TBError) as e:
        ctx.reduce_copy_host(srcs, hd, 4 * n, [d.data_ptr() + 2 for d in ds], dd, 0, st)
    assert e.value.code == tb.TB_EINVAL
    st.synchronize()
    assert np.all(to_host(dd) == 0x7F) and np.all(hd == 0)    # nothing ran
    ctx.reduce_copy_host(srcs, hd, 4 * n, ds, dd, 0, st)
    st.synchronize()
    assert np.all(hd == 3.0)


def test_reduce_copy_host_end_to_end(tb, ctx):
    import torch
    g = np.random.default_rng(9)
    n = 1000003
    srcs = [finite_floats(g, n) for _ in range(3)]
    hs = [torch.from_numpy(s).pin_memory() for s in srcs]
    hd = torch.empty(n, dtype=torch.float32).pin_memory()
    st = torch.cuda.Stream()
    # page-locked and mapped: one kernel across the host link, no device buffers
    ctx.reduce_copy_host(hs, hd, 4 * n, [None] * 3, None, 0, st)
    st.synchronize()
    assert oracle.first_mismatch(hd.numpy(), oracle.dst_reference(srcs)) == -1


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the bench times
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("engine", [0, 1, 2])
def test_three_source_256mib_all_subexecutors(tb, engine):
    """3 x 256 MiB, src_k = PrepSrcValue(k, i), K = 1; sub-executor counts
    1, 4, 16, 32 and auto, with each reduce engine.  dst = 6 *
    PrepSrcValue(0, i) exactly."""
    nb = 256 * MiB
    n = nb // 4
    refs = [oracle.prepare_reference(n, k) for k in range(3)]
    exp = oracle.dst_reference(refs)
    with tb.Context(0, tb.options(reduce_engine=engine)) as c:
        srcs = [dev_bytes(nb) for _ in range(3)]
        for k, s in enumerate(srcs):
            c.fill_source(s, nb, tb.default_pattern(), k)
        for k, s in enumerate(srcs):
            assert c.validate(s, refs[k], nb) is None
        for se in (1, 4, 16, 32, 0):
            dst = dev_bytes(nb, fill=0)
            r = c.run_transfer(srcs, dst, nb, num_subexec=se, iters=2, rotate_bytes=256 * MiB,
                               expected=exp)
            assert r["K"] == 1 and r["mismatch_index"] == -1, se
            got = to_host(dst).view(np.float32)
            assert oracle.first_mismatch(got, exp) == -1
            assert got[:4].tolist() == [186.0, 990.0, 1794.0, 300.0]


@pytest.mark.parametrize("mib", [8, 64, 512])
@pytest.mark.parametrize("rotate", [256 * MiB, 0])
def test_compress_sweep_sizes(tb, mib, rotate):
    nb = mib * MiB
    n = nb // 4
    pct = (40, 20, 0, 20, 20)
    ref = oracle.fill_compress(n, pct, 0x5EED, 0)
    with tb.Context(0) as c:
        plan = tb.rotation_plan(nb, rotate)
        src = dev_bytes(plan.alloc_bytes)
        c.fill_source(src, nb, tb.compress_pattern(pct, 0x5EED), 0)
        assert c.validate(src, ref, nb) is None
        c.prepare_sources([src], nb, rotate)
        last = plan.K - 1
        assert c.validate(src.data_ptr() + last * plan.slice_stride, ref, nb) is None
        dst = dev_bytes(nb, fill=0)
        r = c.run_transfer([src], dst, nb, iters=3, rotate_bytes=rotate, expected=ref)
        assert r["mismatch_index"] == -1 and r["K"] == plan.K

"""GPU parity past 2^32 bytes: a reduce-copy, a rotated transfer whose last
slice starts beyond 4 GiB, and batched copies longer than 4 GiB, each
compared in full with the oracle.  Every byte offset, element index, tile
and chunk position of the kernels is 64-bit; these cases fail if any of
them wraps at 32 bits.  They need about 16 GiB of host memory and 13 GiB of
device memory."""
import numpy as np
import pytest

import oracle
from copy_reduce_dst_gb300 import workloads
from gpu_helpers import dev_bytes, to_dev, to_host

pytestmark = pytest.mark.gpu

MiB = 1 << 20
GiB = 1 << 30


def _host_available_bytes() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


@pytest.fixture(scope="module")
def tb():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    if _host_available_bytes() < 24 * GiB:
        pytest.skip("needs about 24 GiB of free host memory")
    from copy_reduce_dst_gb300 import _build
    _build.build()
    from copy_reduce_dst_gb300 import tb as mod
    return mod


@pytest.fixture(autouse=True)
def _free_device_memory():
    yield
    import gc
    import torch
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("engine", [1, 2])
def test_two_sources_past_4gib(tb, engine):
    nb = 4 * GiB + 4 * MiB + 12
    n = nb // 4
    with tb.Context(0, tb.options(reduce_engine=engine)) as c:
        srcs = [dev_bytes(nb), dev_bytes(nb)]
        for k, s in enumerate(srcs):
            c.fill_source(s, nb, tb.default_pattern(), k)
        dst = dev_bytes(nb + 256, fill=0xC3)
        assert c.reduce_plan(srcs, dst, nb)["engine"] == engine
        c.reduce_copy(srcs, dst, nb, 32)
        got = to_host(dst)
        del srcs, dst
    assert np.all(got[nb:] == 0xC3), "write past the end of dst"
    refs = [oracle.prepare_reference(n, k) for k in range(2)]
    exp = oracle.dst_reference(refs)
    del refs
    mm = oracle.first_mismatch(got[:nb].view(np.uint32), exp.view(np.uint32))
    assert mm == -1, f"first mismatch at element {mm}"


def test_rotated_slice_beyond_4gib(tb):
    """K = 3 slices of 2.25 GiB: slice 2 starts at byte 4.5 GiB of the
    allocation.  Each slice holds a different pattern, so dst shows which
    slice the last iteration read (iteration 2 reads slice 2)."""
    nb = 2 * GiB + 256 * MiB + 8
    n = nb // 4
    rot = 3 * nb
    plan = tb.rotation_plan(nb, rot)
    assert plan.K == 3 and 2 * plan.slice_stride > 4 * GiB
    with tb.Context(0, tb.options(warmup=0)) as c:
        src = dev_bytes(plan.alloc_bytes)
        for j in range(3):
            c.fill_source(src.data_ptr() + j * plan.slice_stride, nb, tb.default_pattern(), j)
        dst = dev_bytes(nb, fill=0)
        expect = oracle.prepare_reference(n, 2)
        r = c.run_transfer([src], dst, nb, iters=3, rotate_bytes=rot, expected=expect)
        assert r["K"] == 3 and r["alloc_bytes"] == plan.alloc_bytes
        assert r["mismatch_index"] == -1


@pytest.mark.parametrize("src_shift,dst_shift", [(0, 0), (3, 5)])
def test_batch_descriptor_past_4gib(tb, src_shift, dst_shift):
    """One descriptor of 4 GiB + 77 bytes: bulk copies when src and dst
    share their address modulo 16, the funnel-shift path otherwise."""
    import torch
    length = 4 * GiB + 77
    pool = length + 64
    src_h = workloads.random_bytes(pool, 91)
    with tb.Context(0) as c:
        src = to_dev(src_h)
        dst = torch.zeros(pool, dtype=torch.uint8, device="cuda")
        desc = np.array([[src.data_ptr() + src_shift, dst.data_ptr() + dst_shift, length]],
                        dtype=np.uint64)
        c.batch_copy(desc)
        st = c.last_batch_stats()
        got = to_host(dst)
        del src, dst
    assert st["descs"] == 1 and st["cta_items"] > 0
    exp = np.zeros(pool, dtype=np.uint8)
    oracle.apply_batch(exp, src_h, [src_shift], [dst_shift], [length])
    mm = oracle.first_mismatch(got, exp)
    assert mm == -1, f"first differing byte {mm}"

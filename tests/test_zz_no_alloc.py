"""tb_batch_copy_noalloc: the batched copy for callers that cannot allocate.

Some callers cannot call cudaMalloc: a serving engine that has handed all
free HBM to its own allocator has none left, and a latency-sensitive loop
cannot afford a call that may synchronize the device.  This entry point
keeps its work items in a fixed array inside the library instead of
context-owned slots, so these checks run it twice in a row on one stream
(the second batch overwrites the shared array after the first kernel has
read it) and compare each whole destination pool byte for byte with the
oracle's memcpy of the same descriptors ("Design of #5040" of the Mooncake
HipTransport RFC: a (src, dst, len) array copied as plain memcpys) and with
what tb_batch_copy writes.  Both launch forms run: a batch with long copies
(bulk pipeline plus warps) and one of short copies only.  An expired wait is
forced in a child process and must come back from the next call.

This file sorts last so that a run stopping at its first failure has run
every other test before it; each test also passes alone in a fresh process.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from copy_reduce_dst_gb300 import workloads

pytestmark = pytest.mark.gpu

MiB = 1 << 20
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tb():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from copy_reduce_dst_gb300 import _build
    _build.build()
    from copy_reduce_dst_gb300 import tb as mod
    return mod


def _mixed(seed, pool):
    # short copies at any byte alignment plus long ones that become CTA chunks
    small = workloads.random_batch(seed, 3000, 16384, pool * 3 // 4, align=1)
    g = workloads.rng(seed + 100)
    big = g.integers(16385, 400000, size=40, dtype=np.uint64)
    so = workloads.scatter_offsets(g, big, pool * 3 // 4, pool, 1)
    do = workloads.scatter_offsets(g, big, pool * 3 // 4, pool, 1)
    return workloads.BatchLayout("mixed", np.concatenate([small.src_off, so]),
                                 np.concatenate([small.dst_off, do]),
                                 np.concatenate([small.lens, big]), pool, pool)


def _index_pages(seed, pool):
    # the 3840 x 2112 B index-page shape (a contiguous source, distinct
    # 2112 B-aligned destination slots) in a smaller pool: short copies only
    g = workloads.rng(seed)
    n, size = 3840, 2112
    slots = g.choice(pool // size, size=n, replace=False).astype(np.uint64)
    return workloads.BatchLayout("index pages", np.arange(n, dtype=np.uint64) * np.uint64(size),
                                 slots * np.uint64(size), np.full(n, size, dtype=np.uint64),
                                 pool, pool)


def _two_calls_in_a_row(tb, layouts, pool, seed):
    import torch
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    src_h = workloads.random_bytes(pool, seed)
    init_h = workloads.random_bytes(pool, seed + 1)
    src = torch.from_numpy(src_h.copy()).cuda()
    ref = [torch.from_numpy(init_h.copy()).cuda() for _ in layouts]
    got = [torch.from_numpy(init_h.copy()).cuda() for _ in layouts]
    torch.cuda.synchronize()

    with tb.Context(0) as ctx:
        for lay, out in zip(layouts, ref):
            ctx.batch_copy(lay.descriptors(src.data_ptr(), out.data_ptr()), stream)
    # two calls back to back on one stream, no synchronization in between
    for lay, out in zip(layouts, got):
        tb.batch_copy_noalloc(lay.descriptors(src.data_ptr(), out.data_ptr()), stream)
    stream.synchronize()

    for lay, r, g in zip(layouts, ref, got):
        exp = init_h.copy()
        oracle.apply_batch(exp, src_h, lay.src_off, lay.dst_off, lay.lens)
        mm = oracle.first_mismatch(g.cpu().numpy(), exp)
        assert mm == -1, f"{lay.name}: first byte differing from the oracle {mm}"
        mm = oracle.first_mismatch(g.cpu().numpy(), r.cpu().numpy())
        assert mm == -1, f"{lay.name}: first byte differing from tb_batch_copy {mm}"
        assert not np.array_equal(exp, init_h)
    # nothing left to report after a clean run
    tb.batch_copy_noalloc(np.empty((0, 3), dtype=np.uint64), stream)


def test_noalloc_mixed_batches_twice_in_a_row(tb):
    _two_calls_in_a_row(tb, [_mixed(1, 64 * MiB), _mixed(2, 64 * MiB)], 64 * MiB, 11)


def test_noalloc_short_only_batches_twice_in_a_row(tb):
    pool = 32 * MiB
    _two_calls_in_a_row(tb, [_index_pages(3, pool),
                             workloads.random_batch(4, 3000, 16384, pool, align=1)], pool, 21)


_CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, ".")
import oracle
from copy_reduce_dst_gb300 import tb, workloads
torch.cuda.set_device(0)
MiB = 1 << 20

def code(descs):
    try:
        tb.batch_copy_noalloc(descs)
        return 0
    except tb.TBError as e:
        return e.code

out = {}
empty = np.empty((0, 3), dtype=np.uint64)
out["probe_before"] = code(empty)
# Long copies: with a wait limit of 0 the bulk pipeline's first wait is one
# non-blocking probe a few instructions after its loads, so it runs out.
lay = workloads.random_batch(61, 40, 4 * MiB, 256 * MiB, align=64, min_len=1 * MiB)
src = torch.zeros(256 * MiB, dtype=torch.uint8, device="cuda")
dst = torch.zeros(256 * MiB, dtype=torch.uint8, device="cuda")
out["launch"] = code(lay.descriptors(src.data_ptr(), dst.data_ptr()))
torch.cuda.synchronize()
out["probe_after"] = code(empty)
out["probe_again"] = code(empty)
# Short copies only have no bounded wait: the next batch copies exactly.
pool = 16 * MiB
sl = workloads.random_batch(62, 2000, 16384, pool, align=1)
src_h = workloads.random_bytes(pool, 63)
dst_h = workloads.random_bytes(pool, 64)
s = torch.from_numpy(src_h.copy()).cuda()
d = torch.from_numpy(dst_h.copy()).cuda()
torch.cuda.synchronize()
out["short"] = code(sl.descriptors(s.data_ptr(), d.data_ptr()))
torch.cuda.synchronize()
oracle.apply_batch(dst_h, src_h, sl.src_off, sl.dst_off, sl.lens)
out["short_mismatch"] = int(oracle.first_mismatch(d.cpu().numpy(), dst_h))
out["probe_end"] = code(empty)
print("RESULT " + json.dumps(out))
"""


def test_noalloc_expired_wait_reported_by_next_call(tb):
    env = dict(os.environ, TB_KERNEL_WAIT_NS="0")
    r = subprocess.run([sys.executable, "-c", _CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULT ")][-1]
    out = json.loads(line[len("RESULT "):])
    assert out["probe_before"] == 0
    assert out["launch"] == 0                    # enqueued; the kernel fails later
    assert out["probe_after"] == tb.TB_ETIMEOUT  # the next call reports it ...
    assert out["probe_again"] == 0               # ... once
    assert out["short"] == 0 and out["short_mismatch"] == -1
    assert out["probe_end"] == 0


def test_noalloc_rejects_batches_beyond_its_capacity(tb):
    import torch
    torch.cuda.set_device(0)
    buf = torch.zeros(2 * MiB, dtype=torch.uint8, device="cuda")
    n = tb.TB_NOALLOC_MAX_ITEMS + 1
    desc = np.empty((n, 3), dtype=np.uint64)
    desc[:, 0] = buf.data_ptr()
    desc[:, 1] = buf.data_ptr() + MiB
    desc[:, 2] = 8
    with pytest.raises(tb.TBError) as e:
        tb.batch_copy_noalloc(desc)
    assert e.value.code == tb.TB_ENOTSUP
    torch.cuda.synchronize()
    assert int(buf.sum().item()) == 0


def test_noalloc_rejects_null_and_wrapping_ranges(tb):
    import torch
    torch.cuda.set_device(0)
    src = torch.full((MiB,), 7, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(MiB, dtype=torch.uint8, device="cuda")
    good = [src.data_ptr(), dst.data_ptr(), 4096]
    for bad in ([0, dst.data_ptr() + 8192, 64],               # null source
                [src.data_ptr(), 0, 64],                      # null destination
                [2**64 - 32, dst.data_ptr() + 8192, 64]):     # source range wraps
        desc = np.array([good, bad], dtype=np.uint64)
        with pytest.raises(tb.TBError) as e:
            tb.batch_copy_noalloc(desc)
        assert e.value.code == tb.TB_EINVAL
    torch.cuda.synchronize()
    assert int(dst.sum().item()) == 0               # nothing copied, not even `good`


def test_noalloc_empty_batches_copy_nothing(tb):
    import torch
    torch.cuda.set_device(0)
    src = torch.full((MiB,), 9, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(MiB, dtype=torch.uint8, device="cuda")
    tb.batch_copy_noalloc(np.empty((0, 3), dtype=np.uint64))
    tb.batch_copy_noalloc(np.array([[src.data_ptr(), dst.data_ptr(), 0],
                                    [0, 0, 0]], dtype=np.uint64))
    torch.cuda.synchronize()
    assert int(dst.sum().item()) == 0


def test_noalloc_refuses_a_capturing_stream(tb):
    import torch
    torch.cuda.set_device(0)
    src = torch.full((MiB,), 5, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(MiB, dtype=torch.uint8, device="cuda")
    x = torch.zeros(16, device="cuda")
    desc = np.array([[src.data_ptr(), dst.data_ptr(), 4096]], dtype=np.uint64)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    codes = []
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        x.add_(1)
        try:
            tb.batch_copy_noalloc(desc, torch.cuda.current_stream())
            codes.append(0)
        except tb.TBError as e:
            codes.append(e.code)
    graph.replay()
    torch.cuda.synchronize()
    assert codes == [tb.TB_ENOTSUP]
    assert int(dst.sum().item()) == 0
    assert float(x.sum().item()) == 16.0

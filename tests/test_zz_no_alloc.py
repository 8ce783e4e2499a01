"""tb_batch_copy_noalloc against tb_batch_copy.

The no-allocation entry point serves callers that cannot call cudaMalloc
(all free HBM already handed to their own allocator, or a loop that cannot
afford a call that may synchronize the device).  Its work items sit in a
fixed array inside the library instead of context-owned slots.  These
checks run it twice in a row on one stream - the second batch overwrites the
shared array after the first kernel has read it - and compare each result
byte for byte with what tb_batch_copy writes for the same batch.
"""
import numpy as np
import pytest

from copy_reduce_dst_gb300 import workloads

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


def _layout(seed):
    # short copies at any byte alignment plus long ones that become CTA chunks
    small = workloads.random_batch(seed, 3000, 16384, 48 * MiB, align=1)
    g = workloads.rng(seed + 100)
    big = g.integers(16385, 400000, size=40, dtype=np.uint64)
    so = workloads.scatter_offsets(g, big, 48 * MiB, 64 * MiB, 1)
    do = workloads.scatter_offsets(g, big, 48 * MiB, 64 * MiB, 1)
    return workloads.BatchLayout("mixed", np.concatenate([small.src_off, so]),
                                 np.concatenate([small.dst_off, do]),
                                 np.concatenate([small.lens, big]), 64 * MiB, 64 * MiB)


def test_noalloc_matches_batch_copy_twice_in_a_row(tb):
    import torch
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    layouts = [_layout(1), _layout(2)]
    src = torch.from_numpy(workloads.random_bytes(64 * MiB, 11).copy()).cuda()
    init = torch.from_numpy(workloads.random_bytes(64 * MiB, 12).copy()).cuda()
    ref = [init.clone(), init.clone()]
    got = [init.clone(), init.clone()]
    torch.cuda.synchronize()

    with tb.Context(0) as ctx:
        for lay, out in zip(layouts, ref):
            ctx.batch_copy(lay.descriptors(src.data_ptr(), out.data_ptr()), stream)
    # two calls back to back on one stream, no synchronization in between
    for lay, out in zip(layouts, got):
        tb.batch_copy_noalloc(lay.descriptors(src.data_ptr(), out.data_ptr()), stream)
    stream.synchronize()

    for r, g in zip(ref, got):
        a, b = r.cpu().numpy(), g.cpu().numpy()
        diff = np.nonzero(a != b)[0]
        assert diff.size == 0, f"first differing byte {diff[0]}"
    assert not np.array_equal(ref[0].cpu().numpy(), init.cpu().numpy())


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

"""CPU tests of the batched copy's host packer (tb_pack.cpp), built with g++
against a small harness: every long copy is covered exactly once by its
pieces, CTA shares are equal, the per-CTA table is consistent, and short
copies come longest first."""
import ctypes as ct
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "copy_reduce_dst_gb300", "csrc")


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("pack") / "libpack.so")
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", f"-I{ROOT}/include", f"-I{CSRC}",
           f"-I{cuda_inc}", os.path.join(CSRC, "tb_pack.cpp"),
           os.path.join(ROOT, "tests", "pack_harness.cpp"), "-o", out]
    subprocess.run(cmd, check=True)
    lib = ct.CDLL(out)
    lib.harness_pack.restype = ct.c_int
    lib.harness_pack.argtypes = [ct.c_void_p, ct.c_size_t, ct.c_uint64, ct.c_int, ct.c_void_p,
                                 ct.c_void_p, ct.c_void_p]
    return lib


def pack(lib, desc, small_max=16384, full_grid=608):
    desc = np.ascontiguousarray(desc, dtype=np.uint64).reshape(-1, 3)
    n = desc.shape[0]
    cap = (n + full_grid) * 24 + (full_grid + 1) * 4
    buf = np.zeros(cap, dtype=np.uint8)
    bucket = np.zeros(8192, dtype=np.uint32)
    out = np.zeros(8, dtype=np.uint64)
    rc = lib.harness_pack(desc.ctypes.data if n else None, n, small_max, full_grid,
                          buf.ctypes.data, bucket.ctypes.data, out.ctypes.data)
    assert rc == 0
    n_long, n_short, grid, toff, upload, bound = (int(x) for x in out[:6])
    assert upload <= bound <= cap
    items = buf[: (n_long + n_short) * 24].view(np.uint64).reshape(-1, 3)
    first = buf[toff: toff + (grid + 1) * 4].view(np.uint32)
    return items[:n_long], items[n_long:], first, grid


def random_desc(g, n, long_frac, small_max):
    lens = np.where(g.random(n) < long_frac, g.integers(small_max + 1, 40 * small_max, n),
                    g.integers(0, small_max + 1, n)).astype(np.uint64)
    src = g.integers(1, 2**40, n, dtype=np.uint64)
    dst = g.integers(1, 2**40, n, dtype=np.uint64)
    return np.stack([src, dst, lens], axis=1)


@pytest.mark.parametrize("seed,n,long_frac,small,grid", [
    (0, 1000, 0.05, 16384, 608), (1, 47540, 0.0005, 16384, 608), (2, 50, 0.5, 1000, 608),
    (3, 3000, 0.0, 16384, 608), (4, 200, 1.0, 64, 16), (5, 7, 0.3, 16384, 1), (6, 0, 0.0, 16384, 608)])
def test_packer_invariants(harness, seed, n, long_frac, small, grid):
    g = np.random.default_rng(seed)
    desc = random_desc(g, n, long_frac, small)
    longs, shorts, first, G = pack(harness, desc, small, grid)
    lens = desc[:, 2] if n else np.zeros(0, np.uint64)
    is_long = lens > small
    assert G >= 1 and G <= grid

    # long copies: pieces in stream order, each descriptor covered exactly once
    k = 0
    for s, d, ln in desc[is_long]:
        off = 0
        while off < ln:
            ps, pd, pl = (int(x) for x in longs[k])
            assert ps == int(s) + off and pd == int(d) + off and pl > 0
            off += pl
            k += 1
        assert off == ln
    assert k == longs.shape[0]

    # per-CTA table and equal shares (cuts on 64-byte stream offsets)
    assert first[0] == 0 and first[G] == longs.shape[0]
    assert np.all(np.diff(first.astype(np.int64)) >= 0)
    total = int(lens[is_long].sum())
    share = np.array([int(longs[first[b]:first[b + 1], 2].sum()) for b in range(G)])
    assert share.sum() == total
    if total:
        assert share.max() - share.min() <= 64 + 64
        assert share.max() <= total // G + 128

    # short copies: the same multiset, longest first by 64-byte bucket
    want = sorted(map(tuple, desc[(lens > 0) & ~is_long].tolist()))
    assert sorted(map(tuple, shorts.tolist())) == want
    shift = 6
    while (small >> shift) > 4096:
        shift += 1
    keys = (shorts[:, 2] >> np.uint64(shift)).astype(np.int64)
    assert np.all(np.diff(keys) <= 0)


def test_packer_batch_47540(harness):
    from copy_reduce_dst_gb300 import workloads
    lay = workloads.batch_head_sliced()
    desc = lay.descriptors(1 << 32, 1 << 36)
    longs, shorts, first, G = pack(harness, desc)
    assert G == 608 and shorts.shape[0] == 47520
    share = np.array([int(longs[first[b]:first[b + 1], 2].sum()) for b in range(G)])
    assert share.sum() == 288 << 20
    assert share.max() - share.min() <= 128

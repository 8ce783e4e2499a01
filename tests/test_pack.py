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
    cap = n * 32 + 8 + (16384 + 1) * 4
    buf = np.zeros(cap, dtype=np.uint8)
    bucket = np.zeros(8192, dtype=np.uint32)
    out = np.zeros(9, dtype=np.uint64)
    rc = lib.harness_pack(desc.ctypes.data if n else None, n, small_max, full_grid,
                          buf.ctypes.data, bucket.ctypes.data, out.ctypes.data)
    assert rc == 0
    n_short, n_long, grid, chunks, total, poff, coff, upload, bound = (int(x) for x in out)
    assert upload <= bound <= cap
    items = buf[: (n_short + n_long) * 24].view(np.uint64).reshape(-1, 3)
    prefix = buf[poff: poff + (n_long + 1) * 8].view(np.uint64)
    cdesc = buf[coff: coff + (chunks + 1) * 4].view(np.uint32)
    return dict(shorts=items[:n_short], longs=items[n_short:], prefix=prefix, chunk_desc=cdesc,
                grid=grid, chunks=chunks, total=total)


def chunk_bytes(lib, p, c):
    lib.harness_chunk_start.restype = ct.c_uint64
    lib.harness_chunk_start.argtypes = [ct.c_uint64, ct.c_uint64, ct.c_uint64]
    return (lib.harness_chunk_start(p["total"], p["chunks"], c + 1) -
            lib.harness_chunk_start(p["total"], p["chunks"], c))


def random_desc(g, n, long_frac, small_max):
    lens = np.where(g.random(n) < long_frac, g.integers(small_max + 1, 40 * small_max, n),
                    g.integers(0, small_max + 1, n)).astype(np.uint64)
    src = g.integers(1, 2**40, n, dtype=np.uint64)
    dst = g.integers(1, 2**40, n, dtype=np.uint64)
    return np.stack([src, dst, lens], axis=1)


@pytest.mark.parametrize("seed,n,long_frac,small,grid", [
    (0, 1000, 0.05, 16384, 608), (1, 47540, 0.0005, 16384, 608), (2, 50, 0.5, 1000, 608),
    (3, 3000, 0.0, 16384, 608), (4, 200, 1.0, 64, 16), (5, 7, 0.3, 16384, 1), (6, 0, 0.0, 16384, 608),
    (7, 300, 1.0, 16384, 608)])
def test_packer_invariants(harness, seed, n, long_frac, small, grid):
    g = np.random.default_rng(seed)
    desc = random_desc(g, n, long_frac, small)
    p = pack(harness, desc, small, grid)
    lens = desc[:, 2] if n else np.zeros(0, np.uint64)
    is_long = lens > small
    G = p["grid"]
    assert 1 <= G <= grid

    # long copies in descriptor order, prefix = running stream offset
    assert np.array_equal(p["longs"], desc[is_long])
    want_prefix = np.concatenate([[0], np.cumsum(lens[is_long])]).astype(np.uint64)
    assert np.array_equal(p["prefix"], want_prefix)
    total = int(want_prefix[-1])
    assert p["total"] == total

    # chunks: a whole number per CTA, equal sizes within 64 bytes, each chunk's
    # first byte inside the long copy the table names
    if is_long.any():
        assert p["chunks"] % G == 0 and p["chunks"] >= G
        sizes = np.array([chunk_bytes(harness, p, c) for c in range(p["chunks"])])
        # both cut points floor to 64 bytes, so every chunk is within 64 of T/C
        assert sizes.sum() == total and np.all(np.abs(sizes - total / p["chunks"]) < 64)
        per_cta = sizes.reshape(-1, G).sum(axis=0)
        assert np.all(np.abs(per_cta - total / G) < 64 * (p["chunks"] // G))
        for c in range(p["chunks"]):
            s0 = total - sizes[c:].sum()
            d = p["chunk_desc"][c]
            assert p["prefix"][d] <= s0 and (s0 < p["prefix"][d + 1] or sizes[c] == 0)
        assert p["chunk_desc"][p["chunks"]] == is_long.sum()
    else:
        assert p["chunks"] == 0

    # short copies: the same multiset, longest first by bucket
    shorts = p["shorts"]
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
    p = pack(harness, desc)
    assert p["grid"] == 608 and p["shorts"].shape[0] == 47520 and p["longs"].shape[0] == 20
    assert p["total"] == 288 << 20 and p["chunks"] == 608 * 8

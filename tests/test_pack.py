"""CPU tests of the batched copy's host packer (tb_pack.cpp), built with g++
against a small harness: the one-pass gather agrees with the counting pass,
short copies keep descriptor order, long copies are listed with their
stream offsets, every CTA gets the same number of equal chunks, and each
chunk's table entry names the long copy that holds its first byte."""
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
    lib.harness_pack.argtypes = [ct.c_void_p, ct.c_size_t, ct.c_uint64, ct.c_uint64, ct.c_int,
                                 ct.c_void_p, ct.c_void_p]
    lib.harness_bad.restype = ct.c_int
    lib.harness_bad.argtypes = [ct.c_void_p, ct.c_size_t, ct.c_void_p]
    lib.harness_overlap.restype = ct.c_int
    lib.harness_overlap.argtypes = [ct.c_void_p, ct.c_size_t, ct.c_void_p]
    lib.harness_short_shape.restype = ct.c_int
    lib.harness_short_shape.argtypes = [ct.c_uint64, ct.c_uint64, ct.c_int, ct.c_uint64]
    return lib


WAVES = 8        # waves of resident CTAs a launch with long copies may span (kBatchWaves)
SHORT_WAVES = 4  # the same for a launch of short copies only (kShortWaves)


def pack(lib, desc, small_max=16384, full_grid=608, ce_min=0):
    desc = np.ascontiguousarray(desc, dtype=np.uint64).reshape(-1, 3)
    n = desc.shape[0]
    cap = 16 + n * 32 + 8 + (16384 + 1) * 4
    buf = np.full(cap, 0xEE, dtype=np.uint8)
    out = np.zeros(12, dtype=np.uint64)
    rc = lib.harness_pack(desc.ctypes.data if n else None, n, small_max, ce_min, full_grid,
                          buf.ctypes.data, out.ctypes.data)
    assert rc == 0
    (n_short, n_long, grid, chunks, total, poff, coff, upload, bound, n_ce, claim,
     direct) = (int(x) for x in out)
    assert upload <= bound <= cap
    assert np.all(buf[:16] == 0)                       # the claim counter starts at 0
    items = buf[16: 16 + (n_short + n_long) * 24].view(np.uint64).reshape(-1, 3)
    prefix = buf[poff: poff + (n_long + 1) * 8].view(np.uint64)
    cdesc = buf[coff: coff + (chunks + 1) * 4].view(np.uint32)
    return dict(shorts=items[:n_short], longs=items[n_short:], prefix=prefix, chunk_desc=cdesc,
                grid=grid, chunks=chunks, total=total, n_ce=n_ce, claim=claim, direct=direct,
                upload=upload)


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
    assert 1 <= G <= grid * (WAVES if is_long.any() else SHORT_WAVES)

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

    # short copies: exactly the short descriptors, in descriptor order
    assert np.array_equal(p["shorts"], desc[(lens > 0) & ~is_long])


@pytest.mark.parametrize("ce_min", [1, 4096, 1 << 20])
def test_packer_copy_engine_split(harness, ce_min):
    g = np.random.default_rng(ce_min)
    desc = random_desc(g, 2000, 0.2, 16384)
    p = pack(harness, desc, ce_min=ce_min)
    lens = desc[:, 2]
    ce = (lens >= ce_min) & (lens > 0)
    assert p["n_ce"] == ce.sum()
    assert np.array_equal(p["shorts"], desc[(lens > 0) & ~ce & (lens <= 16384)])
    assert np.array_equal(p["longs"], desc[~ce & (lens > 16384)])


def test_packer_reports_bad_descriptor(harness):
    desc = np.array([[1, 2, 3], [4, 5, 0], [0, 8, 9], [10, 11, 12]], dtype=np.uint64)
    bad = np.zeros(1, np.uint64)
    assert harness.harness_bad(desc.ctypes.data, 4, bad.ctypes.data) != 0 and bad[0] == 2
    desc[2] = [2**64 - 4, 8, 9]                          # wraps
    assert harness.harness_bad(desc.ctypes.data, 4, bad.ctypes.data) != 0 and bad[0] == 2
    desc[2] = [7, 8, 0]                                  # len 0: skipped, even with null ends
    assert harness.harness_bad(desc.ctypes.data, 4, bad.ctypes.data) == 0


def test_packer_batch_47540(harness):
    from copy_reduce_dst_gb300 import workloads
    lay = workloads.batch_head_sliced()
    desc = lay.descriptors(1 << 32, 1 << 36)
    p = pack(harness, desc)
    assert p["grid"] == 608 * WAVES and p["shorts"].shape[0] == 47520 and p["longs"].shape[0] == 20
    assert p["total"] == 288 << 20 and p["chunks"] == 608 * WAVES
    # its short copies alone: a launch of short copies only, fewer waves
    short = desc[desc[:, 2] <= 16384]
    q = pack(harness, short)
    assert q["grid"] == 608 * SHORT_WAVES and q["chunks"] == 0 and q["claim"] == 2


def short_assignment(n_short, grid, chunks, claim, warps=8):
    """Which warp copies which short copy, following the kernel's rule: the
    warps free at the start take up to `claim` copies each by index (warp
    w: w, w + starters, ...), the rest go out through the counter.  Returns
    the copies of the fixed round and of the counter round, for a coverage
    check."""
    starters = grid * (warps - 1 if chunks else warps)
    fixed = [i for w in range(starters) for i in range(w, starters * claim, starters)
             if i < n_short]
    counted = list(range(starters * claim, n_short))
    return fixed, counted


@pytest.mark.parametrize("n,long_n,expect_grid,expect_claim", [
    (3840, 0, 480, 1), (4864, 0, 608, 1), (4865, 0, 608, 2), (7200, 0, 608, 2),
    (100, 0, 13, 1), (38912, 0, 2432, 2), (47520, 0, 2432, 2), (47520, 20, 4864, 2),
    (1000, 20, 2560, 1)])
def test_grid_claim_items_and_coverage(harness, n, long_n, expect_grid, expect_claim):
    """Short copies only: one warp per copy while a wave's warps suffice,
    else whole waves (at most four) with the copies past the first round
    taken by the warps again.  One copy per starting warp while those warps
    outnumber the short copies, else two; the fixed round and the counter
    together name every short copy exactly once."""
    lens = np.full(n + long_n, 2112, dtype=np.uint64)
    lens[n:] = 8 << 20
    desc = np.stack([np.arange(1, n + long_n + 1, dtype=np.uint64) << np.uint64(24),
                     np.arange(1, n + long_n + 1, dtype=np.uint64) << np.uint64(25), lens], axis=1)
    p = pack(harness, desc)
    assert p["grid"] == expect_grid and p["claim"] == expect_claim
    fixed, counted = short_assignment(n, p["grid"], p["chunks"], p["claim"])
    assert sorted(fixed + counted) == list(range(n))


@pytest.mark.parametrize("n_short,n_long,forced,shape", [
    (3840, 0, 0, 2), (6080, 0, 0, 2), (6081, 0, 0, 1), (47520, 0, 0, 1), (1, 0, 0, 2),
    (3840, 0, 1, 1), (47520, 0, 2, 2), (47520, 20, 1, 0), (0, 3, 2, 0), (3840, 0, 9, 2)])
def test_short_shape_choice(harness, n_short, n_long, forced, shape):
    """Launches with long copies run k_batch (shape 0); short-only ones take a
    forced shape, else the wide shape 2 when every copy gets a warp of its
    first wave (152 SMs x 5 CTAs x 8 warps = 6080 here), else shape 1."""
    assert harness.harness_short_shape(n_short, n_long, forced, 6080) == shape


def _conflict(d, i, j):
    """Brute force: do descriptors i and j (i may equal j) make the result
    order-dependent - a destination over the other's destination (i != j)
    or over a source (its own included)?"""
    def over(a0, alen, b0, blen):
        return alen > 0 and blen > 0 and a0 < b0 + blen and b0 < a0 + alen
    si, di, li = (int(x) for x in d[i])
    sj, dj, lj = (int(x) for x in d[j])
    return ((i != j and over(di, li, dj, lj)) or over(di, li, sj, lj) or over(dj, lj, si, li))


@pytest.mark.parametrize("seed", range(40))
def test_overlap_check_against_brute_force(harness, seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 40))
    span = int(g.integers(200, 20000))      # small address space: overlaps are common
    d = np.stack([g.integers(1, span, n), g.integers(1, span, n),
                  g.integers(0, 300, n)], axis=1).astype(np.uint64)
    pair = np.zeros(2, dtype=np.uint64)
    found = harness.harness_overlap(d.ctypes.data, n, pair.ctypes.data)
    expect = any(_conflict(d, i, j) for i in range(n) for j in range(i, n))
    assert bool(found) == expect
    if found:
        assert _conflict(d, int(min(pair)), int(max(pair)))


def test_overlap_check_cases(harness):
    def run(rows):
        d = np.array(rows, dtype=np.uint64).reshape(-1, 3)
        pair = np.zeros(2, dtype=np.uint64)
        return harness.harness_overlap(d.ctypes.data, d.shape[0], pair.ctypes.data), sorted(pair)
    assert run([[1000, 5000, 100], [1000, 5100, 100]])[0] == 0      # shared source, adjacent dst
    assert run([[1000, 5000, 100], [3000, 5099, 10]]) == (1, [0, 1])  # dst over dst
    assert run([[1000, 5000, 100], [5050, 9000, 10]]) == (1, [0, 1])  # dst over a source
    assert run([[1000, 1050, 100]]) == (1, [0, 0])                    # its own source
    assert run([[1000, 5000, 0], [1000, 5000, 100]])[0] == 0          # empty ranges ignored


@pytest.mark.parametrize("n,long_n,expect", [
    (3840, 0, 1), (1, 0, 1), (7200, 0, 1), (10900, 0, 1), (11000, 0, 0), (3840, 1, 0),
    (0, 5, 0)])
def test_direct_work_list(harness, n, long_n, expect):
    """A launch reads its work list in place from pinned host memory only
    when it has short copies alone, all of them in the fixed first round
    (no counter), and a work list of at most 256 KiB."""
    lens = np.full(n + long_n, 2112, dtype=np.uint64)
    lens[n:] = 8 << 20
    desc = np.stack([np.arange(1, n + long_n + 1, dtype=np.uint64) << np.uint64(24),
                     np.arange(1, n + long_n + 1, dtype=np.uint64) << np.uint64(25), lens], axis=1)
    p = pack(harness, desc)
    assert p["direct"] == expect
    if expect:
        assert p["chunks"] == 0 and p["upload"] <= 256 * 1024
        assert p["shorts"].shape[0] <= p["grid"] * 8 * p["claim"]

"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random numbers and lays out copies; it holds none of the
method's arithmetic (no source pattern, no sum, no copy).  Both the CUDA path
and the CPU oracle receive what it returns.

Workloads (sizes from the configurations the build is measured on):

* ``REDUCE_SINGLE``: TransferBench single transfer, 1 source of 1,048,576
  float32 (4 MiB), SRC_ROTATE_BYTES = 256 MiB so K = 64, 3 warm-up + 10 timed
  iterations (PR #365, "Test Plan": the 4 MB mechanism check).
* ``REDUCE_3SRC``: 3 sources of 67,108,864 float32 (256 MiB each, K = 1),
  sub-executor counts 1, 4, 16, 32; 20 iterations.
* ``COMPRESS_SWEEP``: 1 fillCompress source, 8 MiB .. 512 MiB in powers of
  two, line mix 40% random / 20% 1B0 / 0% 2B0 / 20% 4B0 / 20% 32B0, rotation
  256 MiB and 0 (PR #365's sweep, "cold vs warm, median of 3 reps").
* Batched copies standing in for the Mooncake RFC #5041 P/D shapes
  ("Motivation: measured on real P/D shapes"): the 3840 x 2112 B DSA index
  pages, 7200 block pages of 512 B - 16 KiB, and the 47,520 head-sliced
  pages of 64 B - 16 KiB mixed with 16 x 16 MiB and 4 x 8 MiB copies.  The
  pages' traces are not available; these layouts follow the stated shapes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

KiB = 1 << 10
MiB = 1 << 20
GiB = 1 << 30

DEFAULT_SEED = 0x5EED


# ---------------------------------------------------------------------------
# Reduce-copy workloads
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class ReduceWorkload:
    name: str
    n_src: int
    num_bytes: int
    rotate_bytes: int
    iters: int
    warmup: int
    subexecs: tuple = (0,)
    pattern: str = "default"      # "default" (PrepSrcValue) or "compress"
    compress_pct: tuple = (40, 20, 0, 20, 20)


REDUCE_SINGLE = ReduceWorkload("single transfer, 1 source, 4 MiB, K=64", 1, 4 * MiB, 256 * MiB,
                               iters=10, warmup=3)
REDUCE_3SRC = ReduceWorkload("3-source reduce-copy, 3 x 256 MiB fp32, K=1", 3, 256 * MiB,
                             256 * MiB, iters=20, warmup=3, subexecs=(1, 4, 16, 32))
COMPRESS_SIZES = tuple(s * MiB for s in (8, 16, 32, 64, 128, 256, 512))
COMPRESS_SWEEP = tuple(
    ReduceWorkload(f"fillCompress sweep {s // MiB} MiB", 1, s, 256 * MiB, iters=3, warmup=3,
                   pattern="compress")
    for s in COMPRESS_SIZES)


# ---------------------------------------------------------------------------
# Random bytes
# ---------------------------------------------------------------------------
def random_bytes(n: int, seed: int) -> np.ndarray:
    """n uniformly random bytes from a Philox stream seeded with ``seed``."""
    words = (n + 7) // 8
    raw = np.random.Philox(seed).random_raw(words)
    return raw.view(np.uint8)[:n]


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------------------
# Batch layouts
# ---------------------------------------------------------------------------
@dataclass
class BatchLayout:
    """Copies as byte offsets into a source pool and a destination pool."""
    name: str
    src_off: np.ndarray
    dst_off: np.ndarray
    lens: np.ndarray
    src_pool_bytes: int
    dst_pool_bytes: int
    notes: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.lens.size)

    @property
    def total_bytes(self) -> int:
        return int(self.lens.sum())

    def descriptors(self, src_base: int, dst_base: int) -> np.ndarray:
        """(n, 3) uint64 rows (src address, dst address, len) for pools at the
        given base addresses."""
        d = np.empty((self.n, 3), dtype=np.uint64)
        d[:, 0] = np.uint64(src_base) + self.src_off
        d[:, 1] = np.uint64(dst_base) + self.dst_off
        d[:, 2] = self.lens
        return d


def log_uniform_lengths(g: np.random.Generator, n: int, lo: int, hi: int,
                        multiple: int = 1) -> np.ndarray:
    """L = exp(U(ln lo, ln hi)) rounded down to a multiple of ``multiple``,
    clamped to [lo, hi]."""
    x = np.exp(g.uniform(np.log(lo), np.log(hi), n))
    L = (np.floor(x / multiple) * multiple).astype(np.uint64)
    return np.clip(L, lo, hi).astype(np.uint64)


def scatter_offsets(g: np.random.Generator, lens: np.ndarray, lo: int, hi: int,
                    align: int) -> np.ndarray:
    """Non-overlapping offsets in [lo, hi): the copies are laid out in a random
    order, each start aligned to ``align``, separated by random aligned gaps
    (a random partition of the free space by sorted uniform cut points)."""
    occ = ((lens + np.uint64(align - 1)) // np.uint64(align)) * np.uint64(align)
    free = (hi - lo) - int(occ.sum())
    if free < 0:
        raise ValueError("copies do not fit in the region")
    order = g.permutation(lens.size)
    cuts = np.sort(g.integers(0, free // align + 1, size=lens.size, dtype=np.uint64))
    occ_sorted = occ[order]
    prefix = np.cumsum(occ_sorted, dtype=np.uint64) - occ_sorted
    off = np.empty(lens.size, dtype=np.uint64)
    off[order] = np.uint64(lo) + cuts * np.uint64(align) + prefix
    return off


def batch_index_pages(seed: int = DEFAULT_SEED) -> BatchLayout:
    """3840 copies of 2112 B from a contiguous source into 3840 distinct
    2112 B-aligned slots at random permuted offsets of a 1 GiB pool."""
    g = rng(seed)
    n, size = 3840, 2112
    slots = GiB // size
    dst_slot = g.choice(slots, size=n, replace=False).astype(np.uint64)
    lens = np.full(n, size, dtype=np.uint64)
    src_off = np.arange(n, dtype=np.uint64) * np.uint64(size)
    return BatchLayout("3840 x 2112 B index pages into a 1 GiB pool", src_off,
                       dst_slot * np.uint64(size), lens, n * size, GiB)


def batch_block_pages(seed: int = DEFAULT_SEED + 1) -> BatchLayout:
    """7200 copies, log-uniform 512 B - 16 KiB (any byte count), 64 B-aligned
    random non-overlapping offsets in 1 GiB source and destination pools."""
    g = rng(seed)
    n = 7200
    lens = log_uniform_lengths(g, n, 512, 16 * KiB)
    src_off = scatter_offsets(g, lens, 0, GiB, 64)
    dst_off = scatter_offsets(g, lens, 0, GiB, 64)
    return BatchLayout("7200 block pages, 512 B-16 KiB", src_off, dst_off, lens, GiB, GiB)


def batch_head_sliced(seed: int = DEFAULT_SEED + 2, pool_bytes: int = 2 * GiB,
                      n_small: int = 47520) -> BatchLayout:
    """47,520 copies log-uniform 64 B - 16 KiB (multiples of 64 B) at random
    non-overlapping offsets of two pools, mixed with 16 x 16 MiB and 4 x 8 MiB
    contiguous copies occupying the pools' first 288 MiB; descriptor order is
    a random shuffle of all 47,540."""
    g = rng(seed)
    big = np.array([16 * MiB] * 16 + [8 * MiB] * 4, dtype=np.uint64)
    big_off = np.cumsum(big, dtype=np.uint64) - big
    reserved = int(big.sum())
    small = log_uniform_lengths(g, n_small, 64, 16 * KiB, multiple=64)
    s_src = scatter_offsets(g, small, reserved, pool_bytes, 64)
    s_dst = scatter_offsets(g, small, reserved, pool_bytes, 64)
    lens = np.concatenate([big, small])
    src_off = np.concatenate([big_off, s_src])
    dst_off = np.concatenate([big_off, s_dst])
    order = g.permutation(lens.size)
    return BatchLayout("47,520 head-sliced pages + 16x16 MiB + 4x8 MiB", src_off[order],
                       dst_off[order], lens[order], pool_bytes, pool_bytes,
                       notes={"small": n_small, "large": int(big.size)})


def random_batch(seed: int, n: int, max_len: int, pool_bytes: int,
                 align: int = 1, min_len: int = 0) -> BatchLayout:
    """n copies of uniformly random length in [min_len, max_len] at random
    non-overlapping offsets aligned to ``align`` (1 = any byte)."""
    g = rng(seed)
    lens = g.integers(min_len, max_len + 1, size=n, dtype=np.uint64)
    src_off = scatter_offsets(g, lens, 0, pool_bytes, align)
    dst_off = scatter_offsets(g, lens, 0, pool_bytes, align)
    return BatchLayout(f"{n} random copies up to {max_len} B", src_off, dst_off, lens,
                       pool_bytes, pool_bytes)

"""CPU oracle for the reduce-copy and batched-copy path (test infrastructure).

Only the tests, the smoke check and the bench's CPU-baseline leg may import
this package.  It wraps the plain single-threaded C in ``oracle.c`` (built by
``_build.py`` with gcc) and shares nothing with the CUDA library: no code, no
header, no table.  Each wrapper names the passage it restates:

* TransferBench data validation (ROCm docs 1.66.02): "Expected source pattern"
  (PrepSrcValue, fillCompress, fillPattern), "Expected destination
  (dstReference)", and step 3 of "How validation (ValidateAllTransfers) works".
* TransferBench PR #365 (SRC_ROTATE_BYTES), "Technical Details": the K rule,
  the allocation size and the fold of the iteration into [0, K).
* Mooncake RFC #5041, "Design of #5040": a (src, dst, len) descriptor array
  applied as plain memcpys.

Parity status: every function is pinned by the ``-m "not gpu"`` tests.  The
pages name ``fill_compress``'s zeroing modes without defining them, so it
follows a stated reading, pinned by hand-worked words in
``tests/golden/fill_compress.txt``.
"""
import ctypes as _ct

import numpy as _np

from . import _build

_lib = _ct.CDLL(_build.build())

_u64 = _ct.c_uint64
_i64 = _ct.c_int64
_vp = _ct.c_void_p

_lib.orc_prep_src_value.restype = _ct.c_float
_lib.orc_prep_src_value.argtypes = [_i64, _u64]
_lib.orc_prepare_reference_default.restype = None
_lib.orc_prepare_reference_default.argtypes = [_vp, _u64, _i64]
_lib.orc_fill_pattern.restype = None
_lib.orc_fill_pattern.argtypes = [_vp, _u64, _vp, _u64]
_lib.orc_splitmix64_stream.restype = None
_lib.orc_splitmix64_stream.argtypes = [_u64, _vp, _u64]
_lib.orc_fill_compress.restype = _ct.c_int
_lib.orc_fill_compress.argtypes = [_vp, _u64, _vp, _u64, _i64]
_lib.orc_dst_reference.restype = None
_lib.orc_dst_reference.argtypes = [_vp, _ct.c_int, _u64, _ct.c_uint8, _vp]
_lib.orc_rotation_plan.restype = _ct.c_int
_lib.orc_rotation_plan.argtypes = [_u64, _u64, _u64, _ct.POINTER(_u64),
                                   _ct.POINTER(_u64), _ct.POINTER(_u64)]
_lib.orc_slice_for_iteration.restype = _u64
_lib.orc_slice_for_iteration.argtypes = [_i64, _u64]
_lib.orc_apply_batch.restype = _ct.c_int
_lib.orc_apply_batch.argtypes = [_vp, _u64, _vp, _u64, _vp, _vp, _vp, _u64]
_lib.orc_first_mismatch.restype = _i64
_lib.orc_first_mismatch.argtypes = [_vp, _vp, _u64, _u64]


def _ptr(a: _np.ndarray) -> int:
    if not a.flags.c_contiguous:
        raise ValueError("oracle arrays must be C-contiguous")
    return a.ctypes.data


def prep_src_value(buffer_idx: int, i: int) -> float:
    """PrepSrcValue(bufferIdx, i) of the "Expected source pattern" default row."""
    return float(_lib.orc_prep_src_value(buffer_idx, i))


def prepare_reference(n: int, buffer_idx: int) -> _np.ndarray:
    """The default source pattern for SRC ``buffer_idx``: n float32 values."""
    out = _np.empty(n, dtype=_np.float32)
    _lib.orc_prepare_reference_default(_ptr(out), n, buffer_idx)
    return out


def fill_pattern(n: int, pattern) -> _np.ndarray:
    """fillPattern: the given float vector repeated over n elements."""
    pat = _np.ascontiguousarray(pattern, dtype=_np.float32)
    if pat.size == 0:
        raise ValueError("fillPattern needs at least one value")
    out = _np.empty(n, dtype=_np.float32)
    _lib.orc_fill_pattern(_ptr(out), n, _ptr(pat), pat.size)
    return out


def splitmix64_stream(seed: int, count: int) -> _np.ndarray:
    """The first ``count`` SplitMix64 outputs of the stream seeded with ``seed``."""
    out = _np.empty(count, dtype=_np.uint64)
    _lib.orc_splitmix64_stream(seed & (2**64 - 1), _ptr(out), count)
    return out


def fill_compress(n: int, pct, seed: int, buffer_idx: int = 0) -> _np.ndarray:
    """fillCompress: random floats with per-64-byte-line zeroing (the stated reading,
    pinned by tests/golden/fill_compress.txt)."""
    p = _np.ascontiguousarray(pct, dtype=_np.uint32)
    if p.size != 5:
        raise ValueError("fillCompress takes five percentages")
    out = _np.empty(n, dtype=_np.float32)
    if _lib.orc_fill_compress(_ptr(out), n, _ptr(p), seed & (2**64 - 1), buffer_idx) != 0:
        raise ValueError("fillCompress percentages must sum to 100")
    return out


def dst_reference(src_refs, n: int | None = None, memset_byte: int = 0) -> _np.ndarray:
    """dstReference[len(src_refs)]: the expected destination for that many sources."""
    srcs = [_np.ascontiguousarray(s, dtype=_np.float32) for s in src_refs]
    if n is None:
        if not srcs:
            raise ValueError("n is required when there are no sources")
        n = srcs[0].size
    if any(s.size != n for s in srcs):
        raise ValueError("every source must hold n elements")
    out = _np.empty(n, dtype=_np.float32)
    arr = (_vp * max(1, len(srcs)))(*[_ptr(s) for s in srcs])
    _lib.orc_dst_reference(arr, len(srcs), n, memset_byte & 0xFF, _ptr(out))
    return out


def rotation_plan(num_bytes: int, rotate_bytes: int, byte_offset: int = 0):
    """(K, slice stride, allocation bytes) of SRC_ROTATE_BYTES rotation."""
    k, s, a = _u64(), _u64(), _u64()
    if _lib.orc_rotation_plan(num_bytes, rotate_bytes, byte_offset,
                              _ct.byref(k), _ct.byref(s), _ct.byref(a)) != 0:
        raise ValueError("invalid rotation plan arguments")
    return k.value, s.value, a.value


def slice_for_iteration(iteration: int, k: int) -> int:
    """Slice read by iteration ``iteration`` (folded into [0, K))."""
    return int(_lib.orc_slice_for_iteration(iteration, k))


def apply_batch(dst_pool: _np.ndarray, src_pool: _np.ndarray,
                src_off, dst_off, lens) -> None:
    """Applies the (src, dst, len) descriptors to host pools, in array order."""
    if dst_pool.dtype != _np.uint8 or src_pool.dtype != _np.uint8:
        raise TypeError("pools are uint8 arrays")
    so = _np.ascontiguousarray(src_off, dtype=_np.uint64)
    do = _np.ascontiguousarray(dst_off, dtype=_np.uint64)
    ln = _np.ascontiguousarray(lens, dtype=_np.uint64)
    if not (so.size == do.size == ln.size):
        raise ValueError("descriptor arrays differ in length")
    if _lib.orc_apply_batch(_ptr(dst_pool), dst_pool.size, _ptr(src_pool),
                            src_pool.size, _ptr(so), _ptr(do), _ptr(ln), ln.size) != 0:
        raise ValueError("descriptor outside its pool")


def first_mismatch(actual: _np.ndarray, expected: _np.ndarray) -> int:
    """First differing element index of two same-typed arrays, or -1 if equal."""
    a = _np.ascontiguousarray(actual)
    e = _np.ascontiguousarray(expected)
    if a.nbytes != e.nbytes or a.itemsize != e.itemsize:
        raise ValueError("arrays differ in size or element type")
    return int(_lib.orc_first_mismatch(_ptr(a), _ptr(e), a.nbytes, a.itemsize))

"""Python binding of libtb (include/tb.h): argument marshalling only.

Every operation runs in the CUDA library; this module converts tensors,
integers and streams into the plain pointers and sizes the C ABI takes, and
turns error codes into ``TBError``.  PyTorch is optional here: anything with
``data_ptr()`` (a tensor) or a plain integer address is accepted as a
pointer, and anything with ``cuda_stream`` (a ``torch.cuda.Stream``) or an
integer handle as a stream.

Importing this module loads ``lib/libtb.so`` and fails loudly when it has not
been built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as ct
import os
from dataclasses import dataclass

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libtb.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libtb.so is not built ({LIB_PATH} missing): run "
        "`python -c 'import __graft_entry__ as g; g.build()'` first")

lib = ct.CDLL(LIB_PATH)

TB_OK = 0
TB_EINVAL = -1
TB_ENOMEM = -2
TB_ECUDA = -3
TB_EVALIDATE = -4
TB_ETIMEOUT = -5
TB_ENOTSUP = -6
TB_MAX_SRCS = 16

TB_PATTERN_DEFAULT = 0
TB_PATTERN_COMPRESS = 1
TB_PATTERN_REPEAT = 2

_u64, _i64, _i32, _u32, _vp = ct.c_uint64, ct.c_int64, ct.c_int32, ct.c_uint32, ct.c_void_p


class Options(ct.Structure):
    """tb_options: see include/tb.h for every field's meaning and default."""
    _fields_ = [
        ("rotate_bytes", _u64),
        ("byte_offset", _u64),
        ("warmup", _i32),
        ("always_validate", _i32),
        ("memset_byte", _u32),
        ("ctas_per_subexec", _i32),
        ("block_threads", _i32),
        ("small_max_bytes", _u64),
        ("slot_items", _u32),
        ("num_slots", _u32),
        ("wait_timeout_ns", _u64),
        ("use_gate", _i32),
        ("vec_bytes", _i32),
        ("unroll", _i32),
        ("time_kernels", _i32),
        ("reduce_engine", _i32),
        ("ce_min_bytes", _u64),
        ("use_graph", _i32),
        ("use_pdl", _i32),
        ("kernel_wait_ns", _u64),
        ("validate_direct", _i32),
        ("validate_source", _i32),
        ("check_overlap", _i32),
        ("batch_min_copies", _i32),
        ("batch_short_shape", _i32),
        ("batch_max_ctas", _i32),
        ("early_reads", _i32),
    ]


class Pattern(ct.Structure):
    _fields_ = [
        ("kind", _i32),
        ("compress_pct", _u32 * 5),
        ("seed", _u64),
        ("repeat", ct.POINTER(ct.c_float)),
        ("repeat_len", _u32),
    ]


class Result(ct.Structure):
    _fields_ = [
        ("K", _u64),
        ("slice_stride", _u64),
        ("alloc_bytes", _u64),
        ("prep_h2d_bytes", _u64),
        ("iters", _i32),
        ("num_subexec", _i32),
        ("ctas", _i32),
        ("block_threads", _i32),
        ("gated", _i32),
        ("graphed", _i32),
        ("engine", _i32),
        ("validated", _i32),
        ("total_ms", ct.c_double),
        ("mean_ms", ct.c_double),
        ("median_ms", ct.c_double),
        ("min_ms", ct.c_double),
        ("max_ms", ct.c_double),
        ("gbps", ct.c_double),
        ("iter_ms", ct.POINTER(ct.c_float)),
        ("mismatch_index", _i64),
        ("mismatch_expected", _u32),
        ("mismatch_actual", _u32),
        ("executor", _i32),
    ]


class LaunchInfo(ct.Structure):
    _fields_ = [
        ("engine", _i32),
        ("vec_bytes", _i32),
        ("unroll", _i32),
        ("block_threads", _i32),
        ("grid", _i32),
        ("num_subexec", _i32),
        ("head_elems", _u64),
        ("body_vectors", _u64),
        ("tail_elems", _u64),
        ("smem_bytes", _u64),
        ("stages", _i32),
        ("tile_bytes", _i32),
    ]


class Transfer(ct.Structure):
    _fields_ = [
        ("srcs", ct.POINTER(_vp)),
        ("n_src", _i32),
        ("dst", _vp),
        ("num_bytes", _u64),
        ("num_subexec", _i32),
        ("iters", _i32),
        ("rotate_bytes", _u64),
        ("expected", _vp),
        ("expected_device", _vp),
        ("executor", _i32),
    ]


class CopyDesc(ct.Structure):
    _fields_ = [("src", _u64), ("dst", _u64), ("len", _u64)]


class BatchStats(ct.Structure):
    _fields_ = [
        ("descs", _u64),
        ("warp_items", _u64),
        ("cta_items", _u64),
        ("launches", _u64),
        ("bytes", _u64),
        ("upload_bytes", _u64),
        ("ce_copies", _u64),
        ("direct_launches", _u64),
    ]


class Mismatch(ct.Structure):
    _fields_ = [("index", _i64), ("expected", _u32), ("actual", _u32)]


def _sig(name, restype, *argtypes):
    fn = getattr(lib, name)
    fn.restype = restype
    fn.argtypes = list(argtypes)
    return fn


_P = ct.POINTER
_sig("tb_strerror", ct.c_char_p, ct.c_int)
_sig("tb_last_error", ct.c_char_p, _vp)
_sig("tb_options_default", None, _P(Options))
_sig("tb_options_from_env", ct.c_int, _P(Options))
_sig("tb_parse_bytes", ct.c_int, ct.c_char_p, _P(_u64))
_sig("tb_create", ct.c_int, _P(_vp), ct.c_int, _P(Options))
_sig("tb_destroy", None, _vp)
_sig("tb_get_options", ct.c_int, _vp, _P(Options))
_sig("tb_rotation_plan", ct.c_int, _u64, _u64, _u64, _P(_u64), _P(_u64), _P(_u64))
_sig("tb_slice_for_iteration", _u64, _i64, _u64)
_sig("tb_fill_source", ct.c_int, _vp, _vp, _u64, _P(Pattern), ct.c_int, _vp)
_sig("tb_upload_sources", ct.c_int, _vp, _P(_vp), _P(_vp), ct.c_int, _u64)
_sig("tb_prepare_sources", ct.c_int, _vp, _P(_vp), ct.c_int, _u64, _u64)
_sig("tb_prep_h2d_bytes", _u64, _vp)
_sig("tb_reduce_copy", ct.c_int, _vp, _P(_vp), ct.c_int, _vp, _u64, ct.c_int, _vp)
_sig("tb_reduce_plan", ct.c_int, _vp, _P(_vp), ct.c_int, _vp, _u64, ct.c_int, _P(LaunchInfo))
_sig("tb_run_transfer_ex", ct.c_int, _vp, _P(Transfer), _P(Result))
_sig("tb_run_transfer", ct.c_int, _vp, _P(_vp), ct.c_int, _vp, _u64, ct.c_int, ct.c_int, _u64,
     _P(Result))
_sig("tb_reduce_copy_host", ct.c_int, _vp, _P(_vp), ct.c_int, _vp, _u64, _P(_vp), _vp, ct.c_int,
     _vp)
_sig("tb_batch_copy", ct.c_int, _vp, _vp, ct.c_size_t, _vp)  # desc: a CopyDesc array's address
_sig("tb_last_batch_stats", ct.c_int, _vp, _P(BatchStats))
_sig("tb_last_batch_kernel_ms", ct.c_int, _vp, _P(ct.c_double))
_sig("tb_copy_each", ct.c_int, _vp, _vp, ct.c_size_t, _vp)  # desc: a CopyDesc array's address
_sig("tb_validate", ct.c_int, _vp, _vp, _vp, _u64, _u32, _P(Mismatch))
_sig("tb_validate_device", ct.c_int, _vp, _vp, _vp, _u64, _u32, _P(Mismatch))
_sig("tb_batch_copy_noalloc", ct.c_int, _vp, ct.c_size_t, _vp)  # desc: as tb_batch_copy

TB_NOALLOC_MAX_ITEMS = 65536
TB_EXEC_GPU = 0
TB_EXEC_DMA = 1


class TBError(RuntimeError):
    """A libtb call returned a negative code."""

    def __init__(self, code: int, message: str):
        super().__init__(message)
        self.code = code


def strerror(code: int) -> str:
    return lib.tb_strerror(code).decode()


def _check(code: int, ctx_handle=None, what: str = "") -> int:
    if code != TB_OK:
        detail = lib.tb_last_error(ctx_handle).decode() if ctx_handle else ""
        raise TBError(code, f"{what}: {strerror(code)}" + (f" ({detail})" if detail else ""))
    return code


def addr(x) -> int:
    """Device or host address of a tensor / array / integer."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):  # numpy array
        return int(x.ctypes.data)
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def stream_handle(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError(f"not a stream: {type(s).__name__}")


def _ptr_array(xs):
    arr = (_vp * max(1, len(xs)))(*[addr(x) for x in xs])
    return arr


def options(**overrides) -> Options:
    """Default options (no environment), with keyword overrides."""
    o = Options()
    lib.tb_options_default(ct.byref(o))
    for k, v in overrides.items():
        if not hasattr(o, k):
            raise AttributeError(f"tb_options has no field {k}")
        setattr(o, k, v)
    return o


def options_from_env(base: Options | None = None) -> Options:
    o = base if base is not None else options()
    _check(lib.tb_options_from_env(ct.byref(o)), None, "tb_options_from_env")
    return o


def parse_bytes(text: str) -> int:
    out = _u64()
    _check(lib.tb_parse_bytes(text.encode(), ct.byref(out)), None, f"tb_parse_bytes({text!r})")
    return out.value


@dataclass
class RotationPlan:
    K: int
    slice_stride: int
    alloc_bytes: int


def rotation_plan(num_bytes: int, rotate_bytes: int, byte_offset: int = 0) -> RotationPlan:
    k, s, a = _u64(), _u64(), _u64()
    _check(lib.tb_rotation_plan(num_bytes, rotate_bytes, byte_offset, ct.byref(k), ct.byref(s),
                                ct.byref(a)), None, "tb_rotation_plan")
    return RotationPlan(k.value, s.value, a.value)


def slice_for_iteration(iteration: int, K: int) -> int:
    return int(lib.tb_slice_for_iteration(iteration, K))


def default_pattern() -> Pattern:
    return Pattern(kind=TB_PATTERN_DEFAULT)


def compress_pattern(pct, seed: int) -> Pattern:
    p = Pattern(kind=TB_PATTERN_COMPRESS, seed=seed & (2**64 - 1))
    for i, v in enumerate(pct):
        p.compress_pct[i] = v
    return p


def repeat_pattern(values) -> tuple[Pattern, object]:
    buf = (ct.c_float * len(values))(*values)
    p = Pattern(kind=TB_PATTERN_REPEAT, repeat=ct.cast(buf, ct.POINTER(ct.c_float)),
                repeat_len=len(values))
    return p, buf  # keep buf alive for the call


class Context:
    """A libtb context on one CUDA device (tb_create / tb_destroy)."""

    def __init__(self, device: int = 0, opts: Options | None = None, env: bool = False):
        self._h = _vp()
        if opts is None and env:
            popt = None
        else:
            popt = ct.byref(opts if opts is not None else options())
        code = lib.tb_create(ct.byref(self._h), device, popt)
        if code != TB_OK:
            raise TBError(code, f"tb_create(device={device}): {strerror(code)}")
        self.device = device

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            lib.tb_destroy(self._h)
            self._h = _vp()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ok(self, code, what):
        return _check(code, self._h, what)

    def get_options(self) -> Options:
        o = Options()
        self._ok(lib.tb_get_options(self._h, ct.byref(o)), "tb_get_options")
        return o

    # -- source preparation ------------------------------------------------
    def fill_source(self, dst, num_bytes: int, pattern: Pattern, buffer_idx: int, stream=None):
        self._ok(lib.tb_fill_source(self._h, addr(dst), num_bytes, ct.byref(pattern), buffer_idx,
                                    stream_handle(stream)), "tb_fill_source")

    def upload_sources(self, srcs, host_srcs, num_bytes: int):
        self._ok(lib.tb_upload_sources(self._h, _ptr_array(srcs), _ptr_array(host_srcs), len(srcs),
                                       num_bytes), "tb_upload_sources")

    def prepare_sources(self, srcs, num_bytes: int, rotate_bytes: int):
        self._ok(lib.tb_prepare_sources(self._h, _ptr_array(srcs), len(srcs), num_bytes,
                                        rotate_bytes), "tb_prepare_sources")

    @property
    def prep_h2d_bytes(self) -> int:
        return int(lib.tb_prep_h2d_bytes(self._h))

    # -- reduce-copy -------------------------------------------------------
    def reduce_copy(self, srcs, dst, num_bytes: int, num_subexec: int = 0, stream=None):
        self._ok(lib.tb_reduce_copy(self._h, _ptr_array(srcs), len(srcs), addr(dst), num_bytes,
                                    num_subexec, stream_handle(stream)), "tb_reduce_copy")

    def reduce_plan(self, srcs, dst, num_bytes: int, num_subexec: int = 0) -> dict:
        """The launch tb_reduce_copy would make (tb_reduce_plan), as a dict."""
        info = LaunchInfo()
        self._ok(lib.tb_reduce_plan(self._h, _ptr_array(srcs), len(srcs), addr(dst), num_bytes,
                                    num_subexec, ct.byref(info)), "tb_reduce_plan")
        return {name: getattr(info, name) for name, _ in LaunchInfo._fields_}

    def run_transfer(self, srcs, dst, num_bytes: int, num_subexec: int = 0, iters: int = 1,
                     rotate_bytes: int | None = None, expected=None,
                     expected_device=None, executor: int = 0) -> dict:
        """tb_run_transfer_ex; returns the tb_result fields as a dict.

        ``expected`` (host bytes, e.g. a numpy array) turns on validation; a
        mismatch raises TBError with code TB_EVALIDATE after filling the
        result, which is attached to the exception as ``.result``.
        ``executor``: TB_EXEC_GPU (the reduce-copy kernel) or TB_EXEC_DMA (one
        copy-engine copy per iteration, one source).
        """
        if rotate_bytes is None:
            rotate_bytes = self.get_options().rotate_bytes
        arr = _ptr_array(srcs)
        t = Transfer(srcs=ct.cast(arr, ct.POINTER(_vp)), n_src=len(srcs), dst=addr(dst),
                     num_bytes=num_bytes, num_subexec=num_subexec, iters=iters,
                     rotate_bytes=rotate_bytes, expected=addr(expected) if expected is not None else 0,
                     expected_device=addr(expected_device), executor=executor)
        r = Result()
        code = lib.tb_run_transfer_ex(self._h, ct.byref(t), ct.byref(r))
        res = {name: getattr(r, name) for name, _ in Result._fields_ if name != "iter_ms"}
        res["iter_ms"] = [r.iter_ms[i] for i in range(r.iters)] if r.iters > 0 and r.iter_ms else []
        if code != TB_OK:
            err = TBError(code, f"tb_run_transfer_ex: {strerror(code)} "
                                f"({lib.tb_last_error(self._h).decode()})")
            err.result = res
            raise err
        return res

    def reduce_copy_host(self, host_srcs, host_dst, num_bytes: int, dev_srcs, dev_dst,
                         num_subexec: int = 0, stream=None):
        self._ok(lib.tb_reduce_copy_host(self._h, _ptr_array(host_srcs), len(host_srcs),
                                         addr(host_dst), num_bytes, _ptr_array(dev_srcs),
                                         addr(dev_dst), num_subexec, stream_handle(stream)),
                 "tb_reduce_copy_host")

    # -- batched copy ------------------------------------------------------
    @staticmethod
    def descriptor_array(descs):
        """(address, count, keep-alive) for a ctypes CopyDesc array or an
        (n, 3) uint64 array of (src, dst, len) rows.  The address is taken
        without a ctypes pointer object, which would cost more than the rest
        of a small call's host work."""
        if isinstance(descs, ct.Array):
            return ct.addressof(descs), len(descs), descs
        import numpy as np
        a = np.ascontiguousarray(descs, dtype=np.uint64)
        if a.ndim != 2 or a.shape[1] != 3:
            raise ValueError("descriptors must be an (n, 3) array of (src, dst, len)")
        n = a.shape[0]
        if n == 0:
            return None, 0, a
        try:
            ptr = ct.addressof(ct.c_uint64.from_buffer(a))
        except (TypeError, ValueError):  # a read-only array
            ptr = a.ctypes.data
        return ptr, n, a

    def batch_copy(self, descs, stream=None):
        """tb_batch_copy of (src, dst, len) descriptors (see descriptor_array)."""
        ptr, n, keep = self.descriptor_array(descs)
        self._ok(lib.tb_batch_copy(self._h, ptr, n, stream_handle(stream)), "tb_batch_copy")
        del keep

    def copy_each(self, descs, stream=None):
        """tb_copy_each: one cudaMemcpyAsync per descriptor (the baseline)."""
        ptr, n, keep = self.descriptor_array(descs)
        self._ok(lib.tb_copy_each(self._h, ptr, n, stream_handle(stream)), "tb_copy_each")
        del keep

    def last_batch_kernel_ms(self) -> float:
        ms = ct.c_double()
        self._ok(lib.tb_last_batch_kernel_ms(self._h, ct.byref(ms)), "tb_last_batch_kernel_ms")
        return ms.value

    def last_batch_stats(self) -> dict:
        s = BatchStats()
        self._ok(lib.tb_last_batch_stats(self._h, ct.byref(s)), "tb_last_batch_stats")
        return {name: getattr(s, name) for name, _ in BatchStats._fields_}

    # -- validation --------------------------------------------------------
    def validate_device(self, dst_device, expected_device, num_bytes: int, elem_size: int = 4):
        """tb_validate_device: None when equal, else (index, expected_bits, actual_bits)."""
        m = Mismatch()
        code = lib.tb_validate_device(self._h, addr(dst_device), addr(expected_device), num_bytes,
                                      elem_size, ct.byref(m))
        if code == TB_EVALIDATE:
            return (m.index, m.expected, m.actual)
        self._ok(code, "tb_validate_device")
        return None

    def validate(self, dst_device, expected_host, num_bytes: int, elem_size: int = 4):
        """Returns None when equal, else (index, expected_bits, actual_bits)."""
        m = Mismatch()
        code = lib.tb_validate(self._h, addr(dst_device), addr(expected_host), num_bytes,
                               elem_size, ct.byref(m))
        if code == TB_EVALIDATE:
            return (m.index, m.expected, m.actual)
        self._ok(code, "tb_validate")
        return None


def batch_copy_noalloc(descs, stream=None) -> None:
    """tb_batch_copy_noalloc on the current CUDA device: the batched copy for
    callers that cannot allocate device memory (its work items live in a
    fixed array inside the library).  Raises TBError on a nonzero code."""
    ptr, n, keep = Context.descriptor_array(descs)
    code = lib.tb_batch_copy_noalloc(ptr, n, stream_handle(stream))
    del keep
    _check(code, None, "tb_batch_copy_noalloc")

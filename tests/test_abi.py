"""CPU tests of the C ABI: the library builds, loads and exports every entry
point include/tb.h declares, and its host-only logic (rotation plan, slice
fold, byte parser, options, batch layouts) agrees with the oracle and the
pinned values.  No compute call runs here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from copy_reduce_dst_gb300 import _build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tb.h")


@pytest.fixture(scope="module")
def tb():
    _build.build()
    from copy_reduce_dst_gb300 import tb as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(tb_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tb_create", "tb_destroy", "tb_run_transfer", "tb_batch_copy",
                     "tb_validate", "tb_rotation_plan", "tb_prepare_sources", "tb_reduce_copy",
                     "tb_strerror"):
        assert required in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol(tb):
    lib = ctypes.CDLL(tb.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_library_exports_only_tb_symbols(tb):
    # dynamic symbol table: everything we define globally starts with tb_
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", tb.LIB_PATH], capture_output=True,
                         text=True).stdout
    ours = [l.split()[-1] for l in out.splitlines() if l.split()[-2] == "T"
            and l.split()[-1].startswith("tb_")]
    assert set(ours) >= set(declared_functions())


def test_rotation_plan_matches_oracle_and_pins(tb, golden):
    for nb, rb, off, k, alloc in golden("rotation.txt"):
        p = tb.rotation_plan(int(nb), int(rb), int(off))
        assert (p.K, p.alloc_bytes) == (int(k), int(alloc))
    g = np.random.default_rng(5)
    cases = [(int(g.integers(1, 1 << 34)), int(g.integers(0, 1 << 36)), 4 * int(g.integers(0, 64)))
             for _ in range(300)]
    cases += [(1, 1 << 30, 0), (255, 1000, 4), (256, 256, 0), (257, 256 << 20, 0)]
    for nb, rb, off in cases:
        p = tb.rotation_plan(nb, rb, off)
        assert (p.K, p.slice_stride, p.alloc_bytes) == oracle.rotation_plan(nb, rb, off)
    with pytest.raises(tb.TBError):
        tb.rotation_plan(0, 1)
    with pytest.raises(tb.TBError):
        tb.rotation_plan(1 << 62, 2**64 - 1)


def test_slice_fold_matches_oracle(tb):
    for K in (1, 2, 3, 64, 1000):
        for it in list(range(-70, 70)) + [-(2**40) - 3, 2**40 + 9]:
            assert tb.slice_for_iteration(it, K) == oracle.slice_for_iteration(it, K)


@pytest.mark.parametrize("text,value", [
    ("0", 0), ("4096", 4096), ("256M", 256 << 20), ("256MB", 256 << 20), ("256MiB", 256 << 20),
    ("4k", 4096), (" 2G ", 2 << 30), ("1T", 1 << 40), ("16mb", 16 << 20), ("7b", 7),
    ("18446744073709551615", 2**64 - 1), ("16777215T", 16777215 << 40)])
def test_parse_bytes_accepts(tb, text, value):
    assert tb.parse_bytes(text) == value


@pytest.mark.parametrize("text", ["", "-1", "+5", "12Q", "1.5M", "M", "18446744073709551616",
                                  "16777216T", "99999999999999999999999", "5 M", "0x10"])
def test_parse_bytes_rejects(tb, text):
    with pytest.raises(tb.TBError):
        tb.parse_bytes(text)


def test_options_defaults(tb):
    o = tb.options()
    assert o.rotate_bytes == 256 << 20 and o.warmup == 3 and o.use_gate == 1
    assert o.small_max_bytes == 16384 and o.slot_items == 65536 and o.num_slots == 4
    assert o.always_validate == 0 and o.memset_byte == 0 and o.byte_offset == 0
    assert o.use_graph == 1 and o.reduce_engine == 0 and o.ce_min_bytes == 0 and o.use_pdl == 1
    assert o.time_kernels == 0 and o.vec_bytes == 0 and o.unroll == 0
    assert o.kernel_wait_ns == 2_000_000_000 and o.validate_direct == 0 and o.validate_source == 0
    assert o.batch_short_shape == 0 and o.batch_max_ctas == 0


def test_options_struct_matches_header(tb):
    # every tb_options field of include/tb.h, in order, is in the binding
    text = open(HEADER).read()
    body = text[text.index("typedef struct {\n    /* SRC_ROTATE_BYTES"):text.index("} tb_options;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"^\s*(?:u?int\d+_t)\s+(\w+);", body, flags=re.M)
    assert fields == [name for name, _ in tb.Options._fields_]


@pytest.mark.parametrize("name,cls", [("tb_transfer", "Transfer"), ("tb_result", "Result")])
def test_transfer_and_result_structs_match_header(tb, name, cls):
    # every field of the header's struct, in order, is in the binding
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    end = text.index("} " + name + ";")
    body = text[text.rindex("typedef struct {", 0, end):end]
    fields = []
    for decl in body.split(";")[:-1]:
        decl = decl.split("{")[-1].strip()
        for part in decl.split(","):
            fields.append(re.findall(r"(\w+)\s*$", part.strip())[0])
    assert fields == [f for f, _ in getattr(tb, cls)._fields_]


def test_every_option_has_an_environment_variable(tb):
    # the header's list of variables covers every tb_options field
    text = open(HEADER).read()
    block = text[text.index("Overrides fields of *opt from the environment"):
                 text.index("int tb_options_from_env")]
    names = set(re.findall(r"\bTB_([A-Z_]+)\b", block))
    renamed = {"rotate_bytes": "SRC_ROTATE_BYTES", "memset_byte": "MEMSET_CHAR",
               "batch_min_copies": "BATCH_COPY_MIN"}
    for field, _ in tb.Options._fields_:
        assert renamed.get(field, field.upper()) in names, field


def test_header_environment_list_matches_the_source():
    # every variable the header lists is one tb_options_from_env reads, and back
    text = open(HEADER).read()
    block = text[text.index("Overrides fields of *opt from the environment"):
                 text.index("int tb_options_from_env")]
    listed = set(re.findall(r"\b([A-Z][A-Z0-9]*(?:_[A-Z0-9]+)+)\b", block)) - {"TB_EINVAL"}
    src = open(os.path.join(ROOT, "copy_reduce_dst_gb300", "csrc", "tb_host.cpp")).read()
    body = src[src.index("int tb_options_from_env"):]
    body = body[:body.index("\n}\n")]
    read = set(re.findall(r'env_\w+\("([A-Z0-9_]+)"', body))
    assert listed == read


def test_options_env_new_fields(tb, monkeypatch):
    monkeypatch.setenv("TB_USE_GRAPH", "0")
    monkeypatch.setenv("TB_REDUCE_ENGINE", "2")
    monkeypatch.setenv("TB_CE_MIN_BYTES", "1MiB")
    monkeypatch.setenv("TB_USE_PDL", "0")
    monkeypatch.setenv("TB_KERNEL_WAIT_NS", "0")
    monkeypatch.setenv("TB_BATCH_SHORT_SHAPE", "2")
    monkeypatch.setenv("TB_BATCH_MAX_CTAS", "64")
    monkeypatch.setenv("TB_EARLY_READS", "1")
    o = tb.options_from_env()
    assert o.use_graph == 0 and o.reduce_engine == 2 and o.ce_min_bytes == 1 << 20
    assert o.use_pdl == 0 and o.kernel_wait_ns == 0
    assert o.batch_short_shape == 2 and o.batch_max_ctas == 64 and o.early_reads == 1


def test_validation_options_from_env(tb, monkeypatch):
    # the pages' variable names, and the TB_ ones winning over them
    monkeypatch.setenv("VALIDATE_DIRECT", "1")
    monkeypatch.setenv("VALIDATE_SOURCE", "1")
    o = tb.options_from_env()
    assert o.validate_direct == 1 and o.validate_source == 1
    monkeypatch.setenv("TB_VALIDATE_SOURCE", "0")
    assert tb.options_from_env().validate_source == 0


def test_pages_variable_names_from_env(tb, monkeypatch):
    # TransferBench's MEMSET_CHAR, Mooncake's MC_HIP_BATCH_COPY_MIN
    monkeypatch.setenv("MEMSET_CHAR", "0x")          # does not parse
    with pytest.raises(tb.TBError):
        tb.options_from_env()
    monkeypatch.setenv("MEMSET_CHAR", "90")
    monkeypatch.setenv("MC_HIP_BATCH_COPY_MIN", "16")
    o = tb.options_from_env()
    assert o.memset_byte == 90 and o.batch_min_copies == 16
    monkeypatch.setenv("TB_MEMSET_CHAR", "1")
    monkeypatch.setenv("TB_BATCH_COPY_MIN", "0")
    o = tb.options_from_env()
    assert o.memset_byte == 1 and o.batch_min_copies == 0


def test_options_from_env(tb, monkeypatch):
    monkeypatch.setenv("SRC_ROTATE_BYTES", "64M")
    monkeypatch.setenv("TB_ALWAYS_VALIDATE", "1")
    monkeypatch.setenv("TB_MEMSET_CHAR", "165")
    o = tb.options_from_env()
    assert o.rotate_bytes == 64 << 20 and o.always_validate == 1 and o.memset_byte == 165
    monkeypatch.setenv("TB_SRC_ROTATE_BYTES", "0")
    assert tb.options_from_env().rotate_bytes == 0      # TB_ name wins over the bare one
    monkeypatch.setenv("TB_WARMUP", "-3")
    with pytest.raises(tb.TBError):
        tb.options_from_env()


def test_strerror_names_codes(tb):
    assert "EINVAL" in tb.strerror(tb.TB_EINVAL)
    assert "EVALIDATE" in tb.strerror(tb.TB_EVALIDATE)
    assert "unknown" in tb.strerror(-99)


def test_create_without_gpu_fails_cleanly(tb):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(tb.TBError) as e:
        tb.Context(0)
    assert e.value.code in (tb.TB_ECUDA, tb.TB_EINVAL)


def test_null_context_is_rejected(tb):
    assert tb.lib.tb_reduce_copy(None, None, 0, None, 0, 0, None) == tb.TB_EINVAL
    assert tb.lib.tb_batch_copy(None, None, 0, None) == tb.TB_EINVAL
    tb.lib.tb_destroy(None)


# ---------------------------------------------------------------------------
# Seeded batch layouts: shapes and non-overlap
# ---------------------------------------------------------------------------
def _no_overlap(off, lens):
    o = np.argsort(off, kind="stable")
    s, l = off[o].astype(np.int64), lens[o].astype(np.int64)
    return bool(np.all(s[1:] >= s[:-1] + l[:-1]))


def test_index_pages_layout():
    b = workloads.batch_index_pages()
    assert b.n == 3840 and np.all(b.lens == 2112) and b.dst_pool_bytes == 1 << 30
    assert np.all(b.dst_off % 2112 == 0) and len(set(b.dst_off.tolist())) == 3840
    assert np.all(b.dst_off + b.lens <= b.dst_pool_bytes)
    assert np.array_equal(b.src_off, np.arange(3840, dtype=np.uint64) * 2112)


def test_block_pages_layout():
    b = workloads.batch_block_pages()
    assert b.n == 7200 and b.lens.min() >= 512 and b.lens.max() <= 16384
    assert np.all(b.src_off % 64 == 0) and np.all(b.dst_off % 64 == 0)
    assert _no_overlap(b.src_off, b.lens) and _no_overlap(b.dst_off, b.lens)
    assert np.any(b.lens % 64 != 0)     # unaligned tails occur


def test_head_sliced_layout():
    b = workloads.batch_head_sliced()
    assert b.n == 47540
    big = b.lens > 16384
    assert big.sum() == 20 and sorted(b.lens[big].tolist()) == [8 << 20] * 4 + [16 << 20] * 16
    small = b.lens[~big]
    assert small.min() >= 64 and small.max() <= 16384 and np.all(small % 64 == 0)
    assert _no_overlap(b.src_off, b.lens) and _no_overlap(b.dst_off, b.lens)
    assert b.src_off.max() + 16384 <= 2 << 30 and np.all(b.dst_off + b.lens <= 2 << 30)
    # seeded: the same seed gives the same layout
    b2 = workloads.batch_head_sliced()
    assert np.array_equal(b.dst_off, b2.dst_off) and np.array_equal(b.lens, b2.lens)


def test_random_batch_any_alignment():
    b = workloads.random_batch(3, 500, 3000, 1 << 22, align=1)
    assert _no_overlap(b.src_off, b.lens) and _no_overlap(b.dst_off, b.lens)
    assert len(set((b.src_off % 16).tolist())) > 8

"""libtb from C: tests/c_client.c, built with gcc against include/tb.h,
libtb.so and the CUDA runtime only (no Python, no PyTorch in the client),
runs a 3-source reduce-copy, a transfer on the copy engines (DMA executor)
and a batch of 1000 scattered copies through tb_batch_copy and through
tb_batch_copy_noalloc; every result must equal the oracle's."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_matches_the_oracle(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    from copy_reduce_dst_gb300 import _build
    lib = _build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_client")
    subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
                    f"-I{ROOT}/include", f"-I{cuda}/include", os.path.join(ROOT, "tests", "c_client.c"),
                    "-o", exe, f"-L{libdir}", "-ltb", f"-L{cuda}/lib64", "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cuda}/lib64"], check=True)
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"

    n = (16 << 20) // 4
    refs = [oracle.prepare_reference(n, k) for k in range(3)]
    got = np.fromfile(tmp_path / "reduce.bin", dtype=np.float32)
    assert oracle.first_mismatch(got.view(np.uint32), oracle.dst_reference(refs).view(np.uint32)) == -1
    got = np.fromfile(tmp_path / "dma.bin", dtype=np.float32)
    assert oracle.first_mismatch(got.view(np.uint32), refs[1].view(np.uint32)) == -1

    i = np.arange(1000, dtype=np.uint64)
    src_off = 16384 * i + i % 13
    dst_off = 16384 * ((i * 7919) % 1000) + i % 5
    lens = 64 + 13 * i
    pool = np.zeros(16384 * 1000 + 64, dtype=np.uint8)
    oracle.apply_batch(pool, refs[0].view(np.uint8), src_off, dst_off, lens)
    for name in ("batch.bin", "batch_noalloc.bin"):
        got = np.fromfile(tmp_path / name, dtype=np.uint8)
        assert oracle.first_mismatch(got, pool) == -1, name

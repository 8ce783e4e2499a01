"""bench.py on the GPU: one short run prints one JSON line carrying every key
of the bench contract and of the workloads it reports (the 3-source
reduce-copy, the 47,540 batch, the single 4 MiB transfer, the DMA executor,
the fillCompress rotation sweep, the 3840- and 7200-page batches, GEMM
interference, multi-source fillCompress and device validation), with values
in their plausible ranges."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from copy_reduce_dst_gb300 import _build
    _build.build()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5",
                        "--warmup", "3", "--cpu-seconds", "0.5"], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_contract_keys(line):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["n_gpus"] == 1
    assert line["steps"] == 5 and line["warmup"] == 3 and line["gpu_launches"] == 5
    assert "workload" in line["config"]
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert 0.5 < roof["frac"] < 1.3                      # a copy-bound kernel near its peak
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    assert cpu["batch"]["unit"] == "copies/s" and cpu["batch"]["value"] > 0
    par = cpu["parallel"]
    assert par["bit_exact_vs_oracle"] is True and par["value"] > 0 and par["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 3 * (256 << 20)
    assert e2e["d2h_bytes_per_step"] == 256 << 20 and 0 < e2e["value"] < line["value"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])


def test_workload_keys(line):
    b = line["batch"]
    assert b["descriptors"] == 47540 and b["speedup_vs_memcpy_each"] > 10
    assert b["roofline"]["kernel"].startswith("k_batch")
    s = line["single_4mib_k64"]
    assert s["K"] == 64 and s["alloc_bytes"] == 268435456 and s["prep_h2d_bytes"] == 4 << 20
    assert s["validated"] and s["dma_validated"] and s["gbps"] > 0 and s["dma_gbps"] > 0
    assert 0 < s["floor_us_per_iteration_4kib_64"] < 2 * s["us_per_iteration_64"]
    d = line["dma_executor_256mib"]
    assert d["kernel_gbps"] > 0 and d["dma_gbps"] > 0
    sweep = line["rotation_sweep"]
    assert [r["MiB"] for r in sweep] == [8, 16, 32, 64, 128, 256, 512]
    for r in sweep:
        assert r["on"]["K"] == max(1, 256 // r["MiB"]) and r["off"]["K"] == 1
    for key, n in (("index_pages_3840", 3840), ("block_pages_7200", 7200)):
        assert line[key]["descriptors"] == n and line[key]["bytes_touched_per_cycle"] > 256 << 20
    it = line["interference"]
    assert it["gemm_tflops_alone"] > 0 and it["batch_gbps"] > 0
    assert [r["sources"] for r in line["multi_source_fill_compress"]] == [2, 4, 8]
    assert all(r["K"] == 4 for r in line["multi_source_fill_compress"])
    v = line["validation_256mib"]
    assert 0 < v["device_ms"] < v["host_ms"]

"""The usage example in README.md runs as written on the GPU."""
import os

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from copy_reduce_dst_gb300 import _build
    _build.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    start = text.index("```python") + len("```python")
    code = text[start:text.index("```", start)]
    scope = {}
    exec(compile(code, "README.md", "exec"), scope)
    r, dst, src, nb = scope["r"], scope["dst"], scope["src"], scope["nb"]
    assert r["K"] == 64 and r["gbps"] > 0
    torch.cuda.synchronize()
    # dst holds the 4 MiB transfer except where the batch overwrote it
    assert torch.equal(dst[8192 * 100:], src[8192 * 100:nb])
    for i in (0, 57, 99):
        assert torch.equal(dst[8192 * i:8192 * i + 2112], src[4096 * i:4096 * i + 2112])

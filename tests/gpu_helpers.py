"""Helpers shared by the GPU parity tests: device buffers from torch, host
copies, and finite random float sources.  Torch only allocates memory and
moves bytes here; every computation under test runs in libtb's kernels."""
import numpy as np
import torch


def dev_bytes(nbytes: int, fill: int | None = None) -> torch.Tensor:
    t = torch.empty(max(1, nbytes), dtype=torch.uint8, device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).to("cuda")


def to_host(t: torch.Tensor, nbytes: int | None = None, offset: int = 0) -> np.ndarray:
    torch.cuda.synchronize()
    n = t.numel() - offset if nbytes is None else nbytes
    return t[offset:offset + n].cpu().numpy()


def finite_floats(g: np.random.Generator, n: int, max_exp: int = 200) -> np.ndarray:
    """Random float32 with biased exponent <= max_exp (no inf/NaN, sums of up
    to 16 of them stay finite), with subnormals and signed zeros mixed in."""
    bits = g.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    exp = (bits >> np.uint32(23)) & np.uint32(0xFF)
    exp = np.minimum(exp, np.uint32(max_exp))
    bits = (bits & np.uint32(0x807FFFFF)) | (exp << np.uint32(23))
    bits[::13] &= np.uint32(0x807FFFFF)      # subnormals
    bits[::17] = np.uint32(0x80000000)       # -0.0
    return bits.view(np.float32)

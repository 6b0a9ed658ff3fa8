"""Helpers shared by the GPU tests: moving numpy rank buffers (float32, or
uint16 bf16 patterns) to and from CUDA tensors, and bitwise comparison."""
import numpy as np
import torch


def to_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return torch.from_numpy(x.copy()).to(device)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).to(device).view(torch.bfloat16)
    return torch.from_numpy(x.copy()).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits(a: np.ndarray) -> np.ndarray:
    return a.view({8: np.uint64, 4: np.uint32, 2: np.uint16, 1: np.uint8}[a.itemsize])


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what=""):
    g, w = bits(np.ascontiguousarray(got)), bits(np.ascontiguousarray(want))
    assert g.shape == w.shape, (what, g.shape, w.shape)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        j = int(bad[0])
        raise AssertionError("%s: %d of %d differ, first at %d: got %r (0x%x) want %r (0x%x)" % (
            what, bad.size, g.size, j, got.flat[j], int(g[j]), want.flat[j], int(w[j])))

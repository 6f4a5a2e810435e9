"""Helpers for the GPU parity tests: device transfer, bitwise comparison."""
import numpy as np
import torch


def dev(x, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(x)) if not isinstance(x, torch.Tensor) else x
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def host(t):
    return t.detach().cpu().numpy()


def u32(a):
    return np.ascontiguousarray(a).view(np.uint32)


def assert_bits_equal(got, want, what="", nan_equal=False):
    """Bitwise equality of two float32 (or int) arrays, with a readable diff."""
    g = np.ascontiguousarray(got)
    w = np.ascontiguousarray(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    if g.dtype == np.float32:
        gb, wb = g.view(np.uint32), w.view(np.uint32)
        bad = gb != wb
        if nan_equal:
            bad &= ~(np.isnan(g) & np.isnan(w))
    else:
        bad = g != w
    if bad.any():
        idx = np.argwhere(bad)
        first = [tuple(int(v) for v in i) for i in idx[:8]]
        detail = [(i, g[i], w[i]) for i in first]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first {detail}")

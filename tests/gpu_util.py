"""Helpers shared by the GPU tests: byte-level comparison and the tolerance
checks.  Test infrastructure only."""
import numpy as np
import torch


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def same_bytes(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality of two tensors of the same dtype and shape."""
    assert a.shape == b.shape and a.dtype == b.dtype, (a.shape, b.shape, a.dtype, b.dtype)
    return bool(torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)))


def first_divergence(a: torch.Tensor, b: torch.Tensor):
    """Flat index of the first element whose bytes differ, or None."""
    ai = a.contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32).flatten()
    bi = b.contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32).flatten()
    idx = torch.nonzero(ai != bi)
    return None if idx.numel() == 0 else int(idx[0])


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 2.0 ** -134)


def check_close(g: np.ndarray, r: np.ndarray, bound: np.ndarray, what: str):
    """Assert |g - r| <= bound element-wise; report the worst element."""
    err = np.abs(g - r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d of %d elements out of bound; worst at %s: got %r want %r "
                             "(err %.3g, bound %.3g)" % (what, int(bad.sum()), err.size, i, g[i],
                                                        r[i], err[i], bound[i]))

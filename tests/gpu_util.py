"""Shared helpers of the GPU parity tests (imported by test modules only)."""
import numpy as np
import pytest

TOL = 1e-4  # |y - y_ref| <= TOL * sum_i |w_i * xhat_i| per output


def cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from verify_matvec_gb300 import build
    build.build()
    return torch


def assert_within_bound(y, y_ref, bound, tol=TOL, what="y"):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    lim = tol * bound
    bad = err > lim
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs outside tolerance; first at {tuple(i)}: "
                             f"got {y[tuple(i)]!r} want {y_ref[tuple(i)]!r} bound {lim[tuple(i)]!r}")
    zero = bound == 0
    assert np.all(y[zero] == 0), f"{what}: nonzero output where the bound is zero"


class Guarded:
    """A device output buffer with guard bands of canary bytes on both sides
    (a bounds check in place of a memory checker): `view` is the buffer the
    call writes; `check()` asserts that no byte outside it changed."""

    GUARD = 4096  # bytes on each side (a multiple of 256, so the view stays aligned)
    CANARY = 0xA5

    def __init__(self, torch, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((n + 2 * self.GUARD,), self.CANARY, dtype=torch.uint8, device="cuda")
        self.n = n
        self.view = self.raw[self.GUARD:self.GUARD + n].view(dtype).view(shape)

    def check(self):
        head = self.raw[:self.GUARD].cpu().numpy()
        tail = self.raw[self.GUARD + self.n:].cpu().numpy()
        assert np.all(head == self.CANARY), "bytes before the output buffer were written"
        assert np.all(tail == self.CANARY), "bytes after the output buffer were written"

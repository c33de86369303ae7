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

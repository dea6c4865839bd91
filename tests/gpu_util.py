"""Shared helpers of the GPU parity tests."""
import numpy as np

TOL_REL = 1e-3      # |y - y_ref| <= 1e-3 * sum_k |w * x| + 1e-6
TOL_ABS = 1e-6


def assert_close(name, y_gpu, y_ref, bound):
    y = np.asarray(y_gpu, dtype=np.float64)
    assert y.shape == y_ref.shape, (name, y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{name}: non-finite output"
    err = np.abs(y - y_ref)
    tol = TOL_REL * bound + TOL_ABS
    bad = np.nonzero(err > tol)
    if bad[0].size:
        i = tuple(b[0] for b in bad)
        raise AssertionError(f"{name}: {bad[0].size} outputs out of bound; first at {i}: "
                             f"gpu {y[i]!r} oracle {y_ref[i]!r} err {err[i]:.3e} tol {tol[i]:.3e}")


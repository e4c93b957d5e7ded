"""Helpers for the GPU parity tests: device copies of numpy arrays and the
tolerance the tests apply to floating-point results.

Tolerance (stated for the int4 GEMV/matmul and the f32 control): per element
    |y - y_oracle| <= 1e-3 * sum_k |w_nk * x_mk| + 1e-6
with the bound computed by the oracle in binary64.
"""
import numpy as np
import pytest

REL_TOL = 1e-3
ABS_TOL = 1e-6


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev(a, torch):
    """Copy a numpy array to the GPU (16-bit patterns as int16, same bytes)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t, dtype=None):
    a = t.cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def assert_within_bound(y, y_ref, bound, what=""):
    y = np.asarray(y, np.float64)
    err = np.abs(y - y_ref.astype(np.float64))
    lim = REL_TOL * bound + ABS_TOL
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                             f"1e-3*sum|wx|+1e-6; first {idx.tolist()}, "
                             f"err {err[bad][:5]}, limit {lim[bad][:5]}")
    return float(np.max(err / lim)) if err.size else 0.0

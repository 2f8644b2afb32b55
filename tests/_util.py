"""Helpers shared by the GPU parity tests."""
from __future__ import annotations

import numpy as np

# Bounds on |y - y_ref| relative to c = sum_k |w_k x_k| (fp64, from the
# oracle): the fp32 GEMV paths and the bf16 tensor-core prefill path.
TOL_FP32 = 1e-4
TOL_BF16 = 1e-2


def assert_close_to_oracle(y, y_ref, c, rel, what=""):
    """|y - y_ref| <= rel * c elementwise; where c == 0, y must be exactly 0."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    assert y.shape == y_ref.shape == c.shape, (y.shape, y_ref.shape, c.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    bad = err > rel * c
    if bad.any():
        idx = np.argwhere(bad)[0]
        i = tuple(idx)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs out of bound; first at {i}: "
            f"y={y[i]!r} y_ref={y_ref[i]!r} |err|={err[i]:.3e} bound={rel * c[i]:.3e}")


def to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)

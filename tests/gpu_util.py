"""Shared helpers of the GPU parity tests."""
import numpy as np

# The stack's tolerance against the float64 oracle: an element passes when
# |gpu - ref| <= ATOL + RTOL * |ref|  (2e-4 absolute and 1e-4 relative).
ATOL = 2e-4
RTOL = 1e-4


def assert_within(gpu, ref, atol=ATOL, rtol=RTOL, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside "
            f"{atol:g} + {rtol:g}*|ref|; worst at {idx}: gpu {gpu[idx]!r} ref {ref[idx]!r}; "
            f"max abs err {err.max():.3e}")
    return float(err.max())


def cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()

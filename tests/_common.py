"""Helpers shared by the GPU parity tests: building the library once, moving
synthetic inputs to the device, and the element-wise tolerance check."""
import numpy as np
import pytest
import torch

import __graft_entry__

# Tolerances of the pages' acceptance bar: |gpu - oracle| <= atol + rtol * |oracle|.
BF16_TOL = (2e-2, 1e-2)
F32_TOL = (1e-4, 1e-4)

_built = False


def need_gpu():
    global _built
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not _built:
        __graft_entry__.build()
        _built = True


def to_dev(obj):
    if isinstance(obj, torch.Tensor):
        return obj.cuda()
    if isinstance(obj, dict):
        return {k: to_dev(v) for k, v in obj.items()}
    if isinstance(obj, list):
        return [to_dev(v) for v in obj]
    return obj


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def assert_close(got, ref, tol, what=""):
    got = f64(got)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    atol, rtol = tol
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d/%d elements out of tolerance; worst at %s: got %r ref %r "
                             "(max abs err %.3g)" % (what, bad.sum(), bad.size, i, got[i], ref[i], err.max()))
    return float(err.max())


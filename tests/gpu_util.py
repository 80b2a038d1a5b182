"""Helpers for the GPU parity tests (host <-> device marshalling and the
elementwise bound)."""
import numpy as np
import pytest

import nf_inputs

# Elementwise bound of the fused kernels against the fp64 oracle:
# |gpu - ref| <= ATOL + RTOL * |ref|.  bf16 output rounding alone contributes
# up to 2^-9 relative (0.2%); the remainder covers fp32 accumulation order and
# rsqrtf.
ATOL = 2e-2
RTOL = 1.6e-2


def require_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device (run them with -m gpu on a GB300)")
    return torch.device("cuda:0")


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def to_f64(t):
    import torch
    return nf_inputs.bf16_to_f64(t.detach().view(torch.int16).cpu().numpy().view(np.uint16))


def assert_close(got, want, what, atol=ATOL, rtol=RTOL, extra=None):
    """|got - want| <= atol + rtol |want| (+ extra, an elementwise term that a
    test derives for operands the kernel rounds and the definition does not)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    if extra is not None:
        bound = bound + np.asarray(extra, dtype=np.float64)
    bad = err > bound
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} out of bound; first at {idx}: "
                             f"got {got[idx]!r} want {want[idx]!r}; max err {err.max():.3e}")
    return float(err.max())

"""Shared helpers for the GPU parity tests (comparison and tolerances)."""

import numpy as np
import torch

# Tolerances fixed by the workload statement: float32 paths max |err| <= 1e-5;
# bf16 in / f32 accumulate: O <= 2e-2, LSE <= 1e-3 (absolute).
TOL_F32 = 1e-5
TOL_BF16_O = 2e-2
TOL_BF16_LSE = 1e-3
# bf16 row softmax: y in [0, 1] rounded to bf16 (half an ulp of 1.0 is 2^-9)
TOL_BF16_SOFTMAX = 2.5e-3


def f64(t):
    """Exact float64 copy of a tensor (bf16 and f32 values are representable)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(got, want, tol, what=""):
    got, want = f64(got), np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    fin = np.isfinite(want)
    bad = np.isfinite(got) != fin
    assert not bad.any(), "%s: finiteness differs at %d places (first %s)" % (
        what, bad.sum(), np.argwhere(bad)[:3].tolist())
    assert np.array_equal(got[~fin], want[~fin]), "%s: infinities differ" % what
    if fin.any():
        err = np.abs(got[fin] - want[fin])
        i = int(np.argmax(err))
        assert err[i] <= tol, "%s: max |err| %.3g > %.3g (got %r want %r)" % (
            what, err[i], tol, got[fin][i], want[fin][i])


def bf16_tols(dtype):
    if dtype == torch.float32:
        return TOL_F32, TOL_F32
    return TOL_BF16_O, TOL_BF16_LSE

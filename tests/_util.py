"""Shared test helpers: the parity metric and tolerances."""

import json as _json
import os as _os

import numpy as np

# Per-tensor infinity-norm relative error, max_i |g_i - r_i| / max_i |r_i|.  The
# rustytorch backward_cuda commit gives a 1e-4 bound on the relative error
# between GPU and CPU gradients without defining the metric (stored, with its
# source, in golden/tolerance_backward_cuda.json); this is the reading taken.
# bf16 activations (with fp32 state and grads) get 2e-2.
with open(_os.path.join(_os.path.dirname(__file__), "golden", "tolerance_backward_cuda.json")) as _f:
    _PAGE = _json.load(_f)
TOL = {"f32": float(_PAGE["gpu_vs_cpu_gradient_tolerance"]), "bf16": 2e-2}


def max_rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    diff = float(np.max(np.abs(got - ref)))
    if scale == 0.0:
        return diff
    return diff / scale


def assert_close(got, ref, tol, name=""):
    e = max_rel_err(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite values"
    assert e <= tol, f"{name}: max rel err {e:.3e} > {tol:.1e}"
    return e

"""The seeded generators: determinism, dtype rounding and the stated distributions (CPU only)."""

import numpy as np
import pytest

from workloads import CONFIGS, make_conv_inputs, make_rmsnorm_inputs, make_scan_inputs
from workloads.synth import round_to


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(10000) * 10 ** rng.uniform(-3, 3, 10000),
                        # exact ties between two bf16 values (round to even)
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0])])
    v32 = v.astype(np.float32).astype(np.float64)
    ours = round_to(v32, "bf16")
    theirs = torch.tensor(v32, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, theirs)


def test_scan_inputs_deterministic_and_distributed():
    wl = CONFIGS["tiny"].with_(B=3, L=50, D=32)
    a = make_scan_inputs(wl, seed=0)
    b = make_scan_inputs(wl, seed=0)
    c = make_scan_inputs(wl, seed=1)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    assert not np.array_equal(a["x"], c["x"])
    assert a["delta"].min() > 0
    # softplus(0.5 eps + dt_bias) with dt_bias = softplus^-1(u), u in [1e-3, 1e-1]
    assert np.median(a["delta"]) < 0.2
    np.testing.assert_array_equal(a["A"], -np.arange(1, wl.N + 1)[None].repeat(wl.D, 0))
    np.testing.assert_array_equal(a["Dv"], 1.0)


def test_bf16_workload_values_on_grid():
    wl = CONFIGS["mamba1p4b"].with_(B=1, L=16, D=64)
    d = make_scan_inputs(wl)
    for k in ("x", "delta", "z", "Bm", "Cm", "dy"):
        np.testing.assert_array_equal(d[k], round_to(d[k], "bf16"))


def test_conv_and_rms_inputs():
    wl = CONFIGS["tiny"]
    cv = make_conv_inputs(wl)
    assert cv["w"].shape == (wl.D, wl.d_conv)
    assert np.all(np.abs(cv["w"]) <= 1 / np.sqrt(wl.d_conv))
    r = make_rmsnorm_inputs(wl, rows=7, dim=24)
    assert r["x"].shape == (7, 24) and r["rms"].shape == (7,)
    np.testing.assert_allclose(r["rms"], np.sqrt(np.mean(r["x"] ** 2, 1) + 1e-5), rtol=1e-7)

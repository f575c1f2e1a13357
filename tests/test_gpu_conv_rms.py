"""Conv1d-backward and RMSNorm-backward parity on the GPU against the float64 oracle."""

import numpy as np
import pytest

from oracle import conv1d_causal_bwd_ref, rmsnorm_bwd_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, ss_module
from workloads import CONFIGS, make_conv_inputs, make_rmsnorm_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


@pytest.mark.parametrize("B,L,D,K,dtype", [
    (2, 64, 16, 4, "f32"), (3, 130, 520, 4, "bf16"), (2, 65, 24, 3, "f32"), (1, 7, 8, 2, "bf16"),
    (2, 33, 16, 1, "f32"), (300, 40, 64, 4, "f32"),
])
def test_conv1d_bwd_parity(ss, B, L, D, K, dtype):
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, d_conv=K, dtype=dtype)
    c = make_conv_inputs(wl, seed=L + K)
    rng = np.random.default_rng(0)
    dw0 = rng.standard_normal((D, K)).astype(np.float32).astype(np.float64)
    db0 = rng.standard_normal(D).astype(np.float32).astype(np.float64)
    dx, dw, db = ss.conv1d_causal_bwd(dev(c["dout"]), dev(c["x"], dtype), dev(c["w"]), dw=dev(dw0), db=dev(db0))
    rdx, rdw, rdb = conv1d_causal_bwd_ref(c["dout"], c["x"], c["w"])
    tol = TOL["f32"]  # fp32 arithmetic on exactly representable inputs: fp32 tolerance for both dtypes
    assert_close(host(dx), rdx, tol, "dx")
    assert_close(host(dw) - dw0, rdw, tol, "dw")
    assert_close(host(db) - db0, rdb, tol, "db")


@pytest.mark.parametrize("R,H,dtype", [(37, 768, "f32"), (64, 2048, "bf16"), (5, 8, "f32"), (1500, 96, "bf16"),
                                       (20000, 32, "f32"), (333, 24, "bf16"), (100, 256, "f32"), (50, 264, "bf16"),
                                       (3, 12000, "f32"), (2, 32768, "bf16"), (41, 1536, "f32"), (700, 2040, "bf16"),
                                       (9, 4096, "bf16")])
def test_rmsnorm_bwd_parity(ss, R, H, dtype):
    wl = CONFIGS["tiny"].with_(dtype=dtype)
    r = make_rmsnorm_inputs(wl, seed=R, rows=R, dim=H)
    ds0 = np.random.default_rng(1).standard_normal(H).astype(np.float32).astype(np.float64)
    dx, dscale = ss.rmsnorm_bwd(dev(r["dy"], dtype), dev(r["x"], dtype), dev(r["scale"]), dev(r["rms"]), dscale=dev(ds0))
    rdx, rds = rmsnorm_bwd_ref(r["dy"], r["x"], r["scale"], r["rms"])
    tol = TOL["f32"]
    assert_close(host(dx), rdx, tol, "dx")
    assert_close(host(dscale) - ds0, rds, tol, "dscale")


def test_conv_rms_deterministic(ss):
    wl = CONFIGS["tiny"].with_(B=4, L=300, D=256, dtype="bf16")
    c = make_conv_inputs(wl)
    a = [host(t) for t in ss.conv1d_causal_bwd(dev(c["dout"]), dev(c["x"], "bf16"), dev(c["w"]))]
    b = [host(t) for t in ss.conv1d_causal_bwd(dev(c["dout"]), dev(c["x"], "bf16"), dev(c["w"]))]
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    r = make_rmsnorm_inputs(wl, rows=3000, dim=512)
    a = [host(t) for t in ss.rmsnorm_bwd(dev(r["dy"], "bf16"), dev(r["x"], "bf16"), dev(r["scale"]), dev(r["rms"]))]
    b = [host(t) for t in ss.rmsnorm_bwd(dev(r["dy"], "bf16"), dev(r["x"], "bf16"), dev(r["scale"]), dev(r["rms"]))]
    for u, v in zip(a, b):
        assert np.array_equal(u, v)

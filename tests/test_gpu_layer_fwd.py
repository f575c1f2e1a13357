"""Forward producers of the conv1d and RMSNorm backward inputs on the GPU
(conv1d_causal_fwd with and without SiLU, rmsnorm_fwd) against the float64
oracle, element by element.  Tolerance: per-tensor max |g-r| / max |r| <= 1e-4
for fp32 outputs, 2e-2 for bf16 outputs (one bf16 rounding of an fp32 result)."""

import numpy as np
import pytest

from oracle import conv1d_causal_fwd_ref, conv1d_causal_silu_fwd_ref, rmsnorm_fwd_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, ss_module
from workloads import CONFIGS, RMS_EPS, make_conv_inputs, make_rmsnorm_inputs, round_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


def _bias(D, seed):
    return round_to(0.5 * np.random.default_rng(seed).standard_normal(D), "f32")


@pytest.mark.parametrize("B,L,D,K,dtype,with_bias,silu", [
    (2, 64, 16, 4, "f32", True, False), (3, 130, 520, 4, "bf16", True, True), (2, 65, 24, 3, "f32", False, True),
    (1, 7, 8, 2, "bf16", True, True), (2, 33, 16, 1, "f32", True, False), (300, 40, 64, 4, "f32", False, True),
    (1, 1, 8, 4, "f32", True, True), (2, 97, 136, 3, "bf16", False, False), (1, 300, 8, 4, "bf16", True, True),
])
def test_conv1d_fwd_parity(ss, B, L, D, K, dtype, with_bias, silu):
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, d_conv=K, dtype=dtype)
    c = make_conv_inputs(wl, seed=3 * L + K)
    bias = _bias(D, L) if with_bias else None
    out = ss.conv1d_causal_fwd(dev(c["x"], dtype), dev(c["w"]), None if bias is None else dev(bias), silu=silu)
    assert out.dtype == dev(c["x"][:1, :1], dtype).dtype
    ref = (conv1d_causal_silu_fwd_ref if silu else conv1d_causal_fwd_ref)(c["x"], c["w"], bias)
    assert_close(host(out), ref, TOL[dtype], "out")


def test_conv1d_fwd_full_size_layer(ss):
    """The conv -> SiLU branch of the 1.4B-shaped layer: [4, 2048, 4096] bf16, d_conv 4, every element."""
    wl = CONFIGS["mamba1p4b"]
    c = make_conv_inputs(wl, seed=5)
    bias = _bias(wl.D, 5)
    out = ss.conv1d_causal_fwd(dev(c["x"], "bf16"), dev(c["w"]), dev(bias), silu=True)
    assert_close(host(out), conv1d_causal_silu_fwd_ref(c["x"], c["w"], bias), TOL["bf16"], "out")
    assert ss.device_status() == 0


@pytest.mark.parametrize("R,H,dtype", [(37, 768, "f32"), (64, 2048, "bf16"), (5, 8, "f32"), (1500, 96, "bf16"),
                                       (20000, 32, "f32"), (333, 24, "bf16"), (100, 256, "f32"), (50, 264, "bf16"),
                                       (3, 12000, "f32"), (2, 32768, "bf16"), (8192, 2048, "bf16"), (41, 1536, "f32"),
                                       (700, 2040, "bf16"), (9, 4096, "bf16")])
def test_rmsnorm_fwd_parity(ss, R, H, dtype):
    wl = CONFIGS["tiny"].with_(dtype=dtype)
    r = make_rmsnorm_inputs(wl, seed=R + 1, rows=R, dim=H)
    y, rms = ss.rmsnorm_fwd(dev(r["x"], dtype), dev(r["scale"]), RMS_EPS)
    ry, rrms = rmsnorm_fwd_ref(r["x"], r["scale"], RMS_EPS)
    assert_close(host(y), ry, TOL[dtype], "y")
    assert_close(host(rms), rrms, TOL["f32"], "rms")


def test_rmsnorm_fwd_feeds_bwd(ss):
    """rms from rmsnorm_fwd is the statistic rmsnorm_bwd expects: fwd -> bwd matches the oracle chain."""
    from oracle import rmsnorm_bwd_ref
    wl = CONFIGS["tiny"].with_(dtype="f32")
    r = make_rmsnorm_inputs(wl, seed=9, rows=300, dim=512)
    _, rms = ss.rmsnorm_fwd(dev(r["x"]), dev(r["scale"]), RMS_EPS)
    dx, dscale = ss.rmsnorm_bwd(dev(r["dy"]), dev(r["x"]), dev(r["scale"]), rms)
    _, rrms = rmsnorm_fwd_ref(r["x"], r["scale"], RMS_EPS)
    rdx, rds = rmsnorm_bwd_ref(r["dy"], r["x"], r["scale"], rrms)
    assert_close(host(dx), rdx, TOL["f32"], "dx")
    assert_close(host(dscale), rds, TOL["f32"], "dscale")


def test_layer_fwd_deterministic(ss):
    wl = CONFIGS["tiny"].with_(B=4, L=300, D=256, dtype="bf16")
    c = make_conv_inputs(wl)
    a = host(ss.conv1d_causal_fwd(dev(c["x"], "bf16"), dev(c["w"]), silu=True))
    b = host(ss.conv1d_causal_fwd(dev(c["x"], "bf16"), dev(c["w"]), silu=True))
    assert np.array_equal(a, b)
    r = make_rmsnorm_inputs(wl, rows=3000, dim=512)
    y1, s1 = ss.rmsnorm_fwd(dev(r["x"], "bf16"), dev(r["scale"]), RMS_EPS)
    y2, s2 = ss.rmsnorm_fwd(dev(r["x"], "bf16"), dev(r["scale"]), RMS_EPS)
    assert np.array_equal(host(y1), host(y2)) and np.array_equal(host(s1), host(s2))


@pytest.mark.parametrize("B,L,D,K,dtype,with_bias", [
    (2, 64, 16, 4, "f32", True), (3, 130, 520, 4, "bf16", True), (2, 65, 24, 3, "f32", False),
    (1, 7, 8, 2, "bf16", True), (2, 33, 16, 1, "f32", True), (300, 40, 64, 4, "f32", False), (1, 2, 8, 4, "f32", True),
])
def test_conv1d_silu_bwd_parity(ss, B, L, D, K, dtype, with_bias):
    from oracle import conv1d_causal_silu_bwd_ref
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, d_conv=K, dtype=dtype)
    c = make_conv_inputs(wl, seed=5 * L + K)
    bias = _bias(D, L + 1) if with_bias else None
    rng = np.random.default_rng(2)
    dw0 = round_to(rng.standard_normal((D, K)), "f32")
    db0 = round_to(rng.standard_normal(D), "f32")
    dx, dw, db = ss.conv1d_causal_silu_bwd(dev(c["dout"]), dev(c["x"], dtype), dev(c["w"]),
                                           None if bias is None else dev(bias), dw=dev(dw0), db=dev(db0))
    rdx, rdw, rdb = conv1d_causal_silu_bwd_ref(c["dout"], c["x"], c["w"], bias)
    tol = TOL["f32"]  # fp32 arithmetic on exactly representable inputs, fp32 outputs
    assert_close(host(dx), rdx, tol, "dx")
    assert_close(host(dw) - dw0, rdw, tol, "dw")
    assert_close(host(db) - db0, rdb, tol, "db")


def test_conv1d_silu_bwd_full_size_layer(ss):
    from oracle import conv1d_causal_silu_bwd_ref
    wl = CONFIGS["mamba1p4b"]
    c = make_conv_inputs(wl, seed=6)
    bias = _bias(wl.D, 6)
    dx, dw, db = ss.conv1d_causal_silu_bwd(dev(c["dout"]), dev(c["x"], "bf16"), dev(c["w"]), dev(bias))
    rdx, rdw, rdb = conv1d_causal_silu_bwd_ref(c["dout"], c["x"], c["w"], bias)
    assert_close(host(dx), rdx, TOL["f32"], "dx")
    assert_close(host(dw), rdw, TOL["f32"], "dw")
    assert_close(host(db), rdb, TOL["f32"], "db")

"""Conv1d and RMSNorm parity on seeded random shapes: every call next to the
scan (conv1d forward with and without SiLU, conv1d backward, SiLU-fused conv1d
backward, RMSNorm forward and backward) on shapes drawn with a fixed seed,
against the float64 oracle element by element.

The draws cover the dispatch boundaries of the RMSNorm kernels (rows of up to
256, 2048 and 8192 columns and wider) and the conv kernels' narrow rows (fewer
channel quads than a CTA's threads), sequences shorter than a tile and than the
filter, and every filter width."""

import numpy as np
import pytest

from oracle import (conv1d_causal_bwd_ref, conv1d_causal_fwd_ref, conv1d_causal_silu_bwd_ref,
                    conv1d_causal_silu_fwd_ref, rmsnorm_bwd_ref, rmsnorm_fwd_ref)
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, ss_module
from workloads import CONFIGS, RMS_EPS, make_conv_inputs, make_rmsnorm_inputs, round_to

pytestmark = pytest.mark.gpu


def _conv_cases(n=24, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B, L, D, K = int(rng.integers(1, 40)), int(rng.integers(1, 300)), 8 * int(rng.integers(1, 160)), int(rng.integers(1, 5))
        if B * L * D > 3_000_000:
            continue
        out.append((B, L, D, K, str(rng.choice(["f32", "bf16"])), bool(rng.random() < 0.6), int(rng.integers(1 << 30))))
    return out


def _rms_cases(n=24, seed=11):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        H = 8 * int(rng.choice([rng.integers(1, 33), rng.integers(33, 257), rng.integers(257, 1025), rng.integers(1025, 4097)]))
        R = int(rng.integers(1, max(2, 4_000_000 // H)))
        out.append((R, H, str(rng.choice(["f32", "bf16"])), int(rng.integers(1 << 30))))
    return out


@pytest.fixture(scope="module")
def ss():
    return ss_module()


@pytest.mark.parametrize("B,L,D,K,dtype,with_bias,seed", _conv_cases())
def test_conv1d_random_shape(ss, B, L, D, K, dtype, with_bias, seed):
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, d_conv=K, dtype=dtype)
    c = make_conv_inputs(wl, seed=seed % 100000)
    rng = np.random.default_rng(seed)
    bias = round_to(0.5 * rng.standard_normal(D), "f32") if with_bias else None
    bias_d = None if bias is None else dev(bias)
    x, w, dout = dev(c["x"], dtype), dev(c["w"]), dev(c["dout"])
    for silu in (False, True):
        out = ss.conv1d_causal_fwd(x, w, bias_d, silu=silu)
        ref = (conv1d_causal_silu_fwd_ref if silu else conv1d_causal_fwd_ref)(c["x"], c["w"], bias)
        assert_close(host(out), ref, TOL[dtype], f"out silu={silu}")
    dw0, db0 = round_to(rng.standard_normal((D, K)), "f32"), round_to(rng.standard_normal(D), "f32")
    tol = TOL["f32"]  # fp32 arithmetic on exactly representable inputs, fp32 outputs
    dx, dw, db = ss.conv1d_causal_bwd(dout, x, w, dw=dev(dw0), db=dev(db0))
    rdx, rdw, rdb = conv1d_causal_bwd_ref(c["dout"], c["x"], c["w"])
    assert_close(host(dx), rdx, tol, "dx")
    assert_close(host(dw) - dw0, rdw, tol, "dw")
    assert_close(host(db) - db0, rdb, tol, "db")
    dx, dw, db = ss.conv1d_causal_silu_bwd(dout, x, w, bias_d, dw=dev(dw0), db=dev(db0))
    rdx, rdw, rdb = conv1d_causal_silu_bwd_ref(c["dout"], c["x"], c["w"], bias)
    assert_close(host(dx), rdx, tol, "silu dx")
    assert_close(host(dw) - dw0, rdw, tol, "silu dw")
    assert_close(host(db) - db0, rdb, tol, "silu db")
    assert ss.device_status() == 0


@pytest.mark.parametrize("R,H,dtype,seed", _rms_cases())
def test_rmsnorm_random_shape(ss, R, H, dtype, seed):
    wl = CONFIGS["tiny"].with_(dtype=dtype)
    r = make_rmsnorm_inputs(wl, seed=seed % 100000, rows=R, dim=H)
    y, rms = ss.rmsnorm_fwd(dev(r["x"], dtype), dev(r["scale"]), RMS_EPS)
    ry, rrms = rmsnorm_fwd_ref(r["x"], r["scale"], RMS_EPS)
    assert_close(host(y), ry, TOL[dtype], "y")
    assert_close(host(rms), rrms, TOL["f32"], "rms")
    ds0 = round_to(np.random.default_rng(seed).standard_normal(H), "f32")
    dx, dscale = ss.rmsnorm_bwd(dev(r["dy"], dtype), dev(r["x"], dtype), dev(r["scale"]), dev(r["rms"]), dscale=dev(ds0))
    rdx, rds = rmsnorm_bwd_ref(r["dy"], r["x"], r["scale"], r["rms"])
    assert_close(host(dx), rdx, TOL["f32"], "dx")
    assert_close(host(dscale) - ds0, rds, TOL["f32"], "dscale")
    assert ss.device_status() == 0

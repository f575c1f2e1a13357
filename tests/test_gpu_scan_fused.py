"""The scan with the discretisation of delta fused in (delta = softplus(raw +
dt_bias), or raw + dt_bias) on the GPU against the float64 oracle: forward
outputs and every gradient, including the raw-delta and dt_bias gradients.
Tolerance: 1e-4 (fp32 activations) / 2e-2 (bf16 activations, fp32 state)."""

import numpy as np
import pytest

from oracle import scan_bwd_fused_ref, scan_fwd_fused_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, ss_module
from workloads import CONFIGS, make_scan_inputs, round_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


CASES = [
    # B, L, D, N, dtype, chunk, with dt_bias, softplus
    (2, 100, 40, 16, "f32", 8, True, True),
    (3, 77, 64, 8, "bf16", 32, True, True),
    (1, 300, 136, 16, "bf16", 8, True, False),
    (2, 130, 64, 16, "f32", 256, False, True),
    (1, 1000, 64, 16, "bf16", 8, True, True),  # segments
    (2, 5, 8, 4, "f32", 8, True, True),
    (4, 96, 128, 16, "bf16", 16, True, True),
]


@pytest.mark.parametrize("B,L,D,N,dtype,chunk,with_bias,softplus", CASES)
def test_fused_scan_parity(ss, B, L, D, N, dtype, chunk, with_bias, softplus):
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, N=N, dtype=dtype, chunk=chunk)
    inp = make_scan_inputs(wl, seed=B * 100 + L)
    bias = inp["dt_bias"] if with_bias else None
    if not softplus:  # delta = raw + dt_bias must stay positive: raw = the positive delta, a small positive bias
        inp["delta_raw"] = inp["delta"]
        if with_bias:
            bias = round_to(0.01 * np.abs(np.random.default_rng(L).standard_normal(D)), "f32")
    act = lambda k: dev(inp[k], dtype)
    x, raw, z, Bm, Cm, dy = act("x"), act("delta_raw"), act("z"), act("Bm"), act("Cm"), act("dy")
    A, Dv = dev(inp["A"]), dev(inp["Dv"])
    bias_d = None if bias is None else dev(bias)
    y, ckpt, h_last = ss.ss_scan_fwd(x, raw, A, Bm, Cm, Dv, z, chunk=chunk, dt_bias=bias_d, delta_softplus=softplus)
    g = ss.ss_scan_bwd(x, raw, A, Bm, Cm, Dv, z, ckpt, dy, chunk=chunk, dt_bias=bias_d, delta_softplus=softplus)
    a = (inp["x"], inp["delta_raw"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
    ry, rh, rck = scan_fwd_fused_ref(*a, dt_bias=bias, softplus=softplus, chunk=chunk)
    rg = scan_bwd_fused_ref(*a, inp["dy"], dt_bias=bias, softplus=softplus)
    tol = TOL[dtype]
    assert_close(host(y), ry, tol, "y")
    assert_close(host(ckpt), rck, tol, "ckpt")
    assert_close(host(h_last), rh, tol, "h_last")
    for k in ("dx", "ddelta", "dz", "dB", "dC", "dA", "dD", "dh0", "d_dt_bias"):
        assert_close(host(g[k]), rg[k], tol, k)
    assert ss.device_status() == 0


def test_fused_scan_full_size_layer_sampled(ss):
    """The 1.4B-shaped layer with the fused discretisation, in the bench's launch configuration: the
    per-channel sums over the full sequence (d_dt_bias, dD, dA) and a sampled set of (b, d) channels of
    y and ddelta against the oracle run on those channels alone."""
    wl = CONFIGS["mamba1p4b"]
    inp = make_scan_inputs(wl, seed=2)
    act = lambda k: dev(inp[k], "bf16")
    x, raw, z, Bm, Cm, dy = act("x"), act("delta_raw"), act("z"), act("Bm"), act("Cm"), act("dy")
    A, Dv, bias = dev(inp["A"]), dev(inp["Dv"]), dev(inp["dt_bias"])
    y, ckpt, _ = ss.ss_scan_fwd(x, raw, A, Bm, Cm, Dv, z, chunk=wl.chunk, dt_bias=bias, delta_softplus=True)
    g = ss.ss_scan_bwd(x, raw, A, Bm, Cm, Dv, z, ckpt, dy, chunk=wl.chunk, dt_bias=bias, delta_softplus=True)
    rng = np.random.default_rng(0)
    chans = np.sort(rng.choice(wl.D, size=48, replace=False))
    sl = lambda k: inp[k][:, :, chans]
    a = (sl("x"), sl("delta_raw"), inp["A"][chans], inp["Bm"], inp["Cm"], inp["Dv"][chans], sl("z"))
    ry, _, _ = scan_fwd_fused_ref(*a, dt_bias=inp["dt_bias"][chans], softplus=True)
    rg = scan_bwd_fused_ref(*a, sl("dy"), dt_bias=inp["dt_bias"][chans], softplus=True)
    tol = TOL["bf16"]
    assert_close(host(y)[:, :, chans], ry, tol, "y")
    for k in ("ddelta", "dx", "dz"):
        assert_close(host(g[k])[:, :, chans], rg[k], tol, k)
    for k in ("d_dt_bias", "dD"):
        assert_close(host(g[k])[chans], rg[k], tol, k)
    assert_close(host(g["dA"])[chans], rg["dA"], tol, "dA")

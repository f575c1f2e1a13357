"""Parity at the full workload sizes, in the launch configuration bench.py times.

The CUDA path runs on the whole workload; the float64 oracle is evaluated on
samples it can afford: every per-channel output (y, checkpoints, h_last, dx,
ddelta, dz, dA, dD, dh0) on a set of channels spread over the 64-channel tiles
(channels are independent given B_t, C_t), and the channel sums dB, dC on
whole batch rows (every row of the Mamba layers).  The conv1d backward is
sampled the same way; the RMSNorm backward is compared in full."""

import numpy as np
import pytest

from oracle import conv1d_causal_bwd_ref, rmsnorm_bwd_ref, scan_bwd_ref, scan_fwd_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, run_gpu_scan, scan_inputs_on_device, ss_module
from workloads import get_config, make_conv_inputs, make_rmsnorm_inputs, make_scan_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


def _channels(D, rng, n_rand=8):
    fixed = [0, 1, 62, 63, 64, 65, D // 2, D // 2 + 1, D - 2, D - 1]
    return np.array(sorted({c for c in fixed + list(rng.choice(D, n_rand, replace=False)) if 0 <= c < D}))


@pytest.mark.parametrize("name", ["mamba130m", "mamba1p4b", "short", "long"])
def test_scan_fullsize_sampled(ss, name):
    wl = get_config(name)
    tol = TOL[wl.dtype]
    inp = make_scan_inputs(wl, seed=0)
    d = scan_inputs_on_device(inp, wl.dtype)
    y, ckpt, h_last, g = run_gpu_scan(ss, d, wl.chunk)
    assert ss.device_status() == 0
    rng = np.random.default_rng(0)
    ch = _channels(wl.D, rng)
    bsel = np.arange(wl.B) if wl.B <= 16 else np.sort(rng.choice(wl.B, 16, replace=False))
    pick = lambda a: a[bsel][:, :, ch]
    args = (pick(inp["x"]), pick(inp["delta"]), inp["A"][ch], inp["Bm"][bsel], inp["Cm"][bsel], inp["Dv"][ch],
            pick(inp["z"]))
    yr, hr, cr = scan_fwd_ref(*args, chunk=wl.chunk)
    gr = scan_bwd_ref(*args, pick(inp["dy"]))
    gsel = lambda t: host(t)[bsel][:, :, ch]
    assert_close(gsel(y), yr, tol, "y")
    assert_close(host(ckpt)[bsel][:, :, ch], cr, tol, "ckpt")
    assert_close(host(h_last)[bsel][:, ch], hr, tol, "h_last")
    for k in ("dx", "ddelta", "dz"):
        assert_close(gsel(g[k]), gr[k], tol, k)
    assert_close(host(g["dh0"])[bsel][:, ch], gr["dh0"], tol, "dh0")
    if wl.B <= 16:  # dA, dD sum over every batch row
        assert_close(host(g["dA"])[ch], gr["dA"], tol, "dA")
        assert_close(host(g["dD"])[ch], gr["dD"], tol, "dD")
    # channel sums on whole batch rows: every row of the Mamba layers, 64 rows of the many-batch workload
    rows = list(range(min(wl.B, 64)))
    rows = np.array(rows)
    full = (inp["x"][rows], inp["delta"][rows], inp["A"], inp["Bm"][rows], inp["Cm"][rows], inp["Dv"], inp["z"][rows])
    gf = scan_bwd_ref(*full, inp["dy"][rows])
    assert_close(host(g["dB"])[rows], gf["dB"], tol, "dB")
    assert_close(host(g["dC"])[rows], gf["dC"], tol, "dC")
    if wl.B > 16:  # short many-batch workload: dA, dD over all rows is affordable at D=64
        gall = scan_bwd_ref(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"], inp["dy"])
        assert_close(host(g["dA"]), gall["dA"], tol, "dA")
        assert_close(host(g["dD"]), gall["dD"], tol, "dD")


@pytest.mark.parametrize("name", ["mamba130m", "mamba1p4b"])
def test_conv_rms_fullsize(ss, name):
    wl = get_config(name)
    tol = TOL["f32"]
    c = make_conv_inputs(wl)
    dx, dw, db = ss.conv1d_causal_bwd(dev(c["dout"]), dev(c["x"], wl.dtype), dev(c["w"]))
    ch = _channels(wl.D, np.random.default_rng(1))
    rdx, rdw, rdb = conv1d_causal_bwd_ref(c["dout"][:, :, ch], c["x"][:, :, ch], c["w"][ch])
    assert_close(host(dx)[:, :, ch], rdx, tol, "conv dx")
    assert_close(host(dw)[ch], rdw, tol, "conv dw")
    assert_close(host(db)[ch], rdb, tol, "conv db")
    r = make_rmsnorm_inputs(wl)
    rdx_, rds_ = ss.rmsnorm_bwd(dev(r["dy"], wl.dtype), dev(r["x"], wl.dtype), dev(r["scale"]), dev(r["rms"]))
    odx, ods = rmsnorm_bwd_ref(r["dy"], r["x"], r["scale"], r["rms"])
    assert_close(host(rdx_), odx, tol, "rms dx")
    assert_close(host(rds_), ods, tol, "rms dscale")

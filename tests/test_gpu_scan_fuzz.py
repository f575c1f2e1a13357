"""Selective-scan parity on seeded random shapes: batch rows, sequence length,
channels, N, chunk, dtype, the fused discretisation of delta and h0 / dh_last
drawn at random (a fixed seed, so the case list is the same on every run), the
CUDA path through the C ABI against the float64 oracle element by element.

The draws reach the launch shapes the hand-picked cases of test_gpu_scan.py may
miss: ragged channel tiles of every N, many batch rows on few channels (more
(row, tile) pairs than resident CTAs, uneven rows per CTA), few rows on long
sequences (segments, with and without the recompute pass), L = 1 and short
sequences under long chunks."""

import numpy as np
import pytest

from oracle import scan_bwd_fused_ref, scan_bwd_ref, scan_fwd_fused_ref, scan_fwd_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, scan_inputs_on_device, ss_module
from workloads import CONFIGS, make_scan_inputs

pytestmark = pytest.mark.gpu

MAX_CELLS = 6_000_000  # B * L * D * N per case: the oracle finishes each in about a second


def _draw_cases(n=64, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        N = int(rng.choice([4, 8, 16]))
        dtype = str(rng.choice(["f32", "bf16"]))
        chunk = int(rng.choice([8, 16, 32, 48, 64, 128, 256]))
        kind = rng.random()
        if kind < 0.25:    # many batch rows, few channels, short sequences
            B, L, D = int(rng.integers(200, 1300)), int(rng.integers(1, 25)), 8 * int(rng.integers(1, 5))
        elif kind < 0.5:   # few rows, long sequences: segments
            B, L, D = int(rng.integers(1, 3)), int(rng.integers(300, 1500)), 8 * int(rng.integers(2, 24))
        else:
            B, L, D = int(rng.integers(1, 9)), int(rng.integers(1, 400)), 8 * int(rng.integers(1, 41))
        if B * L * D * N > MAX_CELLS:
            continue
        fused = bool(rng.random() < 0.4)
        with_state = bool(rng.random() < 0.5)
        cases.append((B, L, D, N, dtype, chunk, fused, with_state, int(rng.integers(1 << 30))))
    return cases


CASES = _draw_cases()


@pytest.fixture(scope="module")
def ss():
    return ss_module()


@pytest.mark.parametrize("B,L,D,N,dtype,chunk,fused,with_state,seed", CASES)
def test_scan_parity_random_shape(ss, B, L, D, N, dtype, chunk, fused, with_state, seed):
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, N=N, dtype=dtype, chunk=chunk)
    inp = make_scan_inputs(wl, seed=seed % 100000)
    d = scan_inputs_on_device(inp, dtype)
    rng = np.random.default_rng(seed)
    h0 = dhl = None
    if with_state:  # values on the fp32 grid, as the kernels read them
        h0 = rng.standard_normal((B, D, N)).astype(np.float32).astype(np.float64)
        dhl = rng.standard_normal((B, D, N)).astype(np.float32).astype(np.float64)
    kw = {}
    if (L * N * (2 if dtype == "bf16" else 4)) % 16 != 0:
        # B_t / C_t rows of one batch row must span whole 16-byte units (bf16 with N = 4 and L odd): the call
        # refuses the layout before any launch, as the header states
        from mamba_selective_ssm_gb300._capi import SS_ERR_ALIGN, SSError
        with pytest.raises(SSError) as e:
            ss.ss_scan_fwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"], chunk=chunk)
        assert e.value.code == SS_ERR_ALIGN
        return
    if fused:
        d["delta"] = dev(inp["delta_raw"], dtype)
        kw = dict(dt_bias=dev(inp["dt_bias"]), delta_softplus=True)
    y, ckpt, h_last = ss.ss_scan_fwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"],
                                     h0=None if h0 is None else dev(h0), chunk=chunk, **kw)
    g = ss.ss_scan_bwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"], ckpt, d["dy"],
                       dh_last=None if dhl is None else dev(dhl), chunk=chunk, **kw)
    if fused:
        a = (inp["x"], inp["delta_raw"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
        ry, rh, rck = scan_fwd_fused_ref(*a, dt_bias=inp["dt_bias"], softplus=True, h0=h0, chunk=chunk)
        rg = scan_bwd_fused_ref(*a, inp["dy"], dt_bias=inp["dt_bias"], softplus=True, h0=h0, dh_last=dhl)
    else:
        a = (inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
        ry, rh, rck = scan_fwd_ref(*a, h0=h0, chunk=chunk)
        rg = scan_bwd_ref(*a, inp["dy"], h0=h0, dh_last=dhl)
    tol = TOL[dtype]
    assert_close(host(y), ry, tol, "y")
    assert_close(host(ckpt), rck, tol, "ckpt")
    assert_close(host(h_last), rh, tol, "h_last")
    names = ("dx", "ddelta", "dz", "dB", "dC", "dA", "dD", "dh0") + (("d_dt_bias",) if fused else ())
    for k in names:
        assert_close(host(g[k]), rg[k], tol, k)
    assert ss.device_status() == 0

"""Selective-scan parity on the GPU: the CUDA path through the C ABI against the
float64 oracle on the same seeded inputs, element by element.

Sizes span several 16-step tiles and 64-channel tiles with ragged tails in
both, every supported N, both dtypes, h0 / dh_last, L=1, and accumulation
into existing dA / dD.  Tolerance: per-tensor max |g-r| / max |r| <= 1e-4
(fp32 activations) or 2e-2 (bf16 activations, fp32 state and grads)."""

import numpy as np
import pytest

from oracle import scan_bwd_ref, scan_fwd_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, run_gpu_scan, scan_inputs_on_device, ss_module
from workloads import CONFIGS, make_scan_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


CASES = [
    # B, L, D, N, dtype, chunk
    (2, 64, 16, 4, "f32", 64),      # the tiny workload
    (3, 203, 40, 16, "f32", 32),    # ragged L and D, several chunks
    (2, 100, 72, 8, "bf16", 48),
    (1, 300, 136, 16, "bf16", 64),
    (5, 17, 24, 4, "f32", 16),
    (2, 1, 8, 16, "f32", 16),       # L = 1
    (2, 130, 64, 16, "f32", 256),   # chunk longer than the sequence
    (4, 96, 128, 16, "bf16", 32),
    # chunk = 8: a checkpoint per 8-step window, no recompute pass in the backward
    (2, 100, 40, 16, "f32", 8),
    (3, 77, 64, 8, "bf16", 8),
    (1, 300, 136, 16, "bf16", 8),
    (2, 5, 8, 4, "f32", 8),
    # few (batch row, channel tile) pairs: the sequence is cut into segments whose
    # carries are composed from per-segment summaries; ragged last segments
    (1, 1000, 64, 16, "bf16", 8),
    (1, 700, 200, 16, "bf16", 128),  # 64-channel backward CTAs (recompute pass, chunk >= 128)
    (2, 600, 72, 8, "f32", 256),
]


def _oracle(inp, chunk, h0=None, dh_last=None):
    a = (inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])
    y, h_last, ckpt = scan_fwd_ref(*a, h0=h0, chunk=chunk)
    g = scan_bwd_ref(*a, inp["dy"], h0=h0, dh_last=dh_last)
    return y, h_last, ckpt, g


def _check_all(res, ref, tol, with_h0=True):
    y, ckpt, h_last, g = res
    yr, hr, cr, gr = ref
    assert_close(host(y), yr, tol, "y")
    assert_close(host(ckpt), cr, tol, "ckpt")
    assert_close(host(h_last), hr, tol, "h_last")
    for k in ("dx", "ddelta", "dz", "dB", "dC", "dA", "dD") + (("dh0",) if with_h0 else ()):
        assert_close(host(g[k]), gr[k], tol, k)


@pytest.mark.parametrize("B,L,D,N,dtype,chunk", CASES)
def test_scan_parity(ss, B, L, D, N, dtype, chunk):
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, N=N, dtype=dtype, chunk=chunk)
    inp = make_scan_inputs(wl, seed=B * 1000 + L)
    d = scan_inputs_on_device(inp, dtype)
    res = run_gpu_scan(ss, d, chunk)
    _check_all(res, _oracle(inp, chunk), TOL[dtype])
    assert ss.device_status() == 0


@pytest.mark.parametrize("dtype,chunk", [("f32", 32), ("bf16", 32), ("f32", 8)])
def test_scan_h0_dh_last_and_accumulation(ss, dtype, chunk):
    B, L, D, N = 2, 77, 48, 16
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, N=N, dtype=dtype, chunk=chunk)
    inp = make_scan_inputs(wl, seed=7)
    rng = np.random.default_rng(3)
    h0 = rng.standard_normal((B, D, N)).astype(np.float32).astype(np.float64)
    dhl = rng.standard_normal((B, D, N)).astype(np.float32).astype(np.float64)
    dA0 = rng.standard_normal((D, N)).astype(np.float32).astype(np.float64)
    dD0 = rng.standard_normal(D).astype(np.float32).astype(np.float64)
    d = scan_inputs_on_device(inp, dtype)
    res = run_gpu_scan(ss, d, chunk, h0=dev(h0), dh_last=dev(dhl), dA0=dev(dA0), dD0=dev(dD0))
    y, h_last, ckpt, g = _oracle(inp, chunk, h0=h0, dh_last=dhl)
    g = dict(g)
    tol = TOL[dtype]
    # dA, dD accumulate into what was there; compare the increments
    assert_close(host(res[3]["dA"]) - dA0, g["dA"], tol, "dA increment")
    assert_close(host(res[3]["dD"]) - dD0, g["dD"], tol, "dD increment")
    g["dA"] = g["dA"] + dA0
    g["dD"] = g["dD"] + dD0
    _check_all(res, (y, h_last, ckpt, g), tol)


def test_scan_rows_beyond_the_first_batch_row_use_their_own_state(ss):
    """Each CTA walks several batch rows: the short many-batch shape with more (row, channel tile) pairs than
    resident CTAs in both directions, B odd so that some CTAs get one row fewer than others."""
    B, L, D, N, chunk = 3001, 16, 8, 16, 16
    wl = CONFIGS["short"].with_(B=B, L=L, D=D, N=N, chunk=chunk)
    inp = make_scan_inputs(wl, seed=11)
    d = scan_inputs_on_device(inp, "f32")
    res = run_gpu_scan(ss, d, chunk)
    _check_all(res, _oracle(inp, chunk), TOL["f32"])


def test_scan_deterministic(ss):
    wl = CONFIGS["tiny"].with_(B=3, L=150, D=80, N=16, dtype="bf16", chunk=32)
    inp = make_scan_inputs(wl, seed=5)
    d = scan_inputs_on_device(inp, "bf16")
    r1 = run_gpu_scan(ss, d, 32)
    r2 = run_gpu_scan(ss, d, 32)
    assert np.array_equal(host(r1[0]), host(r2[0]))
    for k in ("dx", "ddelta", "dz", "dB", "dC", "dA", "dD", "dh0"):
        assert np.array_equal(host(r1[3][k]), host(r2[3][k])), k


def test_scan_segment_chaining_on_gpu(ss):
    """fwd(L1) -> h_last -> fwd(L2, h0) equals fwd(L1+L2); the backward chains through dh0 -> dh_last."""
    import torch
    wl = CONFIGS["tiny"].with_(B=2, L=96, D=32, N=8, chunk=32)
    inp = make_scan_inputs(wl, seed=9)
    d = scan_inputs_on_device(inp, "f32")
    full = run_gpu_scan(ss, d, 32)
    cut = 48
    seq = ("x", "delta", "z", "Bm", "Cm", "dy")
    a = {k: (v[:, :cut].contiguous() if k in seq else v) for k, v in d.items()}
    b = {k: (v[:, cut:].contiguous() if k in seq else v) for k, v in d.items()}
    ya, _, ha, _ = run_gpu_scan(ss, a, 32)
    yb, _, hb, gb = run_gpu_scan(ss, b, 32, h0=ha)
    _, _, _, ga = run_gpu_scan(ss, a, 32, dh_last=gb["dh0"])
    tol = 1e-5
    assert_close(host(torch.cat([ya, yb], 1)), host(full[0]), tol, "y")
    assert_close(host(hb), host(full[2]), tol, "h_last")
    for k in ("dx", "ddelta", "dz", "dB", "dC"):
        assert_close(host(torch.cat([ga[k], gb[k]], 1)), host(full[3][k]), tol, k)
    assert_close(host(ga["dA"] + gb["dA"]), host(full[3]["dA"]), tol, "dA")
    assert_close(host(ga["dh0"]), host(full[3]["dh0"]), tol, "dh0")


def test_scan_rejects_misaligned_and_strided(ss):
    import torch
    from mamba_selective_ssm_gb300 import SSError
    wl = CONFIGS["tiny"]
    d = scan_inputs_on_device(make_scan_inputs(wl), "f32")
    with pytest.raises(ValueError):
        ss.ss_scan_fwd(d["x"].transpose(1, 2), d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"])
    big = torch.zeros(d["x"].numel() + 1, device="cuda")
    x_off = big[1:].view_as(d["x"])  # contiguous but 4 bytes off a 16-byte boundary
    with pytest.raises(SSError) as e:
        ss.ss_scan_fwd(x_off, d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"], chunk=64)
    assert e.value.code == -4


@pytest.mark.parametrize("case", ["A_zero", "fast_decay", "saturated_gate", "zero_input"])
def test_scan_degenerate_inputs(ss, case):
    """Limits the recurrence meets in practice: no decay (a = 1: running sums), a strong decay (a down to
    e^-100), a saturated gate (|z| large), and x = 0 (the state only decays).  The GPU path matches the oracle
    and stays finite."""
    wl = CONFIGS["tiny"].with_(B=2, L=150, D=40, N=16, dtype="f32", chunk=8)
    inp = make_scan_inputs(wl, seed=13)
    if case == "A_zero":
        inp["A"] = np.zeros_like(inp["A"])
    elif case == "fast_decay":
        inp["A"] = inp["A"] * 20.0  # delta*A down to about -100 per step: the state forgets within a few steps
    elif case == "saturated_gate":
        inp["z"] = np.where(inp["z"] > 0, 60.0, -60.0)
    else:
        inp["x"] = np.zeros_like(inp["x"])
    d = scan_inputs_on_device(inp, "f32")
    res = run_gpu_scan(ss, d, 8)
    _check_all(res, _oracle(inp, 8), TOL["f32"])
    assert ss.device_status() == 0


def test_scan_many_segments_long_row(ss):
    """One batch row of 4096 steps over 32 channels: the sequence is cut into the maximum number of
    segments (64), each composing its carry from all summaries before / after it."""
    wl = CONFIGS["long"].with_(B=1, L=4096, D=32, N=16, dtype="bf16", chunk=8)
    inp = make_scan_inputs(wl, seed=17)
    d = scan_inputs_on_device(inp, "bf16")
    res = run_gpu_scan(ss, d, 8)
    _check_all(res, _oracle(inp, 8), TOL["bf16"])

"""Single-token decode steps on the GPU (ss_scan_step, conv1d_causal_step)
against the float64 oracle, and chained over L steps against the sequence
kernels.  Tolerance: 1e-4 (fp32 activations) / 2e-2 (bf16 activations);
state comparisons in fp32 at 1e-4."""

import numpy as np
import pytest

from oracle import conv1d_causal_fwd_ref, conv1d_step_fwd_ref, scan_step_ref
from tests._util import TOL, assert_close
from tests.gpu_util import dev, host, ss_module
from workloads import CONFIGS, make_conv_inputs, make_scan_inputs, round_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    return ss_module()


def _step_inputs(B, D, N, dtype, seed):
    wl = CONFIGS["tiny"].with_(B=B, L=1, D=D, N=N, dtype=dtype)
    inp = make_scan_inputs(wl, seed=seed)
    h = round_to(np.random.default_rng(seed).standard_normal((B, D, N)), "f32")
    return {k: (v[:, 0] if v.ndim == 3 and k not in ("A",) else v) for k, v in inp.items()}, h


@pytest.mark.parametrize("B,D,N,dtype", [(3, 40, 16, "f32"), (5, 72, 8, "bf16"), (2, 8, 4, "f32"), (1, 8, 16, "f32"),
                                         (64, 4096, 16, "bf16"), (7, 24, 16, "bf16")])
def test_scan_step_parity(ss, B, D, N, dtype):
    p, h0 = _step_inputs(B, D, N, dtype, seed=B * 7 + D)
    h = dev(h0)
    y = ss.ss_scan_step(dev(p["x"], dtype), dev(p["delta"], dtype), dev(p["A"]), dev(p["Bm"], dtype),
                        dev(p["Cm"], dtype), dev(p["Dv"]), dev(p["z"], dtype), h)
    rh, ry = scan_step_ref(h0, p["x"], p["delta"], p["A"], p["Bm"], p["Cm"], p["Dv"], p["z"])
    assert_close(host(h), rh, TOL["f32"], "h")
    assert_close(host(y), ry, TOL[dtype], "y")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_step_chain_matches_sequence_kernel(ss, dtype):
    """37 decode steps from h0 reproduce ss_scan_fwd over the same 37 steps (y and the final state)."""
    import torch
    B, L, D, N = 3, 37, 48, 16
    wl = CONFIGS["tiny"].with_(B=B, L=L, D=D, N=N, dtype=dtype, chunk=16)
    inp = make_scan_inputs(wl, seed=3)
    h0 = round_to(np.random.default_rng(4).standard_normal((B, D, N)), "f32")
    d = {k: dev(v, dtype if k in ("x", "delta", "z", "Bm", "Cm", "dy") else "f32") for k, v in inp.items()}
    y_seq, _, h_seq = ss.ss_scan_fwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], d["Dv"], d["z"], h0=dev(h0),
                                     chunk=16)
    h = dev(h0)
    ys = []
    for t in range(L):
        ys.append(ss.ss_scan_step(d["x"][:, t].contiguous(), d["delta"][:, t].contiguous(), d["A"],
                                  d["Bm"][:, t].contiguous(), d["Cm"][:, t].contiguous(), d["Dv"],
                                  d["z"][:, t].contiguous(), h))
    y_steps = torch.stack(ys, 1)
    assert_close(host(h), host(h_seq), 1e-5, "h")
    assert_close(host(y_steps), host(y_seq), 1e-5 if dtype == "f32" else TOL["bf16"], "y")


@pytest.mark.parametrize("B,D,K,dtype,silu,with_bias", [(2, 16, 4, "f32", False, True), (3, 520, 4, "bf16", True, True),
                                                        (2, 24, 3, "f32", True, False), (1, 8, 1, "bf16", False, True),
                                                        (64, 4096, 4, "bf16", True, True)])
def test_conv_step_parity(ss, B, D, K, dtype, silu, with_bias):
    rng = np.random.default_rng(B + D + K)
    st0 = round_to(rng.standard_normal((B, D, K)), "f32")
    x = round_to(rng.standard_normal((B, D)), dtype)
    w = round_to(rng.uniform(-0.5, 0.5, (D, K)), "f32")
    bias = round_to(rng.standard_normal(D), "f32") if with_bias else None
    st = dev(st0)
    out = ss.conv1d_causal_step(dev(x, dtype), st, dev(w), None if bias is None else dev(bias), silu=silu)
    rst, rout = conv1d_step_fwd_ref(st0, x, w, bias, silu=silu)
    assert np.array_equal(host(st), rst)  # a shift moves values exactly
    assert_close(host(out), rout, TOL[dtype], "out")


def test_conv_step_chain_matches_sequence_kernel(ss):
    import torch
    wl = CONFIGS["tiny"].with_(B=2, L=50, D=72, d_conv=4, dtype="f32")
    c = make_conv_inputs(wl, seed=8)
    x = dev(c["x"])
    seq = ss.conv1d_causal_fwd(x, dev(c["w"]))
    st = torch.zeros((2, 72, 4), device="cuda", dtype=torch.float32)
    outs = [ss.conv1d_causal_step(x[:, t].contiguous(), st, dev(c["w"])) for t in range(50)]
    assert_close(host(torch.stack(outs, 1)), host(seq), 1e-6, "out")
    assert_close(host(seq), conv1d_causal_fwd_ref(c["x"], c["w"]), TOL["f32"], "seq")
